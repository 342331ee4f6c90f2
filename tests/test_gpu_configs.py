"""GPU parity on the full-size workloads (the GPT-3-style 22B/175B/530B layer
shards and the Llama-3-70B-shaped layer), in the launch configuration the
bench times.  The oracle computes sampled rows one by one -- first, tile-edge,
middle and last query rows of several heads, and key rows near the end of
each sequence -- and properties that hold at any size are checked on the
whole output (finite values; dK summing to zero over keys, because every row
of dS sums to zero)."""
import numpy as np
import pytest
import torch

import oracle
from attention_core_gb300.inputs import WORKLOADS, random_inputs
from tests.gpu_util import LSE_TOL, TOL, row_rel_err, run_gpu, to_np

pytestmark = pytest.mark.gpu

NAMES = ["gpt22b", "gpt175b", "gpt530b", "llama70b_p0", "llama70b_p01"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _query_rows(s, rng):
    base = {0, 1, 2, 127, 128, 129, s // 2, s - 129, s - 128, s - 2, s - 1}
    base |= set(int(x) for x in rng.integers(0, s, size=6))
    return sorted(r for r in base if 0 <= r < s)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_sampled_rows(name):
    w = WORKLOADS[name]
    b, hq, hkv, s, d, p = w["b"], w["h_q"], w["h_kv"], w["s"], w["d"], w["p_drop"]
    idx = NAMES.index(name) + 1
    seed = 0x5EED0000 + idx
    t = random_inputs(b, hq, hkv, s, d, seed=idx)
    out = run_gpu(t, True, p, seed)
    for k_, x in out.items():
        assert torch.isfinite(x).all(), k_

    qn, kn, vn, gn = (x.double().numpy() for x in (t.q, t.k, t.v, t.dout))
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=p, seed=seed)
    rng = np.random.default_rng(idx)
    nbh = b * hq
    heads = sorted({0, nbh - 1, nbh // 2})
    bh_list, rows = [], []
    for h in heads:
        for r in _query_rows(s, rng):
            bh_list.append(h)
            rows.append(r)
    bh_list, rows = np.array(bh_list), np.array(rows)
    ro, rlse = oracle.fwd_rows(pr, qn, kn, vn, bh_list, rows)
    rdq = oracle.dq_rows(pr, qn, kn, vn, gn, bh_list, rows)
    o = to_np(out["o"]).reshape(nbh, s, d)[bh_list, rows]
    lse = to_np(out["lse"]).reshape(nbh, s)[bh_list, rows]
    dq = to_np(out["dq"]).reshape(nbh, s, d)[bh_list, rows]
    assert row_rel_err(o, ro) <= TOL
    assert float(np.abs(lse - rlse).max()) <= LSE_TOL
    assert row_rel_err(dq, rdq) <= TOL

    nkv = b * hkv
    kv_heads = sorted({0, nkv - 1})
    tail = [s - 1, s - 2, s - 127, s - 128, s - 129, s - 200]
    early = [0, 1, 127, 128, s // 2] if hq == hkv else []    # cheap only without GQA
    bkv_list = np.array([h for h in kv_heads for _ in tail + early])
    krows = np.array([r for _ in kv_heads for r in tail + early])
    rdk, rdv = oracle.dkdv_rows(pr, qn, kn, vn, gn, bkv_list, krows)
    dk = to_np(out["dk"]).reshape(nkv, s, d)[bkv_list, krows]
    dv = to_np(out["dv"]).reshape(nkv, s, d)[bkv_list, krows]
    assert row_rel_err(dk, rdk) <= TOL
    assert row_rel_err(dv, rdv) <= TOL

    # sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0 for every KV head
    dk_all = out["dk"].float().reshape(nkv, s, d)
    colsum = dk_all.sum(dim=1).abs()
    scale_ = dk_all.abs().sum(dim=1)
    assert float((colsum / scale_.clamp_min(1e-30)).max()) <= TOL


@pytest.mark.parametrize("name", ["gpt175b", "llama70b_p01"])
def test_full_size_forward_mask_sampled(name):
    """Bit-exact forward mask on one head of the full-size shape (probe inputs),
    for key windows at the start, middle and end of the sequence."""
    from attention_core_gb300.inputs import fwd_mask_probe
    w = WORKLOADS[name]
    b, hq, hkv, s, d = w["b"], w["h_q"], w["h_kv"], w["s"], w["d"]
    seed = 0xABCDEF
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=0.1, seed=seed)
    nbh = b * hq
    for w0 in (0, (s // 2 // d) * d, s - d):
        t = fwd_mask_probe(b, hq, hkv, s, d, w0)
        o = to_np(run_gpu(t, True, 0.1, seed, bwd=False)["o"]).reshape(nbh, s, d)
        for bh in (0, nbh - 1):
            m = oracle.mask_rows(pr, bh, 0, s)[:, w0:w0 + d]
            got = (o[bh] != 0).astype(np.uint8)
            assert np.array_equal(got, m), (bh, w0)
