"""Variable-length (packed) batches on the GPU: each sequence of a packed
[tokens, heads, d] batch against the oracle (sequence i as batch element i
of an ordinary problem, through the sampled-row entry points), ragged and
empty sequences, causal and cross-attention lengths, GQA; and a packed batch
of equal lengths bit-identical to the padded layout."""
import numpy as np
import pytest
import torch

import attention_core_gb300 as ac
import oracle
from tests.gpu_util import LSE_TOL, TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _packed(lens, heads, d, gen):
    return torch.randn((int(sum(lens)), heads, d), generator=gen).to(torch.bfloat16)


def _cu(lens):
    return [0] + list(np.cumsum(lens).astype(int))


def _seq_problem(i, lq, lk, hq, hkv, d, causal, p, seed):
    return oracle.Problem(b=i + 1, h_q=hq, h_kv=hkv, s=lq, d=d, causal=causal, p_drop=p, seed=seed,
                          s_kv=lk)


def _as_batch(x_packed, c0, c1, i, heads):
    """Rows c0..c1 of a packed tensor as batch element i of [i+1, heads, L, d] (others zero)."""
    seq = x_packed[c0:c1].double().numpy().transpose(1, 0, 2)
    out = np.zeros((i + 1,) + seq.shape)
    out[i] = seq
    return out


# (query lengths, key lengths or None, h_q, h_kv, d, causal, p)
CASES = [
    ([130, 1, 256, 0, 77], None, 2, 2, 64, True, 0.1),
    ([200, 64, 129], None, 4, 2, 128, True, 0.1),
    ([100, 300], [257, 40], 2, 1, 128, False, 0.2),
    ([90, 150], None, 2, 2, 160, True, 0.1),
    ([100, 300, 5], [257, 40, 5], 2, 1, 128, True, 0.1),    # causal, top-left per sequence
    ([1, 600, 0, 129, 128, 77, 1000, 3], None, 2, 2, 96, True, 0.1),   # many lengths, one launch
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"q{'-'.join(map(str, c[0]))}_d{c[4]}_{'c' if c[5] else 'nc'}")
def test_varlen_matches_oracle(case):
    lq, lk, hq, hkv, d, causal, p = case
    lk = lk or lq
    gen = torch.Generator(device="cpu").manual_seed(sum(lq) + d)
    q, do = _packed(lq, hq, d, gen), _packed(lq, hq, d, gen)
    k, v = _packed(lk, hkv, d, gen), _packed(lk, hkv, d, gen)
    cq, ck = _cu(lq), _cu(lk)
    seed = 777 + d
    dev = torch.device("cuda:0")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kw = dict(causal=causal, p_drop=p, seed=seed, dev_status=status.data_ptr())
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ac.fwd_varlen(qd, kd, vd, cq, ck, **kw)
    dq, dk, dv = ac.bwd_varlen(qd, kd, vd, o, lse, dod, cq, ck, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o, lse, dq, dk, dv = (to_np(t) for t in (o, lse, dq, dk, dv))
    for i, (a, b) in enumerate(zip(lq, lk)):
        if a == 0:
            continue
        pr = _seq_problem(i, a, b, hq, hkv, d, causal, p, seed)
        qb, dob = _as_batch(q, cq[i], cq[i + 1], i, hq), _as_batch(do, cq[i], cq[i + 1], i, hq)
        kb, vb = _as_batch(k, ck[i], ck[i + 1], i, hkv), _as_batch(v, ck[i], ck[i + 1], i, hkv)
        bh = np.repeat(np.arange(i * hq, (i + 1) * hq), a)
        rows = np.tile(np.arange(a), hq)
        ro, rlse = oracle.fwd_rows(pr, qb, kb, vb, bh, rows)
        rdq = oracle.dq_rows(pr, qb, kb, vb, dob, bh, rows)
        bkv = np.repeat(np.arange(i * hkv, (i + 1) * hkv), b)
        krows = np.tile(np.arange(b), hkv)
        rdk, rdv = oracle.dkdv_rows(pr, qb, kb, vb, dob, bkv, krows)
        # GPU rows in the same (head, row) order
        go = o[cq[i]:cq[i + 1]].transpose(1, 0, 2).reshape(-1, d)
        gdq = dq[cq[i]:cq[i + 1]].transpose(1, 0, 2).reshape(-1, d)
        gdk = dk[ck[i]:ck[i + 1]].transpose(1, 0, 2).reshape(-1, d)
        gdv = dv[ck[i]:ck[i + 1]].transpose(1, 0, 2).reshape(-1, d)
        glse = lse[:, cq[i]:cq[i + 1]].reshape(-1)
        errs = {"o": row_rel_err(go, ro), "dq": row_rel_err(gdq, rdq), "dk": row_rel_err(gdk, rdk),
                "dv": row_rel_err(gdv, rdv)}
        assert float(np.abs(glse - rlse).max()) <= LSE_TOL, i
        assert all(e <= TOL for e in errs.values()), (i, errs)


@pytest.mark.parametrize("d", [64, 128])
def test_equal_lengths_match_padded_layout_bit_for_bit(d):
    b, h, s, p = 3, 2, 200, 0.1
    gen = torch.Generator(device="cpu").manual_seed(d)
    q, k, v, do = (torch.randn((b, h, s, d), generator=gen).to(torch.bfloat16) for _ in range(4))
    dev = torch.device("cuda:0")
    kw = dict(causal=True, p_drop=p, seed=4242)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ac.fwd(qd, kd, vd, **kw)
    dq, dk, dv = ac.bwd_recompute(qd, kd, vd, o, lse, dod, **kw)

    def pack(t):                      # [b, h, s, d] -> [b*s, h, d]
        return t.permute(0, 2, 1, 3).reshape(b * s, h, d).contiguous()

    cu = [i * s for i in range(b + 1)]
    o2, lse2 = ac.fwd_varlen(pack(qd), pack(kd), pack(vd), cu, **kw)
    dq2, dk2, dv2 = ac.bwd_varlen(pack(qd), pack(kd), pack(vd), o2, lse2, pack(dod), cu, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o2, pack(o))
    assert torch.equal(lse2, lse.permute(1, 0, 2).reshape(h, b * s))
    for x, y in ((dq2, dq), (dk2, dk), (dv2, dv)):
        assert torch.equal(x, pack(y))


def test_sequence_without_queries_gets_zero_key_gradients():
    """A cross-attention sequence with keys but no queries: no query sees its
    keys, so their dK and dV rows are zero -- written as zeros, whatever the
    output buffers held before the call.  The other sequence still matches
    the oracle."""
    lq, lk, hq, hkv, d, p = [0, 100], [50, 80], 2, 2, 64, 0.1
    gen = torch.Generator(device="cpu").manual_seed(5)
    q, do = _packed(lq, hq, d, gen), _packed(lq, hq, d, gen)
    k, v = _packed(lk, hkv, d, gen), _packed(lk, hkv, d, gen)
    cq, ck = _cu(lq), _cu(lk)
    seed = 31337
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    pr_c = ac.Params(b=1, h_q=hq, h_kv=hkv, s=1, d=d, causal=False, p_drop=p, seed=seed)
    o, lse = ac.fwd_varlen(qd, kd, vd, cq, ck, causal=False, p_drop=p, seed=seed)
    dq = torch.empty_like(qd)
    dk = torch.full_like(kd, 1.0)
    dv = torch.full_like(vd, -2.0)
    tq, tk, pq, pk = ac._device_tables(cq, ck, dev)
    ws_bytes = ac.attn_core_bwd_varlen_workspace_bytes(pr_c, cq, ck, cu_q_dev=pq, cu_k_dev=pk)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    rc = ac.attn_core_bwd_varlen(pr_c, cq, ck, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), dod.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                 ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream,
                                 cu_q_dev=pq, cu_k_dev=pk)
    assert rc == ac.OK, ac.attn_core_strerror(rc)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk[:50]).item() == 0
    assert torch.count_nonzero(dv[:50]).item() == 0
    i = 1
    pr = _seq_problem(i, lq[i], lk[i], hq, hkv, d, False, p, seed)
    qb, dob = _as_batch(q, cq[i], cq[i + 1], i, hq), _as_batch(do, cq[i], cq[i + 1], i, hq)
    kb, vb = _as_batch(k, ck[i], ck[i + 1], i, hkv), _as_batch(v, ck[i], ck[i + 1], i, hkv)
    bkv = np.repeat(np.arange(i * hkv, (i + 1) * hkv), lk[i])
    krows = np.tile(np.arange(lk[i]), hkv)
    rdk, rdv = oracle.dkdv_rows(pr, qb, kb, vb, dob, bkv, krows)
    gdk = to_np(dk)[ck[i]:ck[i + 1]].transpose(1, 0, 2).reshape(-1, d)
    gdv = to_np(dv)[ck[i]:ck[i + 1]].transpose(1, 0, 2).reshape(-1, d)
    assert row_rel_err(gdk, rdk) <= TOL
    assert row_rel_err(gdv, rdv) <= TOL
