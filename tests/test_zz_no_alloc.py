"""The backward entry point that allocates nothing.

Some callers cannot allocate device memory (their host framework owns every
byte through its own pool, or they run where allocation is forbidden), so
they cannot pass the workspace that attn_core_bwd_recompute needs.
attn_core_bwd_recompute_noalloc uses a fixed scratch array inside the library
instead.  These tests call it through the C ABI twice in a row, on different
inputs, and check each result against the CPU oracle and against the
workspace entry point on the same inputs, with the tolerance the other GPU
tests use.  Here the dK/dV kernel draws the dropout mask itself (the fixed
array holds no keep bits), so a probe also reads that mask out through dV and
compares it bit for bit with the oracle's.  The file is collected last, and
passes alone or after the others.
"""
import numpy as np
import pytest
import torch

import attention_core_gb300 as ac
import oracle
from attention_core_gb300.inputs import dv_mask_probe, random_inputs
from tests.gpu_util import TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(t, seed, noalloc, causal=True, p_drop=0.1):
    dev = torch.device("cuda:0")
    q, k, v, g = (x.to(dev) for x in (t.q, t.k, t.v, t.dout))
    b, hq, s, d = q.shape
    p = ac.Params(b=b, h_q=hq, h_kv=k.shape[1], s=s, d=d, causal=causal, p_drop=p_drop, seed=seed)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    p.dev_status = status.data_ptr()
    o = torch.empty_like(q)
    lse = torch.empty((b, hq, s), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert ac.attn_core_fwd(p, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), stream) == ac.OK
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ptrs = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), g.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr()]
    if noalloc:
        rc = ac.attn_core_bwd_recompute_noalloc(p, *ptrs, stream)
    else:
        ws_bytes = ac.attn_core_bwd_workspace_bytes(p)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        rc = ac.attn_core_bwd_recompute(p, *ptrs, ws.data_ptr(), ws_bytes, stream)
    assert rc == ac.OK, ac.attn_core_strerror(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dq, dk, dv


def test_noalloc_matches_oracle_and_workspace_entry_point_twice():
    cases = [((2, 4, 2, 300, 128), 11, 5), ((1, 8, 1, 512, 64), 12, 6)]
    for shape, in_seed, seed in cases:
        b, hq, hkv, s, d = shape
        t = random_inputs(*shape, seed=in_seed)
        got = _run(t, seed, noalloc=True)
        ref = _run(t, seed, noalloc=False)
        pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=0.1, seed=seed)
        exact = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
        for name, a, r, x in zip(("dq", "dk", "dv"), got, ref, exact):
            assert row_rel_err(to_np(a), x, f"noalloc {shape} {name} vs oracle") <= TOL, name
            assert row_rel_err(to_np(a), to_np(r), f"noalloc {shape} {name} vs workspace") <= TOL, name


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_dv_mask_bit_exact(d):
    """dV column c of key row j is non-zero exactly when (query w0 + c, key j)
    is kept: the mask the dK/dV kernel draws on its own, in its transposed
    orientation, equals the oracle's bit for bit."""
    b, h, s = 1, 2, 300
    seed = 2024 + d
    pr = oracle.Problem(b=b, h_q=h, h_kv=h, s=s, d=d, causal=True, p_drop=0.1, seed=seed)
    masks = [oracle.mask_rows(pr, bh, 0, s) for bh in range(b * h)]
    for w0 in range(0, s, d):
        t = dv_mask_probe(b, h, h, s, d, w0)
        dv = to_np(_run(t, seed, noalloc=True)[2]).reshape(b * h, s, d)
        width = min(d, s - w0)
        for bh in range(b * h):
            got = (dv[bh, :, :width] != 0).astype(np.uint8)           # [key j, query w0+c]
            assert np.array_equal(got, masks[bh][w0:w0 + width, :].T), (bh, w0)


def test_noalloc_rejects_shapes_beyond_its_array():
    p = ac.Params(b=1, h_q=129, h_kv=1, s=8192, d=128)      # 1,056,768 padded rows > 2^20
    assert ac.attn_core_bwd_recompute_noalloc(p, *([0] * 9), 0) == ac.ERR_WORKSPACE_TOO_SMALL
