"""The backward entry point that allocates nothing.

Some callers cannot allocate device memory (their host framework owns every
byte through its own pool, or they run where allocation is forbidden), so
they cannot pass the workspace that attn_core_bwd_recompute needs.
attn_core_bwd_recompute_noalloc uses a fixed scratch array inside the library
instead.  This test calls it through the C ABI twice in a row, on different
inputs, and checks each result against the workspace entry point's on the
same inputs, with the tolerance the other GPU tests use.  It lives in a file
of its own that is collected last, and passes alone or after the others.
"""
import pytest
import torch

import attention_core_gb300 as ac
from attention_core_gb300.inputs import random_inputs
from tests.gpu_util import TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu


def _run(t, seed, noalloc):
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    q, k, v, g = (x.to(dev) for x in (t.q, t.k, t.v, t.dout))
    b, hq, s, d = q.shape
    p = ac.Params(b=b, h_q=hq, h_kv=k.shape[1], s=s, d=d, causal=True, p_drop=0.1, seed=seed)
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


def test_noalloc_matches_workspace_entry_point_twice():
    cases = [((2, 4, 2, 300, 128), 11, 5), ((1, 8, 1, 512, 64), 12, 6)]
    for shape, in_seed, seed in cases:
        t = random_inputs(*shape, seed=in_seed)
        got = _run(t, seed, noalloc=True)
        ref = _run(t, seed, noalloc=False)
        for a, r in zip(got, ref):
            assert row_rel_err(to_np(a), to_np(r)) <= TOL


def test_noalloc_rejects_shapes_beyond_its_array():
    p = ac.Params(b=1, h_q=129, h_kv=1, s=8192, d=128)      # 1,056,768 padded rows > 2^20
    assert ac.attn_core_bwd_recompute_noalloc(p, *([0] * 9), 0) == ac.ERR_WORKSPACE_TOO_SMALL
