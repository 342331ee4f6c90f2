"""Helpers shared by the GPU parity tests: run the library through its C ABI
and compare against the CPU oracle with the row-relative error metric.

Error metric: for each output row (batch, head, position), the largest
absolute difference divided by the largest absolute oracle value of that row
(floor 1e-30); the test value is the maximum over rows.  Limits: 1e-2 for O,
dQ, dK, dV; LSE within 1e-3 absolute.  Dropout masks and byte counts are
compared exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import attention_core_gb300 as ac

TOL = 1e-2
LSE_TOL = 1e-3


def row_rel_err(gpu, ref) -> float:
    g = np.asarray(gpu, dtype=np.float64).reshape(-1, np.shape(ref)[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, np.shape(ref)[-1])
    den = np.maximum(np.abs(r).max(axis=1), 1e-30)
    return float((np.abs(g - r).max(axis=1) / den).max())


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy()


def run_gpu(t, causal: bool, p_drop: float, seed: int, offset: int = 0, scale: float = 0.0,
            bwd: bool = True):
    """Forward (and backward) on cuda:0; checks the device status word."""
    dev = torch.device("cuda:0")
    q, k, v, g = (x.to(dev).contiguous() for x in (t.q, t.k, t.v, t.dout))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kw = dict(causal=causal, p_drop=p_drop, seed=seed, offset=offset, scale=scale,
              dev_status=status.data_ptr())
    o, lse = ac.fwd(q, k, v, **kw)
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv = ac.bwd_recompute(q, k, v, o, lse, g, **kw)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    st = int(status.item())
    assert st == 0, f"device status {st:#x}"
    return out
