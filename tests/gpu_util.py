"""Helpers shared by the GPU parity tests: run the library through its C ABI
and compare against the CPU oracle.

Error metric (the stated bar: max relative error 1e-2 against the oracle's
row-wise max-abs; LSE within 1e-3 absolute).  For each output row (batch,
head, position) the error is the largest absolute difference divided by that
row's own largest absolute oracle value; the test value is the maximum over
rows.  No floor is applied to a row's denominator, with one exception: rows
whose oracle max-abs is below NEAR_ZERO (1e-3) times the median row max-abs
of the compared rows that are not exactly zero.  Those rows cancel to
(nearly) zero by construction -- causal query 0 has dQ = 0 exactly, one key
gives dK = 0 -- and carry the rounding residue of terms as large as a
typical row, which no relative bar can meet.  They are held to an absolute
bound instead: TOL times that median, the absolute error a typical row is
allowed.  Rows that are exactly zero in the oracle (keys that no query sees
under a top-left causal mask with more keys than queries) have no terms at
all, so they do not enter the median that sets the typical row; they are
held to the same absolute bound.  If every compared row is exactly zero the
bound is TOL in absolute terms.

Every call records the strict figure (the largest relative error over the
rows held to the relative bar), the near-zero rows' error against their
absolute bound, and the plain unexempted maximum; the test session prints the
largest ones at the end (tests/conftest.py).
"""
from __future__ import annotations

import numpy as np
import torch

import attention_core_gb300 as ac

TOL = 1e-2
LSE_TOL = 1e-3
NEAR_ZERO = 1e-3

# (test id or label, strict, near-zero rows' error / bound scale, exempt rows, rows)
RECORDS: list = []


def row_errors(gpu, ref) -> dict:
    """The parts of the metric for one output tensor (last axis = a row)."""
    g = np.asarray(gpu, dtype=np.float64).reshape(-1, np.shape(ref)[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, np.shape(ref)[-1])
    rowmax = np.abs(r).max(axis=1)
    err = np.abs(g - r).max(axis=1)
    nonzero = rowmax[rowmax > 0]
    med = float(np.median(nonzero)) if nonzero.size else 0.0
    near = rowmax < NEAR_ZERO * med if med > 0 else np.ones_like(rowmax, dtype=bool)
    strict = float((err[~near] / rowmax[~near]).max()) if (~near).any() else 0.0
    near_err = float(err[near].max() / (med if med > 0 else 1.0)) if near.any() else 0.0
    with np.errstate(divide="ignore", invalid="ignore"):
        unexempt = float(np.max(np.where(rowmax > 0, err / np.where(rowmax > 0, rowmax, 1.0),
                                         np.where(err > 0, np.inf, 0.0))))
    return {"strict": strict, "near_zero": near_err, "n_near": int(near.sum()), "rows": int(len(rowmax)),
            "unexempt": unexempt}


def row_rel_err(gpu, ref, label: str | None = None) -> float:
    """The bar's figure: max(strict relative error, near-zero rows' absolute
    error over TOL's scale); passing means <= TOL."""
    e = row_errors(gpu, ref)
    RECORDS.append((label or _current_test(), e))
    return max(e["strict"], e["near_zero"])


def _current_test() -> str:
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


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
