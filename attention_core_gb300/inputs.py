"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no arithmetic of the attention core: it only draws random
numbers and lays out fixed probe patterns.  Both the CUDA path and the CPU
oracle receive exactly the tensors built here.

Recipe for the random inputs: a CPU ``torch.Generator`` seeded with the given
seed draws Q, K, V and dO, in that order, as fp32 N(0, 1) and rounds each to
bf16 (round to nearest even).  The same bf16 bits go to the GPU and, widened
exactly to fp64, to the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# Named workloads: the GPT-3-style layers of the paper (one tensor-parallel
# rank of eight, so local heads = heads / 8) and a Llama-3-70B-shaped layer.
# Fields: b, h_q, h_kv, s, d, p_drop.
WORKLOADS = {
    "tiny": dict(b=1, h_q=2, h_kv=2, s=128, d=64, p_drop=0.1),
    "gpt22b": dict(b=4, h_q=8, h_kv=8, s=2048, d=96, p_drop=0.1),
    "gpt175b": dict(b=2, h_q=12, h_kv=12, s=2048, d=128, p_drop=0.1),
    "gpt530b": dict(b=1, h_q=16, h_kv=16, s=2048, d=160, p_drop=0.1),
    "llama70b_p0": dict(b=1, h_q=64, h_kv=8, s=8192, d=128, p_drop=0.0),
    "llama70b_p01": dict(b=1, h_q=64, h_kv=8, s=8192, d=128, p_drop=0.1),
}


@dataclass
class Tensors:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor


def random_inputs(b: int, h_q: int, h_kv: int, s: int, d: int, seed: int, s_kv: int = 0) -> Tensors:
    """bf16 Q [b,h_q,s,d], K/V [b,h_kv,s_kv,d], dO [b,h_q,s,d], all N(0,1), on the CPU.

    s_kv = 0 means s_kv = s (self-attention)."""
    s_kv = s_kv or s
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((b, h_q, s, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((b, h_kv, s_kv, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((b, h_kv, s_kv, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    dout = torch.randn((b, h_q, s, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return Tensors(q, k, v, dout)


def growing_scores_inputs(b: int, h_q: int, h_kv: int, s: int, d: int, seed: int) -> Tensors:
    """bf16 inputs whose first two 128-key blocks score far below the rest, on the CPU.

    Q entries are 0.75 + 0.75 N(0,1); K rows have N(0,1) entries plus a common
    mean that puts the scaled scores of keys 0..127 about 20 and of keys
    128..255 about 10 below the others (mean offset / (0.75 sqrt(d)) per entry).
    A query that sees key block 2 then finds its running row maximum rising by
    about 10 at block 1 and again at block 2, while the early keys keep
    probabilities near zero (no large common component of K is left for the
    gradients to cancel).  V and dO are N(0,1)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = (0.75 + 0.75 * torch.randn((b, h_q, s, d), generator=g, dtype=torch.float32)).to(torch.bfloat16)
    blk = torch.arange(s) // 128
    offset = torch.where(blk == 0, -20.0, torch.where(blk == 1, -10.0, 0.0)).to(torch.float32)
    mean_k = (offset / (0.75 * float(d) ** 0.5)).view(1, 1, s, 1)
    k = (torch.randn((b, h_kv, s, d), generator=g, dtype=torch.float32) + mean_k).to(torch.bfloat16)
    v = torch.randn((b, h_kv, s, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    dout = torch.randn((b, h_q, s, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return Tensors(q, k, v, dout)


def fwd_mask_probe(b: int, h_q: int, h_kv: int, s: int, d: int, w0: int) -> Tensors:
    """Inputs that expose the forward dropout mask on a window of keys.

    Q = K = 0 makes every visible score equal, and V row j is the unit vector
    e_(j - w0) for keys j in [w0, w0 + d) (zero elsewhere), so output column c
    of query row i is non-zero exactly when key w0 + c is visible to row i
    and kept by dropout.
    """
    q = torch.zeros((b, h_q, s, d), dtype=torch.bfloat16)
    k = torch.zeros((b, h_kv, s, d), dtype=torch.bfloat16)
    v = torch.zeros((b, h_kv, s, d), dtype=torch.bfloat16)
    for c in range(d):
        j = w0 + c
        if j < s:
            v[:, :, j, c] = 1.0
    dout = torch.zeros((b, h_q, s, d), dtype=torch.bfloat16)
    return Tensors(q, k, v, dout)


def dv_mask_probe(b: int, h_q: int, h_kv: int, s: int, d: int, w0: int) -> Tensors:
    """Inputs that expose the backward dropout mask through dV.

    Q = K = 0 (equal scores), V = 0, and dO row i is e_(i - w0) for query
    rows i in [w0, w0 + d): column c of dV row j then collects only the
    probability of (query w0 + c, key j), non-zero exactly when that pair is
    visible and kept.  Use with one query head per KV head (h_q == h_kv).
    """
    q = torch.zeros((b, h_q, s, d), dtype=torch.bfloat16)
    k = torch.zeros((b, h_kv, s, d), dtype=torch.bfloat16)
    v = torch.zeros((b, h_kv, s, d), dtype=torch.bfloat16)
    dout = torch.zeros((b, h_q, s, d), dtype=torch.bfloat16)
    for c in range(d):
        i = w0 + c
        if i < s:
            dout[:, :, i, c] = 1.0
    return Tensors(q, k, v, dout)


def dq_mask_probe(b: int, h_q: int, h_kv: int, s: int, d: int, w0: int) -> Tensors:
    """Inputs that make dQ depend on the dropout mask of a window of keys.

    Q = 0 (equal scores), V rows and dO rows all e_0, and K row j is
    e_(j - w0) for keys in [w0, w0 + d): dQ column c of row i then takes one
    of two well-separated values depending on whether key w0 + c was kept.
    """
    q = torch.zeros((b, h_q, s, d), dtype=torch.bfloat16)
    k = torch.zeros((b, h_kv, s, d), dtype=torch.bfloat16)
    v = torch.zeros((b, h_kv, s, d), dtype=torch.bfloat16)
    dout = torch.zeros((b, h_q, s, d), dtype=torch.bfloat16)
    v[..., 0] = 1.0
    dout[..., 0] = 1.0
    for c in range(d):
        j = w0 + c
        if j < s:
            k[:, :, j, c] = 1.0
    return Tensors(q, k, v, dout)


# Dropout + residual add + layer norm on either side of the core: the rows are
# tokens (s * b of them), the columns the hidden size h of the layer.
DAL_WORKLOADS = {
    "tiny": dict(n_rows=64, hidden=1024, p_drop=0.1),
    "gpt175b": dict(n_rows=4096, hidden=12288, p_drop=0.1),
}


@dataclass
class DalTensors:
    x: torch.Tensor          # sub-layer output entering the dropout, bf16 [n_rows, hidden]
    residual: torch.Tensor   # residual stream, bf16 [n_rows, hidden]
    gamma: torch.Tensor      # fp32 [hidden]
    beta: torch.Tensor       # fp32 [hidden]
    dy: torch.Tensor         # gradient of the layer-norm output, bf16 [n_rows, hidden]
    dz_next: torch.Tensor    # gradient reaching z through the residual path, bf16


def dal_inputs(n_rows: int, hidden: int, seed: int) -> DalTensors:
    """x, residual, dy, dz_next ~ N(0, 1) in bf16 (drawn in that order after
    gamma = 1 + 0.1 N(0, 1) and beta = 0.1 N(0, 1), fp32), on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    gamma = 1.0 + 0.1 * torch.randn((hidden,), generator=g, dtype=torch.float32)
    beta = 0.1 * torch.randn((hidden,), generator=g, dtype=torch.float32)
    x, r, dy, dzn = (torch.randn((n_rows, hidden), generator=g, dtype=torch.float32).to(torch.bfloat16)
                     for _ in range(4))
    return DalTensors(x, r, gamma, beta, dy, dzn)


def dal_mask_probe(n_rows: int, hidden: int) -> DalTensors:
    """x = 1, residual = 0, gamma = 1, beta = 0: z is the keep factor of each
    element (0 where dropped), so z exposes the dropout mask."""
    ones = torch.ones((n_rows, hidden), dtype=torch.bfloat16)
    zeros = torch.zeros((n_rows, hidden), dtype=torch.bfloat16)
    return DalTensors(ones, zeros, torch.ones(hidden), torch.zeros(hidden), zeros.clone(), zeros.clone())
