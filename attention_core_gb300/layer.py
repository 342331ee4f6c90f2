"""One transformer layer shard around the attention core, for the layer-level
measurement of selective activation recomputation.

"Reducing Activation Recomputation in Large Transformer Models" (Key
takeaways, fourth bullet) compares recomputing the whole layer in the backward
pass with recomputing only the attention core.  This module builds the layer
that comparison is about, as one tensor-parallel rank's shard, GPT-style with
pre-norm residual blocks:

    qkv = y_in Wqkv                        a local heads of d
    O   = attention core(q, k, v)          this library (causal, softmax dropout)
    z1  = r_in + dropout(O Wo)             this library: dropout + residual add
    y1  = LayerNorm(z1)                      + layer norm
    m1  = y1 W1,  g = GeLU(m1)             GeLU: this library
    z2  = z1 + dropout(g W2)               this library
    y2  = LayerNorm(z2)

The GEMMs are plain cuBLAS calls through ``torch.matmul`` (bf16 operands,
fp32 accumulation, bf16 results); every other step runs in this library's
kernels, and ``torch`` only moves data between layouts.  Without
tensor-parallel peers the two projections produce this rank's partial sums
(the all-reduce or reduce-scatter that would follow is not part of the
measurement), and the GEMMs carry no bias.  The layer norm of the layer's own
input is the previous layer's second block, so the layer takes (y_in, r_in)
and returns (y2, z2).

The backward keeps what selective recomputation keeps: every activation
except the attention core's (the core's backward rebuilds its scores,
probabilities and mask from Q, K, V, O, the LSE and the seed).
"""
from __future__ import annotations

from dataclasses import dataclass

import attention_core_gb300 as ac


@dataclass
class LayerShape:
    b: int          # micro-batch
    s: int          # sequence length
    h: int          # hidden size
    a: int          # local attention heads
    d: int          # head dimension
    ffn: int        # local MLP width (4 h / tensor-parallel size)
    p_drop: float = 0.1
    eps: float = 1e-5

    @property
    def n(self) -> int:
        return self.b * self.s

    def gemm_flops_fwd(self) -> int:
        """Multiply-add FLOPs of the four GEMMs of the forward pass."""
        n, h, ad, f = self.n, self.h, self.a * self.d, self.ffn
        return 2 * n * (h * 3 * ad + ad * h + h * f + f * h)


def init_weights(shape: LayerShape, seed: int, device):
    """Random weights: GEMM weights N(0, 0.02^2) in bf16, layer-norm gammas
    1 + 0.1 N(0, 1) and betas 0.1 N(0, 1) in fp32."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    ad = shape.a * shape.d

    def w(rows, cols):
        return (0.02 * torch.randn((rows, cols), generator=g)).to(torch.bfloat16).to(device)

    def vec(scale, base):
        return (base + scale * torch.randn((shape.h,), generator=g)).to(device)

    return {"wqkv": w(shape.h, 3 * ad), "wo": w(ad, shape.h), "w1": w(shape.h, shape.ffn),
            "w2": w(shape.ffn, shape.h), "gamma1": vec(0.1, 1.0), "beta1": vec(0.1, 0.0),
            "gamma2": vec(0.1, 1.0), "beta2": vec(0.1, 0.0)}


def _heads(x2d, shape: LayerShape):
    """[n, a*d] (token t = batch * s + position) -> [b, a, s, d] contiguous."""
    return x2d.view(shape.b, shape.s, shape.a, shape.d).permute(0, 2, 1, 3).contiguous()


def _tokens(x4d, shape: LayerShape):
    """[b, a, s, d] -> [n, a*d] contiguous."""
    return x4d.permute(0, 2, 1, 3).reshape(shape.n, shape.a * shape.d).contiguous()


class StoredCore:
    """The attention core without recomputation, for the measurement only: the
    forward materialises and keeps what the backward needs -- the softmax
    output P (bf16), the dropout mask (one byte per element) and the dropout
    output (bf16), the 5 a s^2 b bytes of the per-layer activation formula --
    and the backward reads them instead of rebuilding them.  Built from
    cuBLAS products and PyTorch's softmax and dropout; its mask comes from
    PyTorch's generator, not this library's Philox stream, so it computes the
    same function as the library's core only in distribution when p > 0 (and
    exactly, up to rounding, at p = 0).  It is the baseline against which
    recomputation is an overhead, not part of the library's path."""

    def __init__(self, shape: "LayerShape"):
        import torch
        self.shape = shape
        self.scale = 1.0 / float(shape.d) ** 0.5
        self._above = None
        self.torch = torch

    def _causal(self, dev):
        if self._above is None:
            s = self.shape.s
            self._above = self.torch.ones((s, s), dtype=self.torch.bool, device=dev).triu(1)
        return self._above

    def fwd(self, q, k, v):
        torch = self.torch
        s_ = torch.matmul(q, k.transpose(-1, -2))
        s_ = s_.float().mul_(self.scale).masked_fill_(self._causal(q.device), float("-inf"))
        p = torch.softmax(s_, dim=-1).to(torch.bfloat16)
        pd, mask = torch.ops.aten.native_dropout(p, self.shape.p_drop, True)
        o = torch.matmul(pd, v)
        return o, (q, k, v, p, mask, pd)

    def bwd(self, saved, do):
        torch = self.torch
        q, k, v, p, mask, pd = saved
        dv = torch.matmul(pd.transpose(-1, -2), do)
        dpd = torch.matmul(do, v.transpose(-1, -2))
        keep = 1.0 / (1.0 - self.shape.p_drop)
        dp = torch.ops.aten.native_dropout_backward(dpd, mask, keep)
        ds = torch.ops.aten._softmax_backward_data(dp, p, -1, torch.bfloat16)
        dq = torch.matmul(ds, k) * self.scale
        dk = torch.matmul(ds.transpose(-1, -2), q) * self.scale
        return dq, dk, dv


def forward(shape: LayerShape, wts: dict, y_in, r_in, seed: int, offset: int = 0, stored: "StoredCore" = None):
    """Returns (y2, z2, ctx); ctx holds what the backward needs.  The three
    dropouts use Philox counter offsets offset, offset + 1 and offset + 2.
    With `stored`, the core is that no-recomputation baseline instead of this
    library's recomputing core."""
    import torch
    ad = shape.a * shape.d
    qkv = torch.matmul(y_in, wts["wqkv"])
    q, k, v = (_heads(qkv[:, i * ad:(i + 1) * ad], shape) for i in range(3))
    core = dict(causal=True, p_drop=shape.p_drop, seed=seed, offset=offset)
    if stored is not None:
        o, saved = stored.fwd(q, k, v)
        lse = None
        core = dict(core, stored=stored, saved=saved)
    else:
        o, lse = ac.fwd(q, k, v, **core)
    o2 = _tokens(o, shape)
    attn = torch.matmul(o2, wts["wo"])
    d1 = dict(p_drop=shape.p_drop, seed=seed, offset=offset + 1, eps=shape.eps)
    z1, y1, mean1, rstd1 = ac.dropout_add_ln_fwd(attn, r_in, wts["gamma1"], wts["beta1"], **d1)
    m1 = torch.matmul(y1, wts["w1"])
    g = ac.gelu_fwd(m1)
    m2 = torch.matmul(g, wts["w2"])
    d2 = dict(p_drop=shape.p_drop, seed=seed, offset=offset + 2, eps=shape.eps)
    z2, y2, mean2, rstd2 = ac.dropout_add_ln_fwd(m2, z1, wts["gamma2"], wts["beta2"], **d2)
    ctx = dict(y_in=y_in, q=q, k=k, v=v, o=o, lse=lse, o2=o2, z1=z1, mean1=mean1, rstd1=rstd1,
               y1=y1, m1=m1, g=g, z2=z2, mean2=mean2, rstd2=rstd2, core=core, d1=d1, d2=d2)
    return y2, z2, ctx


def backward(shape: LayerShape, wts: dict, ctx: dict, dy2, dz2):
    """Gradients for (y_in, r_in) and the weights, from those of (y2, z2)."""
    import torch
    c = ctx
    dm2, dz1, dgamma2, dbeta2 = ac.dropout_add_ln_bwd(dy2, c["z2"], c["mean2"], c["rstd2"], wts["gamma2"],
                                                      dz_next=dz2, **c["d2"])
    dg = torch.matmul(dm2, wts["w2"].t())
    dw2 = torch.matmul(c["g"].t(), dm2)
    dm1 = ac.gelu_bwd(c["m1"], dg)
    dy1 = torch.matmul(dm1, wts["w1"].t())
    dw1 = torch.matmul(c["y1"].t(), dm1)
    dattn, dr_in, dgamma1, dbeta1 = ac.dropout_add_ln_bwd(dy1, c["z1"], c["mean1"], c["rstd1"], wts["gamma1"],
                                                          dz_next=dz1, **c["d1"])
    do2 = torch.matmul(dattn, wts["wo"].t())
    dwo = torch.matmul(c["o2"].t(), dattn)
    if "stored" in c["core"]:
        dq, dk, dv = c["core"]["stored"].bwd(c["core"]["saved"], _heads(do2, shape))
    else:
        dq, dk, dv = ac.bwd_recompute(c["q"], c["k"], c["v"], c["o"], c["lse"], _heads(do2, shape), **c["core"])
    dqkv = torch.cat([_tokens(t, shape) for t in (dq, dk, dv)], dim=1)
    dy_in = torch.matmul(dqkv, wts["wqkv"].t())
    dwqkv = torch.matmul(c["y_in"].t(), dqkv)
    return {"y_in": dy_in, "r_in": dr_in, "wqkv": dwqkv, "wo": dwo, "w1": dw1, "w2": dw2,
            "gamma1": dgamma1, "beta1": dbeta1, "gamma2": dgamma2, "beta2": dbeta2}


def backward_full(shape: LayerShape, wts: dict, y_in, r_in, dy2, dz2, seed: int, offset: int = 0):
    """Full activation recomputation: the forward kept only the layer's inputs
    (y_in, r_in), so the backward first reruns the whole layer forward from
    them (the same seed and offsets, so the same masks) and then runs the
    backward on what that rerun produced."""
    _, _, ctx = forward(shape, wts, y_in, r_in, seed=seed, offset=offset)
    return backward(shape, wts, ctx, dy2, dz2)
