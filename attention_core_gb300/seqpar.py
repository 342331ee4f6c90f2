"""Sequence parallelism around one tensor-parallel layer shard: the converters
between the sequence-split regions and the tensor-parallel regions, and the
layer of ``attention_core_gb300.layer`` run with them over a process group.

"Reducing Activation Recomputation in Large Transformer Models" (Key
takeaways, second and fifth bullets):

* The layer norms, dropouts and residual adds act on each sequence position
  on its own, so with t tensor-parallel ranks each rank keeps only n / t of the
  n = b s tokens there (sequence-split).  The attention block and the MLP stay
  tensor-parallel: all n tokens, a / t heads and f / t MLP columns per rank.
* Entering a tensor-parallel region is an all-gather of the tokens (called g
  below; its backward is a reduce-scatter).  Leaving it is a reduce-scatter of
  the ranks' partial products (g_bar; its backward is an all-gather).  A ring
  all-reduce is a reduce-scatter followed by an all-gather, so the layer's
  four all-gathers and four reduce-scatters (forward and backward) move the
  bytes of the four all-reduces that tensor parallelism alone needs.
* The sequence-split input of each first linear layer is not kept whole: the
  backward all-gathers it again for the weight gradient, and that all-gather
  runs while the input gradient's product is computed (and the reduce-scatter
  of the input gradient while the weight gradient's product is).

Token t of a [n, h] tensor is (batch t // s, position t % s), as in
``layer``; sequence-split rank k holds tokens [k n / t, (k + 1) n / t)
(n divisible by t).  ``Comm`` runs each collective as a ring over
point-to-point messages and counts the bytes each rank sends, so the
bandwidth claim is measured, not assumed.  The per-region arithmetic is a
pluggable ``ops`` object (``LibraryOps``: this library's kernels and cuBLAS
GEMMs on a GPU); the converters and the order of operations are this
module's.
"""
from __future__ import annotations

import threading
from dataclasses import dataclass, field


@dataclass
class Comm:
    """Ring collectives over a torch.distributed group (point-to-point sends),
    with the bytes this rank sent counted per kind of collective."""
    group: object = None
    sent: dict = field(default_factory=lambda: {"all_gather": 0, "reduce_scatter": 0, "all_reduce": 0,
                                                "regather": 0})
    log: list = field(default_factory=list)

    def __post_init__(self):
        import torch.distributed as dist
        self.dist = dist
        self.rank = dist.get_rank(self.group)
        self.world = dist.get_world_size(self.group)
        self._lock = threading.Lock()

    def _peer(self, r):
        return self.dist.get_global_rank(self.group, r) if self.group is not None else r

    def _exchange(self, send, recv, kind):
        """Send `send` to the next rank of the ring while receiving `recv` from
        the previous one."""
        nxt, prv = (self.rank + 1) % self.world, (self.rank - 1) % self.world
        req = self.dist.isend(send.contiguous(), self._peer(nxt), group=self.group)
        self.dist.recv(recv, self._peer(prv), group=self.group)
        req.wait()
        with self._lock:
            self.sent[kind] += send.numel() * send.element_size()

    def _all_gather_chunks(self, chunks, kind):
        """Ring all-gather in place: on entry chunks[rank] holds this rank's part."""
        import torch
        t = self.world
        for step in range(t - 1):
            s_idx = (self.rank - step) % t
            r_idx = (self.rank - step - 1) % t
            buf = torch.empty_like(chunks[r_idx])
            self._exchange(chunks[s_idx], buf, kind)
            chunks[r_idx].copy_(buf)

    def _reduce_scatter_chunks(self, chunks, kind):
        """Ring reduce-scatter in place: afterwards chunks[rank] holds the sum
        over ranks of that chunk."""
        import torch
        t = self.world
        for step in range(t - 1):
            s_idx = (self.rank - step - 1) % t
            r_idx = (self.rank - step - 2) % t
            buf = torch.empty_like(chunks[r_idx])
            self._exchange(chunks[s_idx], buf, kind)
            chunks[r_idx].add_(buf)

    def all_gather(self, x, kind: str = "all_gather"):
        """[m, ...] per rank -> [t m, ...], rank k's rows at [k m, (k + 1) m).
        kind "regather": the backward's second all-gather of a kept input."""
        import torch
        self.log.append((kind, tuple(x.shape)))
        out = torch.empty((self.world * x.shape[0],) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
        chunks = list(out.chunk(self.world))
        chunks[self.rank].copy_(x)
        self._all_gather_chunks(chunks, kind)
        return out

    def reduce_scatter(self, x):
        """[t m, ...] partial sums per rank -> [m, ...]: rows [k m, (k + 1) m) of
        the sum over ranks, on rank k."""
        self.log.append(("reduce_scatter", tuple(x.shape)))
        chunks = [c.clone() for c in x.chunk(self.world)]
        self._reduce_scatter_chunks(chunks, "reduce_scatter")
        return chunks[self.rank]

    def all_reduce(self, x):
        """Sum over ranks: a ring reduce-scatter followed by a ring all-gather."""
        import torch
        self.log.append(("all_reduce", tuple(x.shape)))
        chunks = [c.clone() for c in x.chunk(self.world)]
        self._reduce_scatter_chunks(chunks, "all_reduce")
        self._all_gather_chunks(chunks, "all_reduce")
        return torch.cat(chunks)

    def all_gather_async(self, x, kind: str = "all_gather"):
        """Start an all-gather on a helper thread; .wait() returns its result.
        The caller issues no other collective before waiting."""
        box = {}

        def run():
            box["out"] = self.all_gather(x, kind)

        th = threading.Thread(target=run)
        th.start()

        class _Handle:
            def wait(self_inner):
                th.join()
                return box["out"]
        return _Handle()


@dataclass
class ParallelShape:
    b: int          # micro-batch
    s: int          # sequence length
    h: int          # hidden size
    a: int          # attention heads of the whole layer
    d: int          # head dimension
    ffn: int        # MLP width of the whole layer
    t: int          # tensor-parallel (and sequence-parallel) ranks
    p_drop: float = 0.0
    eps: float = 1e-5

    @property
    def n(self) -> int:
        return self.b * self.s

    def check(self):
        if self.a % self.t or self.ffn % self.t or self.n % self.t:
            raise ValueError("heads, MLP width and tokens must divide by the tensor-parallel size")


def shard_weights(full: dict, shape: ParallelShape, rank: int) -> dict:
    """Rank `rank`'s slices of the layer's weights: the columns of Wqkv that
    produce its a / t heads (of each of q, k, v), the matching rows of Wo, its
    f / t columns of W1 and rows of W2; layer-norm parameters replicated."""
    import torch
    t, ad = shape.t, shape.a * shape.d
    al = ad // t
    cols = torch.cat([torch.arange(i * ad + rank * al, i * ad + (rank + 1) * al) for i in range(3)])
    fl = shape.ffn // t
    return {"wqkv": full["wqkv"][:, cols].contiguous(), "wo": full["wo"][rank * al:(rank + 1) * al].contiguous(),
            "w1": full["w1"][:, rank * fl:(rank + 1) * fl].contiguous(),
            "w2": full["w2"][rank * fl:(rank + 1) * fl].contiguous(),
            **{k: full[k] for k in ("gamma1", "beta1", "gamma2", "beta2")}}


def _heads(x2d, b, s, a, d):
    return x2d.view(b, s, a, d).permute(0, 2, 1, 3).contiguous()


def _tokens(x4d):
    b, a, s, d = x4d.shape
    return x4d.permute(0, 2, 1, 3).reshape(b * s, a * d).contiguous()


def forward(shape: ParallelShape, wts: dict, comm: Comm, y_in, r_in, ops, sequence_parallel: bool = True):
    """One layer on this rank.  Sequence-parallel: y_in and r_in are this
    rank's n / t tokens and so are the outputs (y2, z2).  Tensor-parallel only:
    y_in, r_in and the outputs hold all n tokens on every rank (replicated
    layer norms and dropouts).  Returns (y2, z2, ctx)."""
    shape.check()
    al = shape.a // shape.t
    ad = al * shape.d
    Y = comm.all_gather(y_in) if sequence_parallel else y_in                 # g
    qkv = ops.matmul(Y, wts["wqkv"])
    q, k, v = (_heads(qkv[:, i * ad:(i + 1) * ad], shape.b, shape.s, al, shape.d) for i in range(3))
    o, core = ops.core_fwd(q, k, v)
    o2 = _tokens(o)
    attn = ops.matmul(o2, wts["wo"])                                         # partial sum
    attn = comm.reduce_scatter(attn) if sequence_parallel else comm.all_reduce(attn)   # g_bar
    z1, y1, dal1 = ops.dal_fwd(attn, r_in, wts["gamma1"], wts["beta1"], 1)
    Y1 = comm.all_gather(y1) if sequence_parallel else y1                    # g
    m1 = ops.matmul(Y1, wts["w1"])
    g = ops.gelu_fwd(m1)
    m2 = ops.matmul(g, wts["w2"])
    m2 = comm.reduce_scatter(m2) if sequence_parallel else comm.all_reduce(m2)         # g_bar
    z2, y2, dal2 = ops.dal_fwd(m2, z1, wts["gamma2"], wts["beta2"], 2)
    # Kept for the backward: the sequence-split inputs of the two first linear
    # layers (y_in, y1), not their gathered copies; the core keeps q, k, v, o
    # and its row statistics only.
    ctx = dict(y_in=y_in, y1=y1, q=q, k=k, v=v, core=core, o2=o2, m1=m1, g=g, dal1=dal1, dal2=dal2,
               sp=sequence_parallel)
    return y2, z2, ctx


def _first_linear_backward(comm: Comm, ops, x_kept, w, dout, sp: bool, events: list | None):
    """Backward of a first linear layer out = X w with X = g(x_kept): the input
    gradient's product runs while X is all-gathered again, and the weight
    gradient's product while the input gradient is reduce-scattered."""
    if not sp:
        dX = ops.matmul(dout, w.t())
        dw = ops.matmul(x_kept.t(), dout)
        return comm.all_reduce(dX), dw
    h = comm.all_gather_async(x_kept, "regather")
    if events is not None:
        events.append("gather_started")
    dX = ops.matmul(dout, w.t())                 # overlaps the all-gather
    if events is not None:
        events.append("dx_product_done")
    X = h.wait()
    if events is not None:
        events.append("gather_done")
    box = {}

    def rs():
        box["dx"] = comm.reduce_scatter(dX)
    th = threading.Thread(target=rs)
    th.start()
    dw = ops.matmul(X.t(), dout)                 # overlaps the reduce-scatter
    if events is not None:
        events.append("dw_product_done")
    th.join()
    return box["dx"], dw


def backward(shape: ParallelShape, wts: dict, comm: Comm, ctx: dict, dy2, dz2, ops, events: list | None = None):
    """Gradients of (y_in, r_in) -- sequence-split like them under sequence
    parallelism -- and of this rank's weights, from those of (y2, z2)."""
    c = ctx
    sp = c["sp"]
    dm2, dz1, dgamma2, dbeta2 = ops.dal_bwd(c["dal2"], dy2, dz2)
    dM2 = comm.all_gather(dm2) if sp else dm2                                # backward of g_bar
    dg = ops.matmul(dM2, wts["w2"].t())
    dw2 = ops.matmul(c["g"].t(), dM2)
    dm1 = ops.gelu_bwd(c["m1"], dg)
    dy1, dw1 = _first_linear_backward(comm, ops, c["y1"], wts["w1"], dm1, sp, events)   # backward of g
    dattn, dr_in, dgamma1, dbeta1 = ops.dal_bwd(c["dal1"], dy1, dz1)
    dA = comm.all_gather(dattn) if sp else dattn                            # backward of g_bar
    do2 = ops.matmul(dA, wts["wo"].t())
    dwo = ops.matmul(c["o2"].t(), dA)
    al = shape.a // shape.t
    dq, dk, dv = ops.core_bwd(c["core"], _heads(do2, shape.b, shape.s, al, shape.d))
    import torch
    dqkv = torch.cat([_tokens(x) for x in (dq, dk, dv)], dim=1)
    dy_in, dwqkv = _first_linear_backward(comm, ops, c["y_in"], wts["wqkv"], dqkv, sp, events)
    return {"y_in": dy_in, "r_in": dr_in, "wqkv": dwqkv, "wo": dwo, "w1": dw1, "w2": dw2,
            "gamma1": dgamma1, "beta1": dbeta1, "gamma2": dgamma2, "beta2": dbeta2}


class LibraryOps:
    """The regions' arithmetic on a GPU: this library's attention core,
    dropout + residual add + layer norm and GeLU kernels, and cuBLAS GEMMs
    (torch.matmul).  Ranks hold different tokens (sequence-split) or heads
    (tensor-parallel), so each rank draws its dropout masks with its own
    Philox counter words 3: offset + 3 rank for the core and the two blocks'
    offset + 3 rank + 1 and + 2, as a tensor-parallel run draws independent
    masks per rank."""

    def __init__(self, shape: ParallelShape, seed: int, rank: int, offset: int = 0):
        self.shape, self.seed = shape, seed
        self.off = offset + 3 * rank

    def matmul(self, a, b):
        import torch
        return torch.matmul(a, b)

    def core_fwd(self, q, k, v):
        import attention_core_gb300 as ac
        kw = dict(causal=True, p_drop=self.shape.p_drop, seed=self.seed, offset=self.off)
        o, lse = ac.fwd(q, k, v, **kw)
        return o, (q, k, v, o, lse, kw)

    def core_bwd(self, saved, do):
        import attention_core_gb300 as ac
        q, k, v, o, lse, kw = saved
        return ac.bwd_recompute(q, k, v, o, lse, do.contiguous(), **kw)

    def dal_fwd(self, x, r, gamma, beta, which):
        import attention_core_gb300 as ac
        kw = dict(p_drop=self.shape.p_drop, seed=self.seed, offset=self.off + which, eps=self.shape.eps)
        z, y, mean, rstd = ac.dropout_add_ln_fwd(x.contiguous(), r.contiguous(), gamma, beta, **kw)
        return z, y, (z, mean, rstd, gamma, kw)

    def dal_bwd(self, saved, dy, dz_next):
        import attention_core_gb300 as ac
        z, mean, rstd, gamma, kw = saved
        return ac.dropout_add_ln_bwd(dy.contiguous(), z, mean, rstd, gamma, dz_next=dz_next.contiguous(), **kw)

    def gelu_fwd(self, x):
        import attention_core_gb300 as ac
        return ac.gelu_fwd(x.contiguous())

    def gelu_bwd(self, x, dy):
        import attention_core_gb300 as ac
        return ac.gelu_bwd(x, dy.contiguous())
