"""Sequence-parallel converters on CPU ranks (gloo, world size 2 and 4).

The layer of attention_core_gb300.seqpar, run sequence- and tensor-parallel
over t processes, against a single-process fp64 composition of the same layer
(the oracle's attention core, dropout + residual add + layer norm and GeLU,
fp64 GEMMs); and the collectives' bytes: the four all-gathers and four
reduce-scatters of a sequence-parallel layer (forward and backward) send what
the four all-reduces of the tensor-parallel-only layer send ("Reducing
Activation Recomputation in Large Transformer Models", Key takeaways, second
bullet), with the backward's second gathers of the kept inputs on top (fifth
bullet).  Dropout is off (p = 0): ranks holding different tokens or heads
draw their own masks, so only p = 0 makes every rank count equal to one
process.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from attention_core_gb300 import seqpar

SHAPE = dict(b=2, s=24, h=32, a=4, d=8, ffn=64)


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


class OracleOps:
    """fp64 region arithmetic for the CPU ranks: the oracle's functions (the
    attention core, the dropout + layer norm block, GeLU) and fp64 products."""

    def __init__(self, shape):
        self.shape = shape

    def matmul(self, a, b):
        return a @ b

    def core_fwd(self, q, k, v):
        import oracle
        b, a, s, d = q.shape
        pr = oracle.Problem(b=b, h_q=a, h_kv=a, s=s, d=d, causal=True, p_drop=0.0, seed=0)
        o, _ = oracle.fwd(pr, q.numpy(), k.numpy(), v.numpy())
        return torch.from_numpy(np.ascontiguousarray(o)), (pr, q, k, v)

    def core_bwd(self, saved, do):
        import oracle
        pr, q, k, v = saved
        grads = oracle.bwd(pr, q.numpy(), k.numpy(), v.numpy(), do.contiguous().numpy())
        return tuple(torch.from_numpy(np.ascontiguousarray(g)) for g in grads)

    def dal_fwd(self, x, r, gamma, beta, which):
        import oracle
        pr = oracle.DalProblem(n_rows=x.shape[0], hidden=x.shape[1], p_drop=0.0, eps=self.shape.eps, seed=0)
        z, y, _, _ = oracle.dal_fwd(pr, x.numpy(), r.numpy(), gamma.numpy(), beta.numpy())
        return torch.from_numpy(z), torch.from_numpy(y), (pr, x, r, gamma)

    def dal_bwd(self, saved, dy, dz_next):
        import oracle
        pr, x, r, gamma = saved
        out = oracle.dal_bwd(pr, x.numpy(), r.numpy(), gamma.numpy(), dy.contiguous().numpy(),
                             dz_next.contiguous().numpy())
        return tuple(torch.from_numpy(np.ascontiguousarray(o)) for o in out)

    def gelu_fwd(self, x):
        import oracle
        return torch.from_numpy(oracle.gelu(x.numpy()))

    def gelu_bwd(self, x, dy):
        import oracle
        return dy * torch.from_numpy(oracle.gelu_grad(x.numpy()))


class SoloComm:
    """One process: every collective is the identity."""
    rank, world = 0, 1

    def all_gather(self, x, kind="all_gather"):
        return x

    def reduce_scatter(self, x):
        return x

    def all_reduce(self, x):
        return x

    def all_gather_async(self, x, kind="all_gather"):
        class H:
            def wait(self_inner):
                return x
        return H()


def _inputs(shape):
    g = torch.Generator().manual_seed(17)
    ad = shape.a * shape.d

    def w(r, c):
        return 0.2 * torch.randn((r, c), generator=g, dtype=torch.float64)

    wts = {"wqkv": w(shape.h, 3 * ad), "wo": w(ad, shape.h), "w1": w(shape.h, shape.ffn),
           "w2": w(shape.ffn, shape.h),
           "gamma1": 1 + 0.1 * torch.randn(shape.h, generator=g, dtype=torch.float64),
           "beta1": 0.1 * torch.randn(shape.h, generator=g, dtype=torch.float64),
           "gamma2": 1 + 0.1 * torch.randn(shape.h, generator=g, dtype=torch.float64),
           "beta2": 0.1 * torch.randn(shape.h, generator=g, dtype=torch.float64)}
    acts = [torch.randn((shape.n, shape.h), generator=g, dtype=torch.float64) for _ in range(4)]
    return wts, acts


def _reference(shape1):
    wts, (y_in, r_in, dy2, dz2) = _inputs(shape1)
    ops = OracleOps(shape1)
    y2, z2, ctx = seqpar.forward(shape1, wts, SoloComm(), y_in, r_in, ops, sequence_parallel=False)
    grads = seqpar.backward(shape1, wts, SoloComm(), ctx, dy2, dz2, ops)
    return {"y2": y2, "z2": z2, **grads}


def _worker(rank, world, port, sp, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shape = seqpar.ParallelShape(**SHAPE, t=world)
        full, (y_in, r_in, dy2, dz2) = _inputs(shape)
        wts = seqpar.shard_weights(full, shape, rank)
        m = shape.n // world
        sl = slice(rank * m, (rank + 1) * m) if sp else slice(None)
        comm = seqpar.Comm()
        events = []
        ops = OracleOps(shape)
        y2, z2, ctx = seqpar.forward(shape, wts, comm, y_in[sl].clone(), r_in[sl].clone(), ops, sequence_parallel=sp)
        grads = seqpar.backward(shape, wts, comm, ctx, dy2[sl].clone(), dz2[sl].clone(), ops, events=events)
        out[rank] = {"y2": y2.numpy(), "z2": z2.numpy(), **{k: v.numpy() for k, v in grads.items()},
                     "sent": dict(comm.sent), "log": list(comm.log), "events": events}
    finally:
        dist.destroy_process_group()


def _run(world, sp):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, sp, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        return dict(out)


@pytest.fixture(scope="module")
def reference():
    import oracle
    oracle.build()
    return _reference(seqpar.ParallelShape(**SHAPE, t=1))


def _assemble(res, world, shape, sp):
    """Whole-layer tensors from the ranks' pieces."""
    m = shape.n // world
    ad, al, fl = shape.a * shape.d, shape.a * shape.d // world, shape.ffn // world
    got = {}
    for k in ("y2", "z2", "y_in", "r_in"):
        got[k] = np.concatenate([res[r][k] for r in range(world)]) if sp else res[0][k]
    wqkv = np.zeros((shape.h, 3 * ad))
    wo = np.zeros((ad, shape.h))
    w1 = np.zeros((shape.h, shape.ffn))
    w2 = np.zeros((shape.ffn, shape.h))
    for r in range(world):
        for i in range(3):
            wqkv[:, i * ad + r * al:i * ad + (r + 1) * al] = res[r]["wqkv"][:, i * al:(i + 1) * al]
        wo[r * al:(r + 1) * al] = res[r]["wo"]
        w1[:, r * fl:(r + 1) * fl] = res[r]["w1"]
        w2[r * fl:(r + 1) * fl] = res[r]["w2"]
    got.update(wqkv=wqkv, wo=wo, w1=w1, w2=w2)
    for k in ("gamma1", "beta1", "gamma2", "beta2"):
        # sequence-split: each rank's sum over its own tokens; replicated: every rank has the whole sum
        got[k] = sum(res[r][k] for r in range(world)) if sp else res[0][k]
    return got


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("sp", [True, False], ids=["sequence_parallel", "tensor_parallel_only"])
def test_parallel_layer_matches_single_process(world, sp, reference):
    shape = seqpar.ParallelShape(**SHAPE, t=world)
    res = _run(world, sp)
    got = _assemble(res, world, shape, sp)
    for k, ref in reference.items():
        r = ref.numpy()
        assert np.allclose(got[k], r, rtol=1e-9, atol=1e-9 * np.abs(r).max()), k
    if not sp:
        for r in range(1, world):     # replicated regions agree across ranks
            for k in ("y2", "z2", "y_in", "r_in"):
                assert np.array_equal(res[r][k], res[0][k]), k


@pytest.mark.parametrize("world", [2, 4])
def test_converters_move_the_bytes_of_the_all_reduces(world):
    """4 all-gathers + 4 reduce-scatters (sequence-parallel) send exactly the
    bytes of 4 all-reduces (tensor-parallel only), per rank; the backward's
    two second gathers of the kept inputs come on top."""
    shape = seqpar.ParallelShape(**SHAPE, t=world)
    sp = _run(world, True)
    tp = _run(world, False)
    n_bytes = shape.n * shape.h * 8                    # one [n, h] fp64 tensor
    for r in range(world):
        kinds = [k for k, _ in sp[r]["log"]]
        assert kinds.count("all_gather") == 4 and kinds.count("reduce_scatter") == 4
        assert kinds.count("regather") == 2 and "all_reduce" not in kinds
        assert [k for k, _ in tp[r]["log"]].count("all_reduce") == 4
        conv = sp[r]["sent"]["all_gather"] + sp[r]["sent"]["reduce_scatter"]
        assert conv == tp[r]["sent"]["all_reduce"] == 4 * 2 * (world - 1) * n_bytes // world
        assert sp[r]["sent"]["regather"] == 2 * (world - 1) * n_bytes // world


def test_backward_gather_overlaps_the_input_gradient_product():
    """The kept input's second all-gather is started before the input
    gradient's product and waited for after it; the weight gradient's product
    runs before the input gradient's reduce-scatter is joined."""
    res = _run(2, True)
    order = ["gather_started", "dx_product_done", "gather_done", "dw_product_done"]
    for r in res.values():
        assert r["events"] == order * 2
