"""GPU parity of the layer shard around the core (attention_core_gb300.layer)
against an fp64 CPU composition of the oracles: the attention core, the
dropout + residual add + layer norm block and GeLU, with the GEMMs as plain
fp64 products.  The reference rounds to bf16 wherever the layer stores a bf16
tensor, so each step sees the same kind of input on both sides.

Tolerance: each of the layer's stored bf16 tensors carries a rounding of at
most 2^-9 relative, and a gradient passes through up to eight of them between
an input and an output, so the bar is 2e-2 (the core's own bar, 1e-2, plus
those roundings), row-relative as in the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
from attention_core_gb300 import layer
from tests.gpu_util import row_rel_err, to_np

pytestmark = pytest.mark.gpu
LAYER_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _bf(x):
    """Round fp64 values to bf16 (nearest even) and back."""
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def _heads(x2d, sh):
    return x2d.reshape(sh.b, sh.s, sh.a, sh.d).transpose(0, 2, 1, 3)


def _tokens(x4d, sh):
    return x4d.transpose(0, 2, 1, 3).reshape(sh.n, sh.a * sh.d)


def _reference(sh, w, y_in, r_in, dy2, dz2, seed):
    """fp64 forward and backward of the layer, bf16 at the stored tensors."""
    ad = sh.a * sh.d
    W = {k: v.double().cpu().numpy() for k, v in w.items()}
    core = oracle.Problem(b=sh.b, h_q=sh.a, h_kv=sh.a, s=sh.s, d=sh.d, causal=True, p_drop=sh.p_drop,
                          seed=seed, offset=0)
    dal1 = oracle.DalProblem(n_rows=sh.n, hidden=sh.h, p_drop=sh.p_drop, eps=sh.eps, seed=seed, offset=1)
    dal2 = oracle.DalProblem(n_rows=sh.n, hidden=sh.h, p_drop=sh.p_drop, eps=sh.eps, seed=seed, offset=2)
    qkv = _bf(y_in @ W["wqkv"])
    q, k, v = (np.ascontiguousarray(_heads(qkv[:, i * ad:(i + 1) * ad], sh)) for i in range(3))
    o, _ = oracle.fwd(core, q, k, v)
    o2 = _bf(_tokens(o, sh))
    attn = _bf(o2 @ W["wo"])
    z1, y1, _, _ = oracle.dal_fwd(dal1, attn, r_in, W["gamma1"], W["beta1"])
    z1, y1 = _bf(z1), _bf(y1)
    m1 = _bf(y1 @ W["w1"])
    g = _bf(oracle.gelu(m1))
    m2 = _bf(g @ W["w2"])
    z2, y2, _, _ = oracle.dal_fwd(dal2, m2, z1, W["gamma2"], W["beta2"])
    dm2, dz1, dgamma2, dbeta2 = oracle.dal_bwd(dal2, m2, z1, W["gamma2"], dy2, dz2)
    dm2, dz1 = _bf(dm2), _bf(dz1)
    dg = _bf(dm2 @ W["w2"].T)
    dw2 = g.T @ dm2
    dm1 = _bf(dg * oracle.gelu_grad(m1))
    dy1 = _bf(dm1 @ W["w1"].T)
    dw1 = y1.T @ dm1
    dattn, dr_in, dgamma1, dbeta1 = oracle.dal_bwd(dal1, attn, r_in, W["gamma1"], dy1, dz1)
    dattn = _bf(dattn)
    do2 = _bf(dattn @ W["wo"].T)
    dwo = o2.T @ dattn
    dq, dk, dv = oracle.bwd(core, q, k, v, np.ascontiguousarray(_heads(do2, sh)))
    dqkv = np.concatenate([_bf(_tokens(t, sh)) for t in (dq, dk, dv)], axis=1)
    dy_in = dqkv @ W["wqkv"].T
    dwqkv = y_in.T @ dqkv
    return {"y2": y2, "z2": z2, "y_in": dy_in, "r_in": dr_in, "wqkv": dwqkv, "wo": dwo, "w1": dw1,
            "w2": dw2, "gamma1": dgamma1, "beta1": dbeta1, "gamma2": dgamma2, "beta2": dbeta2}


@pytest.mark.parametrize("dims", [(1, 256, 512, 4, 64, 1024), (2, 130, 384, 3, 128, 768)],
                         ids=lambda t: "b{}_s{}_h{}_a{}_d{}_f{}".format(*t))
def test_layer_matches_composed_oracles(dims):
    b, s, h, a, d, f = dims
    sh = layer.LayerShape(b=b, s=s, h=h, a=a, d=d, ffn=f, p_drop=0.1)
    dev = torch.device("cuda:0")
    w = layer.init_weights(sh, seed=5, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(9)
    y_in, r_in, dy2, dz2 = (torch.randn((sh.n, h), generator=gen).to(torch.bfloat16) for _ in range(4))
    seed = 31337
    y2, z2, ctx = layer.forward(sh, w, y_in.to(dev), r_in.to(dev), seed=seed)
    grads = layer.backward(sh, w, ctx, dy2.to(dev), dz2.to(dev))
    torch.cuda.synchronize()
    ref = _reference(sh, w, *(t.double().numpy() for t in (y_in, r_in, dy2, dz2)), seed=seed)
    got = {"y2": y2, "z2": z2, **grads}
    errs = {}
    for name, r in ref.items():
        g = to_np(got[name])
        errs[name] = row_rel_err(g[None] if g.ndim == 1 else g, r[None] if r.ndim == 1 else r)
    assert all(e <= LAYER_TOL for e in errs.values()), errs


def test_stored_core_baseline_computes_the_same_layer():
    """The no-recomputation baseline core of the layer study (it keeps the
    dense probabilities) computes the same layer as this library's core: at
    p = 0 (where its own dropout mask plays no part) both match the composed
    oracles."""
    b, s, h, a, d, f = 1, 256, 512, 4, 64, 1024
    sh = layer.LayerShape(b=b, s=s, h=h, a=a, d=d, ffn=f, p_drop=0.0)
    dev = torch.device("cuda:0")
    w = layer.init_weights(sh, seed=5, device=dev)
    gen = torch.Generator(device="cpu").manual_seed(10)
    y_in, r_in, dy2, dz2 = (torch.randn((sh.n, h), generator=gen).to(torch.bfloat16) for _ in range(4))
    seed = 99
    stored = layer.StoredCore(sh)
    y2, z2, ctx = layer.forward(sh, w, y_in.to(dev), r_in.to(dev), seed=seed, stored=stored)
    grads = layer.backward(sh, w, ctx, dy2.to(dev), dz2.to(dev))
    full = layer.backward_full(sh, w, y_in.to(dev), r_in.to(dev), dy2.to(dev), dz2.to(dev), seed=seed)
    torch.cuda.synchronize()
    ref = _reference(sh, w, *(t.double().numpy() for t in (y_in, r_in, dy2, dz2)), seed=seed)
    for got in ({"y2": y2, "z2": z2, **grads}, full):
        errs = {}
        for name, r in ref.items():
            if name not in got:
                continue
            g = to_np(got[name])
            errs[name] = row_rel_err(g[None] if g.ndim == 1 else g, r[None] if r.ndim == 1 else r)
        assert all(e <= LAYER_TOL for e in errs.values()), errs
