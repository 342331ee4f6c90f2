"""Pins for the CPU oracle of the dropout + residual add + layer norm block
(no GPU): torch's fp64 layer norm and autograd, the oracle's own mask under
autograd, central differences, the mask mapping stated a second time, and
row invariants of the normalised output."""
import numpy as np
import pytest
import torch

import oracle
from attention_core_gb300.inputs import dal_inputs
from tests.test_oracle import _philox_from_spec


def _torch_reference(t, pr, z_factor=None):
    """fp64 autograd: z = r + x * Z, y = layer_norm(z); loss = <dy, y> + <dz_next, z>."""
    x = t.x.double().requires_grad_(True)
    r = t.residual.double().requires_grad_(True)
    gm = t.gamma.double().requires_grad_(True)
    bt = t.beta.double().requires_grad_(True)
    z = r + (x if z_factor is None else x * z_factor)
    y = torch.nn.functional.layer_norm(z, (pr.hidden,), gm, bt, eps=pr.eps)
    ((y * t.dy.double()).sum() + (z * t.dz_next.double()).sum()).backward()
    return (z.detach().numpy(), y.detach().numpy(), x.grad.numpy(), r.grad.numpy(), gm.grad.numpy(),
            bt.grad.numpy())


@pytest.mark.parametrize("shape", [(7, 64), (3, 200), (16, 1024)])
def test_p0_equals_torch_layer_norm(shape):
    n, h = shape
    pr = oracle.DalProblem(n_rows=n, hidden=h)
    t = dal_inputs(n, h, seed=n + h)
    z, y, mean, rstd = oracle.dal_fwd(pr, t.x, t.residual, t.gamma, t.beta)
    dx, dres, dg, db = oracle.dal_bwd(pr, t.x, t.residual, t.gamma, t.dy, t.dz_next)
    rz, ry, rdx, rdr, rdg, rdb = _torch_reference(t, pr)
    for a, b in ((z, rz), (y, ry), (dx, rdx), (dres, rdr), (dg, rdg), (db, rdb)):
        assert np.max(np.abs(a - b)) < 1e-10
    zz = rz
    assert np.max(np.abs(mean - zz.mean(1))) < 1e-12
    assert np.max(np.abs(rstd - 1 / np.sqrt(zz.var(1) + pr.eps))) < 1e-9


def test_dropout_matches_autograd_with_oracle_mask():
    n, h = 9, 136
    pr = oracle.DalProblem(n_rows=n, hidden=h, p_drop=0.3, seed=4242, offset=17)
    t = dal_inputs(n, h, seed=3)
    m = oracle.dal_mask(pr)
    assert 0 < (m == 0).sum() < m.size
    zf = torch.from_numpy(m / (1 - oracle.drop_threshold16(0.3) / 65536))
    z, y, _, _ = oracle.dal_fwd(pr, t.x, t.residual, t.gamma, t.beta)
    dx, dres, dg, db = oracle.dal_bwd(pr, t.x, t.residual, t.gamma, t.dy, t.dz_next)
    rz, ry, rdx, rdr, rdg, rdb = _torch_reference(t, pr, zf)
    for a, b in ((z, rz), (y, ry), (dx, rdx), (dres, rdr), (dg, rdg), (db, rdb)):
        assert np.max(np.abs(a - b)) < 1e-10
    # without the residual-path gradient, d_residual is the layer norm's gradient alone
    dx0, dres0, _, _ = oracle.dal_bwd(pr, t.x, t.residual, t.gamma, t.dy, None)
    assert np.max(np.abs((dres - dres0) - t.dz_next.double().numpy())) < 1e-12


def test_gradients_by_central_differences():
    n, h = 3, 16
    pr = oracle.DalProblem(n_rows=n, hidden=h, p_drop=0.25, seed=9)
    t = dal_inputs(n, h, seed=4)
    x, r = t.x.double().numpy().copy(), t.residual.double().numpy().copy()
    gm, bt = t.gamma.double().numpy().copy(), t.beta.double().numpy().copy()
    dy, dzn = t.dy.double().numpy(), t.dz_next.double().numpy()
    dx, dres, dg, db = oracle.dal_bwd(pr, x, r, gm, dy, dzn)

    def loss():
        z, y, _, _ = oracle.dal_fwd(pr, x, r, gm, bt)
        return float((y * dy).sum() + (z * dzn).sum())

    step = 1e-5
    for name, arr, grad in (("x", x, dx), ("r", r, dres), ("gamma", gm, dg), ("beta", bt, db)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            orig = arr[idx]
            arr[idx] = orig + step
            lp = loss()
            arr[idx] = orig - step
            lm = loss()
            arr[idx] = orig
            fd[idx] = (lp - lm) / (2 * step)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(grad)), 1e-30)
        assert err < 1e-6, (name, err)


def test_mask_mapping_follows_definition():
    """Element (row, col) uses counter (col // 8, row, 0xFFFFFFFF, offset) and
    half (col % 8) % 2 of word (col % 8) // 2; kept iff the draw >= thr."""
    pr = oracle.DalProblem(n_rows=40, hidden=96, p_drop=0.4, seed=0xFEDCBA9876543210, offset=3)
    thr = oracle.drop_threshold16(0.4)
    key = [pr.seed & 0xFFFFFFFF, pr.seed >> 32]
    rng = np.random.default_rng(5)
    for _ in range(300):
        row, col = int(rng.integers(0, 40)), int(rng.integers(0, 96))
        w = _philox_from_spec([col // 8, row, 0xFFFFFFFF, pr.offset], key)
        e = col % 8
        draw = (w[e // 2] >> (16 * (e % 2))) & 0xFFFF
        assert oracle.dal_keep(pr, row, col) == int(draw >= thr)
    # p = 0 keeps everything; the drop rate at p = 0.4 is close to p_eff
    assert oracle.dal_mask(oracle.DalProblem(n_rows=4, hidden=64)).all()
    m = oracle.dal_mask(pr)
    p_eff = thr / 65536
    assert abs((1 - m.mean()) - p_eff) < 5 * np.sqrt(p_eff * (1 - p_eff) / m.size)


def test_normalised_rows_have_zero_mean_and_unit_scale():
    n, h = 5, 512
    pr = oracle.DalProblem(n_rows=n, hidden=h, p_drop=0.1, seed=2, eps=1e-5)
    t = dal_inputs(n, h, seed=6)
    z, y, mean, rstd = oracle.dal_fwd(pr, t.x, t.residual, t.gamma, t.beta)
    xhat = (y - t.beta.double().numpy()) / t.gamma.double().numpy()
    assert np.max(np.abs(xhat.mean(1))) < 1e-12
    var = z.var(1)
    assert np.max(np.abs(xhat.var(1) - var / (var + pr.eps))) < 1e-12
    # dbeta is the column sum of dy, dgamma of dy * xhat
    dx, dres, dg, db = oracle.dal_bwd(pr, t.x, t.residual, t.gamma, t.dy)
    assert np.max(np.abs(db - t.dy.double().numpy().sum(0))) < 1e-10
    assert np.max(np.abs(dg - (t.dy.double().numpy() * xhat).sum(0))) < 1e-9
