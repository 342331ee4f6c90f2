"""GPU parity of the dropout + residual add + layer norm block against the CPU
oracle: several row lengths (one to several 8-column vectors per thread,
ragged against the thread count), p = 0 and p > 0, with and without a
residual-path gradient; the dropout mask read out bit-exactly through probe
inputs; bit-reproducible dgamma and dbeta."""
import numpy as np
import pytest
import torch

import attention_core_gb300 as ac
import oracle
from attention_core_gb300.inputs import dal_inputs, dal_mask_probe
from tests.gpu_util import TOL, row_rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(t, p_drop, seed, offset=0, eps=1e-5, with_dzn=True):
    dev = torch.device("cuda:0")
    x, r, dy, dzn = (v.to(dev) for v in (t.x, t.residual, t.dy, t.dz_next))
    g, b = t.gamma.to(dev), t.beta.to(dev)
    kw = dict(p_drop=p_drop, seed=seed, offset=offset, eps=eps)
    z, y, mean, rstd = ac.dropout_add_ln_fwd(x, r, g, b, **kw)
    dx, dres, dg, db = ac.dropout_add_ln_bwd(dy, z, mean, rstd, g, dz_next=dzn if with_dzn else None, **kw)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in dict(z=z, y=y, mean=mean, rstd=rstd, dx=dx, dres=dres, dg=dg,
                                           db=db).items()}


# (n_rows, hidden, p_drop, with dz_next)
CASES = [
    (64, 1024, 0.1, True),
    (37, 4608, 0.1, True),       # 22B-layer hidden size, ragged vs 2048 columns per pass
    (130, 12288, 0.1, False),    # 175B-layer hidden size
    (5, 20480, 0.1, True),       # 530B-layer hidden size
    (9, 2056, 0.0, True),        # one vector past a full pass
    (1, 8, 0.3, True),           # one vector
    (300, 512, 0.5, False),      # many rows per CTA
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"n{c[0]}_h{c[1]}_p{c[2]}_{'dzn' if c[3] else 'nodzn'}")
def test_dal_matches_oracle(case):
    n, h, p, with_dzn = case
    seed = 1000 + n + h
    t = dal_inputs(n, h, seed=n * 31 + h)
    out = _run(t, p, seed, with_dzn=with_dzn)
    pr = oracle.DalProblem(n_rows=n, hidden=h, p_drop=p, seed=seed)
    z, y, mean, rstd = oracle.dal_fwd(pr, t.x, t.residual, t.gamma, t.beta)
    dx, dres, dg, db = oracle.dal_bwd(pr, t.x, t.residual, t.gamma, t.dy,
                                      t.dz_next if with_dzn else None)
    errs = {"z": row_rel_err(out["z"], z), "y": row_rel_err(out["y"], y),
            "dx": row_rel_err(out["dx"], dx), "dres": row_rel_err(out["dres"], dres),
            "dgamma": row_rel_err(out["dg"][None], dg[None]), "dbeta": row_rel_err(out["db"][None], db[None])}
    assert all(e <= TOL for e in errs.values()), errs
    # statistics: the mean within 1% of a standard deviation, rstd within 1%
    assert np.max(np.abs(out["mean"] - mean) * rstd) <= TOL
    assert np.max(np.abs(out["rstd"] / rstd - 1)) <= TOL


@pytest.mark.parametrize("shape", [(3, 1024), (2, 12288)])
def test_dal_mask_bit_exact(shape):
    """x = 1, residual = 0: z is the keep factor, so z != 0 exactly where kept."""
    n, h = shape
    t = dal_mask_probe(n, h)
    out = _run(t, 0.3, seed=77, offset=5)
    pr = oracle.DalProblem(n_rows=n, hidden=h, p_drop=0.3, seed=77, offset=5)
    m = np.array([[oracle.dal_keep(pr, i, c) for c in range(h)] for i in range(n)], dtype=np.uint8)
    assert ((out["z"] != 0).astype(np.uint8) == m).all()
    # and the backward applies the same mask: dx = 0 exactly where dropped
    t2 = dal_inputs(n, h, seed=1)
    out2 = _run(t2, 0.3, seed=77, offset=5)
    assert ((out2["dx"] == 0) >= (m == 0)).all() and (out2["dx"][m == 0] == 0).all()


def test_dal_bit_reproducible():
    t = dal_inputs(200, 4096, seed=8)
    a = _run(t, 0.1, seed=3)
    b = _run(t, 0.1, seed=3)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
