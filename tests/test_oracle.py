"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: published
known-answer vectors, the pages' worked example, textbook attention from an
independent library routine, finite differences, closed forms and
statistics.  A plausible slip in the oracle -- a dropped term, a wrong sign
or index, a transposed operand, a wrong head mapping -- fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_core_gb300.inputs import random_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- Philox ---

def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = [int(x, 16) for x in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,expect", _kat_rows())
def test_philox_known_answers(ctr, key, expect):
    assert list(oracle.philox4x32_10(ctr, key)) == expect


def _philox_from_spec(ctr, key, rounds=10):
    """Second, independent statement of the SC'11 round function."""
    m = (0xD2511F53, 0xCD9E8D57)
    w = (0x9E3779B9, 0xBB67AE85)
    x = list(ctr)
    k = list(key)
    for _ in range(rounds):
        p0 = m[0] * x[0]
        p1 = m[1] * x[2]
        x = [((p1 >> 32) ^ x[1] ^ k[0]) & 0xFFFFFFFF, p1 & 0xFFFFFFFF,
             ((p0 >> 32) ^ x[3] ^ k[1]) & 0xFFFFFFFF, p0 & 0xFFFFFFFF]
        k = [(k[0] + w[0]) & 0xFFFFFFFF, (k[1] + w[1]) & 0xFFFFFFFF]
    return x


def test_philox_matches_second_statement():
    rng = np.random.default_rng(7)
    for _ in range(200):
        ctr = [int(x) for x in rng.integers(0, 2**32, size=4, dtype=np.uint64)]
        key = [int(x) for x in rng.integers(0, 2**32, size=2, dtype=np.uint64)]
        assert list(oracle.philox4x32_10(ctr, key)) == _philox_from_spec(ctr, key)


def test_drop_threshold_closed_form():
    assert oracle.drop_threshold(0.0) == 0
    assert oracle.drop_threshold(0.1) == 26            # round(25.6)
    assert oracle.drop_threshold(0.5) == 128
    assert oracle.drop_threshold(0.99999) == 255       # capped: some draw always survives
    assert oracle.drop_threshold(0.001) == 0           # below half a step: no dropout
    assert oracle.drop_threshold(-1.0) == 0
    # the dropout + layer norm block's 16-bit reading
    assert oracle.drop_threshold16(0.1) == 6554        # round(6553.6)
    assert oracle.drop_threshold16(0.99999) == 65535


def test_mask_mapping_follows_header_definition():
    """Element (i, j) of head bh uses counter (j//16, i, bh, offset), key
    (seed lo, seed hi), and byte (j%16)%4 of output word (j%16)//4."""
    pr = oracle.Problem(b=2, h_q=3, h_kv=3, s=64, d=16, p_drop=0.25,
                        seed=0x0123456789ABCDEF, offset=77)
    rng = np.random.default_rng(3)
    key = [pr.seed & 0xFFFFFFFF, pr.seed >> 32]
    for _ in range(300):
        bh, i, j = int(rng.integers(0, 6)), int(rng.integers(0, 64)), int(rng.integers(0, 64))
        w = _philox_from_spec([j // 16, i, bh, pr.offset], key)
        e = j % 16
        draw = (w[e // 4] >> (8 * (e % 4))) & 0xFF
        assert oracle.draw8(pr, bh, i, j) == draw
        assert oracle.keep(pr, bh, i, j) == int(draw >= 64)


def test_mask_statistics():
    """Drop rate within 5 sigma of p_eff; 8-bit draws uniform (chi^2, 256 bins)."""
    pr = oracle.Problem(b=1, h_q=4, h_kv=4, s=1024, d=64, causal=False, p_drop=0.1,
                        seed=987654321, offset=5)
    masks = np.concatenate([oracle.mask_rows(pr, bh, 0, 1024).ravel() for bh in range(4)])
    n = masks.size
    p_eff = 26 / 256
    drop = 1.0 - masks.mean()
    sigma = math.sqrt(p_eff * (1 - p_eff) / n)
    assert abs(drop - p_eff) < 5 * sigma, (drop, p_eff, sigma)
    draws = np.array([oracle.draw8(pr, 0, i, j) for i in range(64) for j in range(256)])
    hist = np.bincount(draws, minlength=256)
    expected = len(draws) / 256
    chi2 = float(((hist - expected) ** 2 / expected).sum())
    # 255 degrees of freedom: mean 255, sd ~22.6; 5 sigma band
    assert 255 - 5 * 22.6 < chi2 < 255 + 5 * 22.6, chi2


def test_mask_independent_of_inputs_and_depends_on_stream():
    base = dict(b=1, h_q=2, h_kv=2, s=32, d=16, p_drop=0.3, seed=11, offset=0)
    m0 = oracle.mask_rows(oracle.Problem(**base), 1, 0, 32)
    m1 = oracle.mask_rows(oracle.Problem(**{**base, "offset": 1}), 1, 0, 32)
    m2 = oracle.mask_rows(oracle.Problem(**{**base, "seed": 12}), 1, 0, 32)
    m3 = oracle.mask_rows(oracle.Problem(**base), 0, 0, 32)
    assert (m0 != m1).any() and (m0 != m2).any() and (m0 != m3).any()
    # causal: keys above the diagonal are reported as 0
    assert (np.triu(m0, 1) == 0).all()


# ------------------------------------------------------------ stored bytes -

def test_stored_bytes_worked_example():
    """The Llama 3 70B totals the activation-checkpointing page prints."""
    units = {"TB": 1e12, "GB": 1e9}
    with open(os.path.join(GOLDEN, "llama3_70b_activation_bytes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for name, s, b, hidden, heads, layers, val, unit in rows:
        s, b, hidden, heads, layers = int(s), int(b), int(hidden), int(heads), int(layers)
        pr = oracle.Problem(b=b, h_q=heads, h_kv=heads, s=s, d=hidden // heads)
        per_layer = oracle.stored_bytes(pr)["layer_" + name]
        total = per_layer * layers
        printed = float(val)
        decimals = len(val.split(".")[1]) if "." in val else 0
        assert round(total / units[unit], decimals) == printed, (name, total)
    # exact integers of the per-token forms, 34d + 5HT, 34d and 2d
    pr = oracle.Problem(b=1, h_q=64, h_kv=64, s=8192, d=128)
    sb = oracle.stored_bytes(pr)
    assert sb["layer_none"] * 80 == 1_900_523_028_480
    assert sb["layer_selective"] * 80 == 182_536_110_080
    assert sb["layer_full"] * 80 == 10_737_418_240


def test_stored_bytes_layer_formula_and_core_terms():
    """sbh(34 + 5as/h) per layer; the core keeps Q, K, V, O in bf16 plus LSE."""
    pr = oracle.Problem(b=2, h_q=12, h_kv=4, s=2048, d=128)
    sb = oracle.stored_bytes(pr)
    s, b, a, d = 2048, 2, 12, 128
    h = a * d
    assert sb["layer_none"] == s * b * h * 34 + s * b * h * 5 * a * s // h
    assert sb["layer_none"] - sb["layer_selective"] == sb["core_scores_avoided"]
    assert sb["core_kept"] == 2 * (2 * b * 12 * s * d + 2 * b * 4 * s * d)
    assert sb["core_recompute_state"] == 4 * b * a * s + 16


def test_stored_bytes_cross_attention_core_terms():
    """With s_kv keys the core avoids 5 a s s_kv b score bytes and keeps Q, O
    (s rows) and K, V (s_kv rows); the layer terms stay those of s tokens."""
    s, skv, b, a, akv, d = 512, 1536, 3, 8, 2, 64
    sq = oracle.stored_bytes(oracle.Problem(b=b, h_q=a, h_kv=akv, s=s, d=d))
    sx = oracle.stored_bytes(oracle.Problem(b=b, h_q=a, h_kv=akv, s=s, d=d, s_kv=skv))
    assert sx["core_scores_avoided"] == 5 * a * s * skv * b
    assert sx["core_kept"] == 2 * b * d * (2 * a * s + 2 * akv * skv)
    for name in ("layer_none", "layer_selective", "layer_full", "core_recompute_state"):
        assert sx[name] == sq[name], name


# ------------------------------------------------------ softmax invariants -

def test_softmax_rows_and_lse():
    pr = oracle.Problem(b=1, h_q=2, h_kv=1, s=40, d=16, p_drop=0.2, seed=5)
    t = random_inputs(1, 2, 1, 40, 16, seed=1)
    for bh in range(2):
        S, P, M = oracle.head_matrices(pr, t.q, t.k, bh)
        assert np.all(P >= 0)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) < 1e-12
        assert np.all(P[np.triu_indices(40, 1)] == 0)
        _, lse = oracle.fwd(pr, t.q, t.k, t.v)
        for i in range(40):
            row = S[i, : i + 1]
            assert abs(lse[0, bh, i] - math.log(np.exp(row).sum())) < 1e-12


# ------------------------------------------------ textbook attention, p=0 --

def _torch_reference(t, pr, z=None):
    """fp64 autograd reference: SDPA for p = 0, else (softmax(S) * Z) @ V."""
    q = t.q.double().requires_grad_(True)
    k = t.k.double().requires_grad_(True)
    v = t.v.double().requires_grad_(True)
    scale = oracle.resolved_scale(pr)
    g = pr.h_q // pr.h_kv
    if z is None:
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=pr.causal, scale=scale, enable_gqa=(g > 1))
    else:
        kk = k.repeat_interleave(g, dim=1)
        vv = v.repeat_interleave(g, dim=1)
        s = (q @ kk.transpose(-1, -2)) * scale
        if pr.causal:
            s = s.masked_fill(torch.triu(torch.ones(pr.s, pr.keys, dtype=torch.bool), 1), -math.inf)
        o = (torch.softmax(s, dim=-1) * z) @ vv
    o.backward(t.dout.double())
    return o.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 2, 2, 33, 16), (2, 4, 2, 20, 8)])
def test_p0_equals_textbook_attention(causal, shape):
    b, hq, hkv, s, d = shape
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=causal)
    t = random_inputs(b, hq, hkv, s, d, seed=2)
    o, lse = oracle.fwd(pr, t.q, t.k, t.v)
    dq, dk, dv = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
    ro, rdq, rdk, rdv = _torch_reference(t, pr)
    for a, r in ((o, ro), (dq, rdq), (dk, rdk), (dv, rdv)):
        assert np.max(np.abs(a - r)) < 1e-11


# (b, h_q, h_kv, s queries, s_kv keys, d)
CROSS_SHAPES = [(1, 2, 2, 21, 37, 16), (2, 4, 2, 30, 9, 8), (1, 2, 1, 1, 19, 8)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", CROSS_SHAPES)
def test_p0_cross_attention_equals_textbook(causal, shape):
    """s_kv != s: textbook attention of s queries over s_kv keys (torch's causal
    mask for unequal lengths is also top-left aligned)."""
    b, hq, hkv, s, skv, d = shape
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=causal, s_kv=skv)
    t = random_inputs(b, hq, hkv, s, d, seed=21, s_kv=skv)
    assert tuple(t.k.shape) == (b, hkv, skv, d) and tuple(t.q.shape) == (b, hq, s, d)
    o, lse = oracle.fwd(pr, t.q, t.k, t.v)
    dq, dk, dv = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
    ro, rdq, rdk, rdv = _torch_reference(t, pr)
    for a, r in ((o, ro), (dq, rdq), (dk, rdk), (dv, rdv)):
        assert a.shape == r.shape
        assert np.max(np.abs(a - r)) < 1e-11
    # LSE against its definition, straight from the inputs
    q, k = t.q.double(), t.k.double()
    g = hq // hkv
    sc = (q @ k.repeat_interleave(g, dim=1).transpose(-1, -2)) * oracle.resolved_scale(pr)
    if causal:
        sc = sc.masked_fill(torch.triu(torch.ones(s, skv, dtype=torch.bool), 1), -math.inf)
    assert np.max(np.abs(lse - torch.logsumexp(sc, dim=-1).numpy())) < 1e-12


@pytest.mark.parametrize("shape", CROSS_SHAPES[:2])
def test_cross_attention_dropout_matches_autograd_with_oracle_mask(shape):
    b, hq, hkv, s, skv, d = shape
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=False, p_drop=0.3,
                        seed=77, offset=4, s_kv=skv)
    t = random_inputs(b, hq, hkv, s, d, seed=22, s_kv=skv)
    p_eff = oracle.drop_threshold(0.3) / 256
    z = np.zeros((b, hq, s, skv))
    for bh in range(b * hq):
        m = oracle.mask_rows(pr, bh, 0, s)
        assert m.shape == (s, skv)
        z[bh // hq, bh % hq] = m / (1 - p_eff)
    assert 0 < (z == 0).sum() < z.size
    o, _ = oracle.fwd(pr, t.q, t.k, t.v)
    dq, dk, dv = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
    ro, rdq, rdk, rdv = _torch_reference(t, pr, torch.from_numpy(z))
    for a, r in ((o, ro), (dq, rdq), (dk, rdk), (dv, rdv)):
        assert np.max(np.abs(a - r)) < 1e-11


def test_cross_attention_mask_is_the_self_attention_mask():
    """The keep decision of (i, j) depends only on (seed, offset, head, i, j),
    not on how many queries or keys the call has."""
    base = dict(b=1, h_q=2, h_kv=2, d=16, p_drop=0.3, seed=5, offset=2, causal=False)
    m_sq = oracle.mask_rows(oracle.Problem(s=40, **base), 1, 0, 40)
    m_x = oracle.mask_rows(oracle.Problem(s=25, s_kv=40, **base), 1, 0, 25)
    m_y = oracle.mask_rows(oracle.Problem(s=40, s_kv=13, **base), 1, 0, 40)
    assert (m_x == m_sq[:25]).all()
    assert (m_y == m_sq[:, :13]).all()


def test_p0_custom_scale():
    pr = oracle.Problem(b=1, h_q=2, h_kv=2, s=17, d=8, causal=True, scale=0.37)
    t = random_inputs(1, 2, 2, 17, 8, seed=4)
    o, _ = oracle.fwd(pr, t.q, t.k, t.v)
    ro = _torch_reference(t, pr)[0]
    assert np.max(np.abs(o - ro)) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_dropout_matches_autograd_with_oracle_mask(causal):
    b, hq, hkv, s, d = 1, 4, 2, 24, 8
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=causal, p_drop=0.3,
                        seed=2024, offset=9)
    t = random_inputs(b, hq, hkv, s, d, seed=3)
    p_eff = oracle.drop_threshold(0.3) / 256
    z = np.zeros((b, hq, s, s))
    for bh in range(b * hq):
        z[bh // hq, bh % hq] = oracle.mask_rows(pr, bh, 0, s) / (1 - p_eff)
    if not causal:
        assert (z > 0).sum() > s * s  # really non-causal
    o, _ = oracle.fwd(pr, t.q, t.k, t.v)
    dq, dk, dv = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
    ro, rdq, rdk, rdv = _torch_reference(t, pr, torch.from_numpy(z))
    for a, r in ((o, ro), (dq, rdq), (dk, rdk), (dv, rdv)):
        assert np.max(np.abs(a - r)) < 1e-11


# ------------------------------------------------------ finite differences -

def test_gradients_by_central_differences():
    """Central differences of the oracle's own forward (mask fixed by seed)."""
    b, hq, hkv, s, d = 1, 2, 1, 10, 8
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=0.3, seed=99)
    t = random_inputs(b, hq, hkv, s, d, seed=5)
    q, k, v = (x.double().numpy().copy() for x in (t.q, t.k, t.v))
    g = t.dout.double().numpy()
    dq, dk, dv = oracle.bwd(pr, q, k, v, g)

    def loss(qq, kk, vv):
        return float((oracle.fwd(pr, qq, kk, vv)[0] * g).sum())

    h = 1e-4
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            orig = x[idx]
            x[idx] = orig + h
            lp = loss(q, k, v)
            x[idx] = orig - h
            lm = loss(q, k, v)
            x[idx] = orig
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(grad)), 1e-30)
        assert err < 1e-7, (name, err)


def test_cross_attention_gradients_by_central_differences():
    b, hq, hkv, s, skv, d = 1, 2, 1, 6, 11, 8
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=False, p_drop=0.3, seed=98,
                        s_kv=skv)
    t = random_inputs(b, hq, hkv, s, d, seed=23, s_kv=skv)
    q, k, v = (x.double().numpy().copy() for x in (t.q, t.k, t.v))
    g = t.dout.double().numpy()
    dq, dk, dv = oracle.bwd(pr, q, k, v, g)

    def loss(qq, kk, vv):
        return float((oracle.fwd(pr, qq, kk, vv)[0] * g).sum())

    h = 1e-4
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            orig = x[idx]
            x[idx] = orig + h
            lp = loss(q, k, v)
            x[idx] = orig - h
            lm = loss(q, k, v)
            x[idx] = orig
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(grad)), 1e-30)
        assert err < 1e-7, (name, err)


# -------------------------------------------------- sampled-row entry points

def test_sampled_rows_agree_with_full():
    b, hq, hkv, s, d = 1, 4, 2, 70, 16
    for causal in (True, False):
        pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=causal, p_drop=0.15, seed=8)
        t = random_inputs(b, hq, hkv, s, d, seed=6)
        o, lse = oracle.fwd(pr, t.q, t.k, t.v)
        dq, dk, dv = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
        bh = np.array([0, 1, 3, 2, 3])
        rows = np.array([0, 69, 33, 5, 68])
        so, slse = oracle.fwd_rows(pr, t.q, t.k, t.v, bh, rows)
        sdq = oracle.dq_rows(pr, t.q, t.k, t.v, t.dout, bh, rows)
        ref_o = o.reshape(-1, s, d)[bh, rows]
        assert np.max(np.abs(so - ref_o)) < 1e-12
        assert np.max(np.abs(slse - lse.reshape(-1, s)[bh, rows])) < 1e-12
        assert np.max(np.abs(sdq - dq.reshape(-1, s, d)[bh, rows])) < 1e-12
        bkv = np.array([0, 1, 1, 0])
        krows = np.array([0, 69, 12, 40])
        sdk, sdv = oracle.dkdv_rows(pr, t.q, t.k, t.v, t.dout, bkv, krows)
        assert np.max(np.abs(sdk - dk.reshape(-1, s, d)[bkv, krows])) < 1e-12
        assert np.max(np.abs(sdv - dv.reshape(-1, s, d)[bkv, krows])) < 1e-12


def test_sampled_rows_agree_with_full_cross_attention():
    b, hq, hkv, s, skv, d = 1, 4, 2, 50, 83, 16
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=False, p_drop=0.15, seed=8,
                        s_kv=skv)
    t = random_inputs(b, hq, hkv, s, d, seed=24, s_kv=skv)
    o, lse = oracle.fwd(pr, t.q, t.k, t.v)
    dq, dk, dv = oracle.bwd(pr, t.q, t.k, t.v, t.dout)
    bh = np.array([0, 1, 3, 2])
    rows = np.array([0, 49, 33, 5])
    so, slse = oracle.fwd_rows(pr, t.q, t.k, t.v, bh, rows)
    sdq = oracle.dq_rows(pr, t.q, t.k, t.v, t.dout, bh, rows)
    assert np.max(np.abs(so - o.reshape(-1, s, d)[bh, rows])) < 1e-12
    assert np.max(np.abs(slse - lse.reshape(-1, s)[bh, rows])) < 1e-12
    assert np.max(np.abs(sdq - dq.reshape(-1, s, d)[bh, rows])) < 1e-12
    bkv = np.array([0, 1, 1])
    krows = np.array([0, 82, 60])
    sdk, sdv = oracle.dkdv_rows(pr, t.q, t.k, t.v, t.dout, bkv, krows)
    assert np.max(np.abs(sdk - dk.reshape(-1, skv, d)[bkv, krows])) < 1e-12
    assert np.max(np.abs(sdv - dv.reshape(-1, skv, d)[bkv, krows])) < 1e-12


def test_sampled_rows_p0_against_textbook():
    """Sampled entry points on a several-tile size with a ragged tail, p = 0."""
    b, hq, hkv, s, d = 1, 2, 1, 300, 32
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True)
    t = random_inputs(b, hq, hkv, s, d, seed=10)
    ro, rdq, rdk, rdv = _torch_reference(t, pr)
    bh = np.array([0, 1, 1])
    rows = np.array([299, 0, 150])
    so, _ = oracle.fwd_rows(pr, t.q, t.k, t.v, bh, rows)
    assert np.max(np.abs(so - ro.reshape(-1, s, d)[bh, rows])) < 1e-11
    sdq = oracle.dq_rows(pr, t.q, t.k, t.v, t.dout, bh, rows)
    assert np.max(np.abs(sdq - rdq.reshape(-1, s, d)[bh, rows])) < 1e-11
    sdk, sdv = oracle.dkdv_rows(pr, t.q, t.k, t.v, t.dout, np.array([0, 0]), np.array([0, 299]))
    assert np.max(np.abs(sdk - rdk.reshape(-1, s, d)[[0, 0], [0, 299]])) < 1e-11
    assert np.max(np.abs(sdv - rdv.reshape(-1, s, d)[[0, 0], [0, 299]])) < 1e-11


def test_fwd_mask_probe_reads_out_mask():
    """The forward probe inputs turn the oracle output into its own mask."""
    from attention_core_gb300.inputs import fwd_mask_probe
    b, hq, s, d = 1, 2, 40, 16
    pr = oracle.Problem(b=b, h_q=hq, h_kv=hq, s=s, d=d, causal=True, p_drop=0.3, seed=1)
    for w0 in (0, 16, 32):
        t = fwd_mask_probe(b, hq, hq, s, d, w0)
        o, _ = oracle.fwd(pr, t.q, t.k, t.v)
        for bh in range(hq):
            m = oracle.mask_rows(pr, bh, 0, s)
            width = min(d, s - w0)
            got = (o[0, bh, :, :width] != 0).astype(np.uint8)
            assert (got == m[:, w0:w0 + width]).all()


# ------------------------------------------------------ stored-output model

def test_stored_output_model_relation():
    """With the row statistic taken from the bf16-stored output, dS changes by
    exactly -P_ij (D_stored_i - D_exact_i); so dQ moves by -scale dD_i (P K)_i,
    dK by -scale sum_i P_ij dD_i q_i, and dV not at all.  Checked against
    pieces formed independently: the oracle's own O rounded to bf16 by torch,
    its dense P, and plain matrix products."""
    b, hq, hkv, s, d = 1, 2, 1, 24, 16
    base = dict(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=True, p_drop=0.25, seed=31)
    t = random_inputs(b, hq, hkv, s, d, seed=12)
    ex = oracle.Problem(**base)
    st = oracle.Problem(**base, stored_o_bf16=True)
    o, _ = oracle.fwd(ex, t.q, t.k, t.v)
    dq0, dk0, dv0 = oracle.bwd(ex, t.q, t.k, t.v, t.dout)
    dq1, dk1, dv1 = oracle.bwd(st, t.q, t.k, t.v, t.dout)
    g = t.dout.double().numpy()
    o16 = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
    dD = (g * o16).sum(-1) - (g * o).sum(-1)                    # [b, h, s]
    scale = oracle.resolved_scale(ex)
    q = t.q.double().numpy()
    k = t.k.double().numpy()
    assert np.array_equal(dv0, dv1)
    exp_dk = np.zeros_like(dk0)
    for h in range(hq):
        _, P, _ = oracle.head_matrices(ex, t.q, t.k, h)
        pk = P @ k[0, h // (hq // hkv)]
        assert np.max(np.abs((dq1 - dq0)[0, h] + scale * dD[0, h][:, None] * pk)) < 1e-12
        exp_dk[0, h // (hq // hkv)] -= scale * P.T @ (dD[0, h][:, None] * q[0, h])
    assert np.max(np.abs((dk1 - dk0) - exp_dk)) < 1e-12
    # and the perturbation is at the bf16 storage level, not larger
    assert np.max(np.abs(dD)) <= 2.0 ** -8 * np.max(np.abs(g * o).sum(-1)) + 1e-12


def test_stored_output_model_is_exact_when_output_is_bf16():
    """s = 1 with p = 0: O = V exactly (bf16), so the model equals the exact backward."""
    base = dict(b=1, h_q=2, h_kv=2, s=1, d=16, causal=True)
    t = random_inputs(1, 2, 2, 1, 16, seed=13)
    a = oracle.bwd(oracle.Problem(**base), t.q, t.k, t.v, t.dout)
    c = oracle.bwd(oracle.Problem(**base, stored_o_bf16=True), t.q, t.k, t.v, t.dout)
    for x, y in zip(a, c):
        assert np.max(np.abs(x - y)) < 1e-15
