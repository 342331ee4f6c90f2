"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol the public header declares, validates its arguments before touching
the device, and reports the activation-byte accounting exactly."""
import ctypes
import os
import re

import pytest

import attention_core_gb300 as ac
import oracle
from attention_core_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return ac.load_library()


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(attn_core_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("attn_core_fwd", "attn_core_bwd_recompute", "attn_core_stored_bytes",
              "attn_core_bwd_workspace_bytes", "attn_core_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(ac.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(raw, n), n


def test_strerror(lib):
    assert ac.attn_core_strerror(ac.OK) == "ok"
    assert "workspace" in ac.attn_core_strerror(ac.ERR_WORKSPACE_TOO_SMALL)
    assert "time limit" in ac.attn_core_strerror(ac.ERR_DEVICE_TIMEOUT | (3 << 8))


def _p(**kw):
    base = dict(b=1, h_q=2, h_kv=2, s=128, d=64, causal=True, p_drop=0.1, seed=1, offset=0)
    base.update(kw)
    return ac.Params(**base)


FAKE = 0x7f0000000000  # 16-byte aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("kw,code", [
    (dict(b=0), ac.ERR_INVALID_ARG),
    (dict(s=-1), ac.ERR_INVALID_ARG),
    (dict(h_q=3, h_kv=2), ac.ERR_INVALID_ARG),
    (dict(p_drop=1.0), ac.ERR_INVALID_ARG),
    (dict(p_drop=-0.1), ac.ERR_INVALID_ARG),
    (dict(p_drop=float("nan")), ac.ERR_INVALID_ARG),
    (dict(offset=2**32), ac.ERR_INVALID_ARG),
    (dict(causal=2), ac.ERR_INVALID_ARG),
    (dict(s_kv=-1), ac.ERR_INVALID_ARG),
    (dict(s_kv=200, d=80), ac.ERR_UNSUPPORTED),      # causal cross-attention is valid; d is not
    (dict(s_kv=200, causal=False, d=80), ac.ERR_UNSUPPORTED),
    (dict(d=80), ac.ERR_UNSUPPORTED),
    (dict(d=256), ac.ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_params(lib, kw, code):
    assert ac.attn_core_fwd(_p(**kw), FAKE, FAKE, FAKE, FAKE, FAKE, 0) == code


def test_fwd_rejects_null_and_misaligned(lib):
    assert ac.attn_core_fwd(_p(), 0, FAKE, FAKE, FAKE, FAKE, 0) == ac.ERR_INVALID_ARG
    assert ac.attn_core_fwd(_p(), FAKE + 8, FAKE, FAKE, FAKE, FAKE, 0) == ac.ERR_MISALIGNED
    assert ac.attn_core_fwd(_p(), FAKE, FAKE, FAKE, FAKE, FAKE + 4, 0) == ac.ERR_MISALIGNED


def test_cross_attention_params(lib):
    # s_kv == s is self-attention; without dropout the workspace follows the queries only
    assert ac.attn_core_bwd_workspace_bytes(_p(s_kv=128)) == ac.attn_core_bwd_workspace_bytes(_p())
    assert (ac.attn_core_bwd_workspace_bytes(_p(s=200, s_kv=1000, causal=False, p_drop=0.0))
            == ac.attn_core_bwd_workspace_bytes(_p(s=200, p_drop=0.0)) == 2 * 4 * 2 * 256)
    # with dropout it adds 2 KB of keep bits per 128 x 128 block: 2 heads x 2 x 8 blocks
    assert (ac.attn_core_bwd_workspace_bytes(_p(s=200, s_kv=1000, causal=False))
            == 2 * 4 * 2 * 256 + 2048 * 2 * 2 * 8)
    # causal with s_kv != s (top-left aligned) is valid; its mask is drawn twice, so the
    # workspace holds the row statistics only
    assert ac.attn_core_bwd_workspace_bytes(_p(s=200, s_kv=1000)) == 2 * 4 * 2 * 256
    assert ac.attn_core_bwd_workspace_bytes(_p(s=1000, s_kv=200)) == 2 * 4 * 2 * 1024


def test_bwd_workspace_and_validation(lib):
    p = _p(s=200)
    ws = ac.attn_core_bwd_workspace_bytes(p)
    # two fp32 statistics per padded query row, and (p > 0) 2 KB of keep bits for
    # each of the 3 causal 128 x 128 blocks of the 2 heads
    assert ws == 2 * 4 * 1 * 2 * 256 + 2048 * 2 * 3
    assert ac.attn_core_bwd_workspace_bytes(_p(s=200, p_drop=0.0)) == 2 * 4 * 1 * 2 * 256
    assert ac.attn_core_bwd_workspace_bytes(_p(s=200, causal=False)) == 2 * 4 * 1 * 2 * 256 + 2048 * 2 * 4
    assert ac.attn_core_bwd_workspace_bytes(_p(s=200, d=160)) == 2 * 4 * 1 * 2 * 256    # d = 160 draws twice
    assert ac.attn_core_bwd_workspace_bytes(_p(b=0)) == 0
    args = [FAKE] * 10
    assert ac.attn_core_bwd_recompute(p, *args, ws - 1, 0) == ac.ERR_WORKSPACE_TOO_SMALL
    a2 = list(args)
    a2[9] = FAKE + 16                  # workspace needs 256-byte alignment
    assert ac.attn_core_bwd_recompute(p, *a2, ws, 0) == ac.ERR_MISALIGNED
    a3 = list(args)
    a3[5] = 0                          # dout
    assert ac.attn_core_bwd_recompute(p, *a3, ws, 0) == ac.ERR_INVALID_ARG
    assert ac.attn_core_bwd_recompute(_p(d=48), *args, ws, 0) == ac.ERR_UNSUPPORTED


@pytest.mark.parametrize("shape", [(1, 64, 64, 8192, 128), (2, 12, 12, 2048, 128),
                                   (4, 8, 8, 2048, 96), (1, 16, 16, 2048, 160),
                                   (1, 64, 8, 8192, 128), (3, 6, 2, 333, 64)])
def test_stored_bytes_match_oracle(lib, shape):
    b, hq, hkv, s, d = shape
    got = ac.stored_bytes(b, hq, hkv, s, d)
    ref = oracle.stored_bytes(oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d))
    assert got == ref


@pytest.mark.parametrize("shape", [(2, 8, 2, 512, 1536, 64), (1, 4, 4, 300, 77, 128)])
def test_stored_bytes_cross_attention_match_oracle(lib, shape):
    b, hq, hkv, s, skv, d = shape
    got = ac.stored_bytes(b, hq, hkv, s, d, s_kv=skv)
    ref = oracle.stored_bytes(oracle.Problem(b=b, h_q=hq, h_kv=hkv, s=s, d=d, s_kv=skv))
    assert got == ref
    assert got["core_scores_avoided"] == 5 * hq * s * skv * b


def test_stored_bytes_llama_worked_example(lib):
    sb = ac.stored_bytes(1, 64, 8, 8192, 128)
    assert sb["layer_none"] * 80 == 1_900_523_028_480
    assert sb["layer_selective"] * 80 == 182_536_110_080
    assert sb["layer_full"] * 80 == 10_737_418_240
    # what the core actually keeps under GQA: Q and O at 64 heads, K and V at 8
    assert sb["core_kept"] == 2 * 8192 * 128 * (2 * 64 + 2 * 8)


def test_binding_fails_loudly_without_library(tmp_path):
    saved = ac._lib
    try:
        ac._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            ac.load_library(str(tmp_path / "missing.so"))
    finally:
        ac._lib = saved


# ------------------------------------------- dropout + residual + layer norm

def _dp(**kw):
    base = dict(n_rows=64, hidden=1024, p_drop=0.1, eps=1e-5, seed=1, offset=0)
    base.update(kw)
    return ac.DalParams(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(n_rows=0), ac.ERR_INVALID_ARG),
    (dict(hidden=1020), ac.ERR_INVALID_ARG),          # not a multiple of 8
    (dict(hidden=0), ac.ERR_INVALID_ARG),
    (dict(hidden=28680), ac.ERR_UNSUPPORTED),          # above the column-sum buffer
    (dict(p_drop=1.0), ac.ERR_INVALID_ARG),
    (dict(eps=0.0), ac.ERR_INVALID_ARG),
    (dict(eps=float("nan")), ac.ERR_INVALID_ARG),
    (dict(offset=2**32), ac.ERR_INVALID_ARG),
])
def test_dal_rejects_bad_params(lib, kw, code):
    assert ac.attn_core_dropout_add_ln_fwd(_dp(**kw), *([FAKE] * 8), 0) == code
    assert ac.attn_core_dropout_add_ln_bwd_workspace_bytes(_dp(**kw)) == 0


def test_dal_workspace_and_validation(lib):
    # per-CTA column sums of dgamma and dbeta: 2 x 4 bytes x hidden x min(n_rows, 320)
    assert ac.attn_core_dropout_add_ln_bwd_workspace_bytes(_dp()) == 8 * 1024 * 64
    assert ac.attn_core_dropout_add_ln_bwd_workspace_bytes(_dp(n_rows=4096, hidden=12288)) == 8 * 12288 * 320
    p = _dp()
    ws = ac.attn_core_dropout_add_ln_bwd_workspace_bytes(p)
    args = [FAKE] * 11                                 # dy, dz_next, z, ..., dbeta, workspace
    assert ac.attn_core_dropout_add_ln_bwd(p, *args, ws - 1, 0) == ac.ERR_WORKSPACE_TOO_SMALL
    a1 = list(args)
    a1[1] = FAKE + 8                                   # dz_next is optional, but aligned if given
    assert ac.attn_core_dropout_add_ln_bwd(p, *a1, ws, 0) == ac.ERR_MISALIGNED
    a2 = list(args)
    a2[0] = FAKE + 8                                   # dy misaligned
    assert ac.attn_core_dropout_add_ln_bwd(p, *a2, ws, 0) == ac.ERR_MISALIGNED
    a3 = list(args)
    a3[2] = 0                                          # z missing
    assert ac.attn_core_dropout_add_ln_bwd(p, *a3, ws, 0) == ac.ERR_INVALID_ARG
    assert ac.attn_core_dropout_add_ln_fwd(p, 0, *([FAKE] * 7), 0) == ac.ERR_INVALID_ARG


# ------------------------------------------------ variable-length batches

@pytest.mark.parametrize("cu_q,cu_k,causal", [
    ([1, 5], None, True),              # table must start at 0
    ([0, 5, 3], None, True),           # nondecreasing
    ([0, 5, 9], [0, 0, 3], False),     # queries without keys
])
def test_varlen_rejects_bad_tables(lib, cu_q, cu_k, causal):
    p = _p(causal=causal)
    dev = dict(cu_q_dev=FAKE, cu_k_dev=FAKE if cu_k is not None else 0)
    assert ac.attn_core_fwd_varlen(p, cu_q, cu_k, *([FAKE] * 5), 0, **dev) == ac.ERR_INVALID_ARG
    assert ac.attn_core_bwd_varlen_workspace_bytes(p, cu_q, cu_k, **dev) == 0


def test_varlen_needs_the_device_tables(lib):
    """The kernels read the sequence tables' device copies: a call without them
    (or with a key table but no device copy of it) is rejected before anything runs."""
    p = _p()
    assert ac.attn_core_fwd_varlen(p, [0, 5, 9], None, *([FAKE] * 5), 0) == ac.ERR_INVALID_ARG
    assert ac.attn_core_fwd_varlen(p, [0, 5, 9], [0, 5, 9], *([FAKE] * 5), 0, cu_q_dev=FAKE) == ac.ERR_INVALID_ARG
    assert ac.attn_core_bwd_varlen_workspace_bytes(p, [0, 5, 9], None) == 0


def test_varlen_workspace_formula_of_the_header(lib):
    """8 h_q (round_up(total_q, 4) + 132 n_seq) bytes of row statistics, rounded
    up to 256: every sequence's rows padded to whole 128-row blocks and aligned
    to 16 bytes, no keep bits."""
    p = _p(p_drop=0.1, h_q=4, h_kv=2)
    cu = [0, 200, 200, 300]            # lengths 200, 0 (skipped), 100
    want = 8 * 4 * (300 + 132 * 3)
    assert ac.attn_core_bwd_varlen_workspace_bytes(p, cu, None, cu_q_dev=FAKE) == (want + 255) // 256 * 256
    pt = _p(p_drop=0.1)
    pt.timing_events = FAKE           # per-kernel events are not offered for packed batches
    assert ac.attn_core_fwd_varlen(pt, cu, None, *([FAKE] * 5), 0, cu_q_dev=FAKE) == ac.ERR_INVALID_ARG


def test_bwd_workspace_formula_of_the_header(lib):
    """8 b h_q ceil(s/128) 128 bytes of row statistics, plus (p > 0, d <= 128)
    2048 b h_q N bytes of keep bits, N = n(n+1)/2 causal blocks per head or
    ceil(s/128) ceil(s_kv/128), as the public header states."""
    rng = __import__("random").Random(7)
    for _ in range(200):
        b, hkv = rng.randint(1, 4), rng.randint(1, 3)
        hq = hkv * rng.randint(1, 4)
        s = rng.randint(1, 3000)
        d = rng.choice([64, 96, 128, 160])
        causal = rng.random() < 0.5
        skv = s if causal else rng.choice([0, rng.randint(1, 3000)])
        p_drop = rng.choice([0.0, 0.1])
        kv = skv or s
        n, nk = -(-s // 128), -(-kv // 128)
        stats = 8 * b * hq * n * 128
        blocks = n * (n + 1) // 2 if causal else n * nk
        bits = 2048 * b * hq * blocks if (p_drop > 0 and d <= 128) else 0
        p = ac.Params(b=b, h_q=hq, h_kv=hkv, s=s, d=d, causal=causal, p_drop=p_drop, s_kv=skv)
        assert ac.attn_core_bwd_workspace_bytes(p) == stats + bits, (b, hq, hkv, s, skv, d, causal, p_drop)
