"""CPU oracle for the attention core (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product library never does: it shares
no code with this package, and this package imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (the attention core) and
``dropout_add_ln_oracle.c`` (the dropout, residual add and layer norm on
either side of it): plain C, fp64, OpenMP over rows or heads.  This module
compiles them with gcc and exposes them through ctypes with numpy float64
arrays.  See the headers of the C files for what each function computes and
which passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "attn_oracle.c"), os.path.join(_HERE, "dropout_add_ln_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src) for src in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
                ("s", ctypes.c_int32), ("d", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("p_drop", ctypes.c_float), ("scale", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
                ("stored_o_bf16", ctypes.c_int32), ("s_kv", ctypes.c_int32)]


class _DalParams(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("hidden", ctypes.c_int32), ("p_drop", ctypes.c_float),
                ("eps", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


class _Bytes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("layer_none", "layer_selective", "layer_full", "core_scores_avoided",
                 "core_kept", "core_recompute_state")]


_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_U32 = ctypes.POINTER(ctypes.c_uint32)
_PP = ctypes.POINTER(_Params)


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_philox4x32_10.argtypes = [_U32, _U32, _U32]
        lib.oracle_drop_threshold.argtypes = [ctypes.c_float]
        lib.oracle_drop_threshold.restype = ctypes.c_uint32
        lib.oracle_drop_threshold16.argtypes = [ctypes.c_float]
        lib.oracle_drop_threshold16.restype = ctypes.c_uint32
        lib.oracle_draw8.argtypes = [_PP, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_draw8.restype = ctypes.c_uint32
        lib.oracle_keep.argtypes = [_PP, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_keep.restype = ctypes.c_int
        lib.oracle_resolved_scale.argtypes = [_PP]
        lib.oracle_resolved_scale.restype = ctypes.c_double
        lib.oracle_fwd.argtypes = [_PP, _D, _D, _D, _D, _D]
        lib.oracle_fwd_rows.argtypes = [_PP, _D, _D, _D, ctypes.c_int64, _I64, _I64, _D, _D]
        lib.oracle_head_matrices.argtypes = [_PP, _D, _D, ctypes.c_int64, _D, _D, _U8]
        lib.oracle_mask_rows.argtypes = [_PP, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _U8]
        lib.oracle_bwd.argtypes = [_PP, _D, _D, _D, _D, _D, _D, _D]
        lib.oracle_dq_rows.argtypes = [_PP, _D, _D, _D, _D, ctypes.c_int64, _I64, _I64, _D]
        lib.oracle_dkdv_rows.argtypes = [_PP, _D, _D, _D, _D, ctypes.c_int64, _I64, _I64, _D, _D]
        lib.oracle_stored_bytes.argtypes = [_PP, ctypes.POINTER(_Bytes)]
        DP = ctypes.POINTER(_DalParams)
        lib.oracle_dal_keep.argtypes = [DP, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_dal_keep.restype = ctypes.c_int
        lib.oracle_dal_fwd.argtypes = [DP, _D, _D, _D, _D, _D, _D, _D, _D]
        lib.oracle_dal_bwd.argtypes = [DP, _D, _D, _D, _D, _D, _D, _D, _D, _D]
        _lib = lib
    return _lib


@dataclass
class Problem:
    """Shape and method parameters of one attention-core call."""
    b: int
    h_q: int
    h_kv: int
    s: int
    d: int
    causal: bool = True
    p_drop: float = 0.0
    scale: float = 0.0      # <= 0: 1/sqrt(d) rounded to fp32
    seed: int = 0
    offset: int = 0
    # Backward row statistic sum_j P_ij dP_ij taken as dO_i . bf16(O_i), the
    # way a method that stores only the bf16 output must form it.  False: the
    # exact definition.
    stored_o_bf16: bool = False
    # Keys (and value rows) per KV head; 0 means s (self-attention).
    s_kv: int = 0

    @property
    def keys(self) -> int:
        return self.s_kv or self.s

    def _c(self) -> _Params:
        return _Params(self.b, self.h_q, self.h_kv, self.s, self.d, int(bool(self.causal)),
                       float(self.p_drop), float(self.scale), int(self.seed) & (2**64 - 1),
                       int(self.offset) & (2**64 - 1), int(bool(self.stored_o_bf16)),
                       int(self.s_kv))


def _f64(x) -> np.ndarray:
    """Exact widening of a tensor or array (bf16 widens exactly) to contiguous fp64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _ip(a: np.ndarray):
    return a.ctypes.data_as(_I64)


def philox4x32_10(counter, key) -> np.ndarray:
    """Philox-4x32-10 of a 4-word counter and 2-word key (SC'11 definition)."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(c.ctypes.data_as(_U32), k.ctypes.data_as(_U32), out.ctypes.data_as(_U32))
    return out


def drop_threshold(p_drop: float) -> int:
    """The attention core's threshold on an 8-bit draw: round(p * 256), at most 255."""
    return int(_load().oracle_drop_threshold(ctypes.c_float(p_drop)))


def drop_threshold16(p_drop: float) -> int:
    """The dropout + layer norm block's threshold on a 16-bit draw:
    round(p * 65536), at most 65535."""
    return int(_load().oracle_drop_threshold16(ctypes.c_float(p_drop)))


def draw8(pr: Problem, bh: int, i: int, j: int) -> int:
    return int(_load().oracle_draw8(ctypes.byref(pr._c()), bh, i, j))


def keep(pr: Problem, bh: int, i: int, j: int) -> int:
    return int(_load().oracle_keep(ctypes.byref(pr._c()), bh, i, j))


def resolved_scale(pr: Problem) -> float:
    return float(_load().oracle_resolved_scale(ctypes.byref(pr._c())))


def fwd(pr: Problem, q, k, v):
    """Full forward: returns (O [b,h_q,s,d] fp64, LSE [b,h_q,s] fp64)."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    o = np.zeros((pr.b, pr.h_q, pr.s, pr.d))
    lse = np.zeros((pr.b, pr.h_q, pr.s))
    lib.oracle_fwd(ctypes.byref(pr._c()), _dp(q), _dp(k), _dp(v), _dp(o), _dp(lse))
    return o, lse


def fwd_rows(pr: Problem, q, k, v, bh, rows):
    """Forward for sampled (flattened query head, row) pairs: (O [n,d], LSE [n])."""
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    bh = np.ascontiguousarray(np.asarray(bh, dtype=np.int64))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = len(rows)
    o = np.zeros((n, pr.d))
    lse = np.zeros(n)
    lib.oracle_fwd_rows(ctypes.byref(pr._c()), _dp(q), _dp(k), _dp(v), n, _ip(bh), _ip(rows),
                        _dp(o), _dp(lse))
    return o, lse


def head_matrices(pr: Problem, q, k, bh: int):
    """Dense S, P (fp64, s x s_kv) and keep mask M (uint8) of one query head."""
    lib = _load()
    q, k = _f64(q), _f64(k)
    S = np.zeros((pr.s, pr.keys))
    P = np.zeros((pr.s, pr.keys))
    M = np.zeros((pr.s, pr.keys), dtype=np.uint8)
    lib.oracle_head_matrices(ctypes.byref(pr._c()), _dp(q), _dp(k), bh, _dp(S), _dp(P),
                             M.ctypes.data_as(_U8))
    return S, P, M


def mask_rows(pr: Problem, bh: int, i0: int, i1: int) -> np.ndarray:
    """Keep mask (uint8, rows [i0,i1) x s_kv keys) of one query head; hidden keys are 0."""
    M = np.zeros((i1 - i0, pr.keys), dtype=np.uint8)
    _load().oracle_mask_rows(ctypes.byref(pr._c()), bh, i0, i1, M.ctypes.data_as(_U8))
    return M


def bwd(pr: Problem, q, k, v, dout):
    """Full backward: (dQ [b,h_q,s,d], dK [b,h_kv,s_kv,d], dV [b,h_kv,s_kv,d]), fp64."""
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    dq = np.zeros((pr.b, pr.h_q, pr.s, pr.d))
    dk = np.zeros((pr.b, pr.h_kv, pr.keys, pr.d))
    dv = np.zeros((pr.b, pr.h_kv, pr.keys, pr.d))
    lib.oracle_bwd(ctypes.byref(pr._c()), _dp(q), _dp(k), _dp(v), _dp(dout), _dp(dq), _dp(dk),
                   _dp(dv))
    return dq, dk, dv


def dq_rows(pr: Problem, q, k, v, dout, bh, rows) -> np.ndarray:
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    bh = np.ascontiguousarray(np.asarray(bh, dtype=np.int64))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(rows), pr.d))
    lib.oracle_dq_rows(ctypes.byref(pr._c()), _dp(q), _dp(k), _dp(v), _dp(dout), len(rows),
                       _ip(bh), _ip(rows), _dp(out))
    return out


def dkdv_rows(pr: Problem, q, k, v, dout, bkv, rows):
    lib = _load()
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    bkv = np.ascontiguousarray(np.asarray(bkv, dtype=np.int64))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dk = np.zeros((len(rows), pr.d))
    dv = np.zeros((len(rows), pr.d))
    lib.oracle_dkdv_rows(ctypes.byref(pr._c()), _dp(q), _dp(k), _dp(v), _dp(dout), len(rows),
                         _ip(bkv), _ip(rows), _dp(dk), _dp(dv))
    return dk, dv


def stored_bytes(pr: Problem) -> dict:
    out = _Bytes()
    _load().oracle_stored_bytes(ctypes.byref(pr._c()), ctypes.byref(out))
    return {n: int(getattr(out, n)) for n, _ in _Bytes._fields_}


# ------------------------------------------- dropout + residual + layer norm

@dataclass
class DalProblem:
    """z = residual + dropout(x), y = LayerNorm(z) over rows of ``hidden`` values."""
    n_rows: int
    hidden: int
    p_drop: float = 0.0
    eps: float = 1e-5
    seed: int = 0
    offset: int = 0

    def _c(self) -> _DalParams:
        return _DalParams(self.n_rows, self.hidden, float(self.p_drop), float(self.eps),
                          int(self.seed) & (2**64 - 1), int(self.offset) & (2**64 - 1))


def dal_keep(pr: DalProblem, row: int, col: int) -> int:
    return int(_load().oracle_dal_keep(ctypes.byref(pr._c()), row, col))


def dal_mask(pr: DalProblem) -> np.ndarray:
    """Keep mask (uint8, n_rows x hidden)."""
    return np.array([[dal_keep(pr, i, c) for c in range(pr.hidden)] for i in range(pr.n_rows)],
                    dtype=np.uint8)


def dal_fwd(pr: DalProblem, x, r, gamma, beta):
    """(z, y) [n_rows, hidden] and (mean, rstd) [n_rows], fp64."""
    lib = _load()
    x, r, gamma, beta = _f64(x), _f64(r), _f64(gamma), _f64(beta)
    z = np.zeros((pr.n_rows, pr.hidden))
    y = np.zeros((pr.n_rows, pr.hidden))
    mean = np.zeros(pr.n_rows)
    rstd = np.zeros(pr.n_rows)
    lib.oracle_dal_fwd(ctypes.byref(pr._c()), _dp(x), _dp(r), _dp(gamma), _dp(beta), _dp(z), _dp(y),
                       _dp(mean), _dp(rstd))
    return z, y, mean, rstd


def dal_bwd(pr: DalProblem, x, r, gamma, dy, dz_next=None):
    """(dx, d_residual) [n_rows, hidden] and (dgamma, dbeta) [hidden], fp64."""
    lib = _load()
    x, r, gamma, dy = _f64(x), _f64(r), _f64(gamma), _f64(dy)
    dzn = _f64(dz_next) if dz_next is not None else None
    dx = np.zeros((pr.n_rows, pr.hidden))
    dres = np.zeros((pr.n_rows, pr.hidden))
    dgamma = np.zeros(pr.hidden)
    dbeta = np.zeros(pr.hidden)
    lib.oracle_dal_bwd(ctypes.byref(pr._c()), _dp(x), _dp(r), _dp(gamma), _dp(dy),
                       _dp(dzn) if dzn is not None else None, _dp(dx), _dp(dres), _dp(dgamma),
                       _dp(dbeta))
    return dx, dres, dgamma, dbeta


# ------------------------------------------------------------------ GeLU ---
# The MLP activation of the layer around the core, tanh form (Hendrycks and
# Gimpel): y = x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), fp64.

_GELU_C = math.sqrt(2.0 / math.pi)
_GELU_A = 0.044715


def gelu(x) -> np.ndarray:
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(_GELU_C * (x + _GELU_A * x ** 3)))


def gelu_grad(x) -> np.ndarray:
    """d gelu / dx."""
    x = _f64(x)
    t = np.tanh(_GELU_C * (x + _GELU_A * x ** 3))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * _GELU_C * (1.0 + 3.0 * _GELU_A * x * x)
