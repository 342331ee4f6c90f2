"""GB300 (sm_103a) attention core under selective activation recomputation.

Thin Python binding of the C ABI in ``include/attn_core.h``: the functions
below marshal torch tensors into device pointers and the current CUDA stream
and call the library; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if ``libattn_core.so`` is missing or
cannot be loaded, the first call raises.

The attention core (QK^T, softmax, softmax dropout, attention over V) is the
part of a transformer layer that selective activation recomputation drops
after the forward pass and recomputes in the backward pass ("Reducing
Activation Recomputation in Large Transformer Models", Key takeaways, fourth
bullet).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

__all__ = [
    "AttnCoreError", "Params", "load_library", "attn_core_fwd", "attn_core_bwd_recompute",
    "attn_core_bwd_workspace_bytes", "attn_core_stored_bytes", "attn_core_strerror",
    "attn_core_bwd_recompute_noalloc",
    "fwd", "bwd_recompute", "stored_bytes", "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED",
    "ERR_MISALIGNED", "ERR_WORKSPACE_TOO_SMALL", "ERR_CUDA", "ERR_DEVICE_TIMEOUT",
    "FLAG_TEST_WAIT_TIMEOUT", "FLAG_REDRAW_MASK", "SUPPORTED_HEAD_DIMS",
    "DalParams", "attn_core_dropout_add_ln_fwd", "attn_core_dropout_add_ln_bwd",
    "attn_core_dropout_add_ln_bwd_workspace_bytes", "dropout_add_ln_fwd", "dropout_add_ln_bwd",
    "attn_core_gelu_fwd", "attn_core_gelu_bwd", "gelu_fwd", "gelu_bwd",
    "attn_core_fwd_varlen", "attn_core_bwd_varlen", "attn_core_bwd_varlen_workspace_bytes",
    "fwd_varlen", "bwd_varlen",
]

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_MISALIGNED = 3
ERR_WORKSPACE_TOO_SMALL = 4
ERR_CUDA = 5
ERR_DEVICE_TIMEOUT = 6
FLAG_REDRAW_MASK = 0x1
FLAG_TEST_WAIT_TIMEOUT = 0x100
SUPPORTED_HEAD_DIMS = (64, 96, 128, 160)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libattn_core.so")


class AttnCoreError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {attn_core_strerror(code)} (code {code})")


class _CParams(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
                ("s", ctypes.c_int32), ("d", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("p_drop", ctypes.c_float), ("scale", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
                ("dev_status", ctypes.c_void_p), ("flags", ctypes.c_int32),
                ("wait_timeout_ms", ctypes.c_uint32), ("timing_events", ctypes.c_void_p),
                ("s_kv", ctypes.c_int32)]


class _CVarlenParams(ctypes.Structure):
    _fields_ = [("base", _CParams), ("n_seq", ctypes.c_int32),
                ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int32)),
                ("cu_seqlens_k", ctypes.POINTER(ctypes.c_int32)),
                ("cu_seqlens_q_dev", ctypes.c_void_p), ("cu_seqlens_k_dev", ctypes.c_void_p)]


class _CDalParams(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("hidden", ctypes.c_int32), ("p_drop", ctypes.c_float),
                ("eps", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64),
                ("dev_status", ctypes.c_void_p), ("wait_timeout_ms", ctypes.c_uint32)]


class _CBytes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("layer_none", "layer_selective", "layer_full", "core_scores_avoided",
                 "core_kept", "core_recompute_state")]


@dataclass
class Params:
    """Mirror of ``attn_core_params`` (see include/attn_core.h)."""
    b: int
    h_q: int
    h_kv: int
    s: int
    d: int
    causal: bool = True
    p_drop: float = 0.0
    scale: float = 0.0
    seed: int = 0
    offset: int = 0
    dev_status: int = 0          # device address of an int32, or 0
    flags: int = 0
    wait_timeout_ms: int = 0
    timing_events: int = 0       # address of a void*[2 * n_kernels] array, or 0
    s_kv: int = 0                # keys per KV head; 0 means s

    @property
    def keys(self) -> int:
        return self.s_kv or self.s

    def to_c(self) -> _CParams:
        return _CParams(self.b, self.h_q, self.h_kv, self.s, self.d, int(self.causal),
                        float(self.p_drop), float(self.scale), int(self.seed) & (2**64 - 1),
                        int(self.offset) & (2**64 - 1), self.dev_status or None, int(self.flags),
                        int(self.wait_timeout_ms), self.timing_events or None, int(self.s_kv))


@dataclass
class DalParams:
    """Mirror of ``attn_core_dal_params`` (dropout + residual add + layer norm)."""
    n_rows: int
    hidden: int
    p_drop: float = 0.0
    eps: float = 1e-5
    seed: int = 0
    offset: int = 0
    dev_status: int = 0          # device address of an int32, or 0
    wait_timeout_ms: int = 0

    def to_c(self) -> _CDalParams:
        return _CDalParams(int(self.n_rows), int(self.hidden), float(self.p_drop), float(self.eps),
                           int(self.seed) & (2**64 - 1), int(self.offset) & (2**64 - 1),
                           self.dev_status or None, int(self.wait_timeout_ms))


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libattn_core.so (raises if it is absent: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"attention-core library not built ({path} missing); run "
            "`python -m attention_core_gb300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    P = ctypes.POINTER(_CParams)
    lib.attn_core_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp]
    lib.attn_core_fwd.restype = ctypes.c_int
    lib.attn_core_bwd_workspace_bytes.argtypes = [P]
    lib.attn_core_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_core_bwd_recompute.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.attn_core_bwd_recompute.restype = ctypes.c_int
    lib.attn_core_bwd_recompute_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.attn_core_bwd_recompute_noalloc.restype = ctypes.c_int
    lib.attn_core_stored_bytes.argtypes = [P, ctypes.POINTER(_CBytes)]
    lib.attn_core_stored_bytes.restype = ctypes.c_int
    lib.attn_core_strerror.argtypes = [ctypes.c_int]
    lib.attn_core_strerror.restype = ctypes.c_char_p
    DP = ctypes.POINTER(_CDalParams)
    lib.attn_core_dropout_add_ln_fwd.argtypes = [DP, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.attn_core_dropout_add_ln_fwd.restype = ctypes.c_int
    lib.attn_core_dropout_add_ln_bwd_workspace_bytes.argtypes = [DP]
    lib.attn_core_dropout_add_ln_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_core_dropout_add_ln_bwd.argtypes = [DP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 ctypes.c_size_t, vp]
    lib.attn_core_dropout_add_ln_bwd.restype = ctypes.c_int
    VP = ctypes.POINTER(_CVarlenParams)
    lib.attn_core_fwd_varlen.argtypes = [VP, vp, vp, vp, vp, vp, vp]
    lib.attn_core_fwd_varlen.restype = ctypes.c_int
    lib.attn_core_bwd_varlen_workspace_bytes.argtypes = [VP]
    lib.attn_core_bwd_varlen_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_core_bwd_varlen.argtypes = [VP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.attn_core_bwd_varlen.restype = ctypes.c_int
    lib.attn_core_gelu_fwd.argtypes = [ctypes.c_int64, vp, vp, vp]
    lib.attn_core_gelu_fwd.restype = ctypes.c_int
    lib.attn_core_gelu_bwd.argtypes = [ctypes.c_int64, vp, vp, vp, vp]
    lib.attn_core_gelu_bwd.restype = ctypes.c_int
    _lib = lib
    return lib


# ------------------------------------------------------------ raw C ABI ---
# Same names and arguments as the C functions; pointers are plain integers.

def attn_core_strerror(code: int) -> str:
    return load_library().attn_core_strerror(int(code)).decode()


def attn_core_fwd(p: Params, q: int, k: int, v: int, o: int, lse: int, stream: int) -> int:
    cp = p.to_c()
    return load_library().attn_core_fwd(ctypes.byref(cp), q, k, v, o, lse, stream or None)


def attn_core_bwd_workspace_bytes(p: Params) -> int:
    cp = p.to_c()
    return int(load_library().attn_core_bwd_workspace_bytes(ctypes.byref(cp)))


def attn_core_bwd_recompute(p: Params, q: int, k: int, v: int, o: int, lse: int, dout: int,
                            dq: int, dk: int, dv: int, workspace: int, workspace_bytes: int,
                            stream: int) -> int:
    cp = p.to_c()
    return load_library().attn_core_bwd_recompute(ctypes.byref(cp), q, k, v, o, lse, dout, dq, dk,
                                                  dv, workspace, workspace_bytes, stream or None)


def attn_core_bwd_recompute_noalloc(p: Params, q: int, k: int, v: int, o: int, lse: int, dout: int,
                                    dq: int, dk: int, dv: int, stream: int) -> int:
    """Backward for callers that cannot allocate device memory: no workspace
    argument; the library's own fixed scratch array is used (see the header
    for its size limit and for why calls that overlap on the GPU race)."""
    cp = p.to_c()
    return load_library().attn_core_bwd_recompute_noalloc(ctypes.byref(cp), q, k, v, o, lse, dout, dq,
                                                          dk, dv, stream or None)


def attn_core_stored_bytes(p: Params) -> tuple[int, dict]:
    cp = p.to_c()
    out = _CBytes()
    rc = load_library().attn_core_stored_bytes(ctypes.byref(cp), ctypes.byref(out))
    return rc, {n: int(getattr(out, n)) for n, _ in _CBytes._fields_}


def attn_core_dropout_add_ln_fwd(p: DalParams, x: int, residual: int, gamma: int, beta: int, z: int,
                                 y: int, mean: int, rstd: int, stream: int) -> int:
    cp = p.to_c()
    return load_library().attn_core_dropout_add_ln_fwd(ctypes.byref(cp), x, residual, gamma, beta, z, y,
                                                       mean, rstd, stream or None)


def attn_core_dropout_add_ln_bwd_workspace_bytes(p: DalParams) -> int:
    cp = p.to_c()
    return int(load_library().attn_core_dropout_add_ln_bwd_workspace_bytes(ctypes.byref(cp)))


def attn_core_dropout_add_ln_bwd(p: DalParams, dy: int, dz_next: int, z: int, mean: int, rstd: int,
                                 gamma: int, dx: int, d_residual: int, dgamma: int, dbeta: int,
                                 workspace: int, workspace_bytes: int, stream: int) -> int:
    cp = p.to_c()
    return load_library().attn_core_dropout_add_ln_bwd(ctypes.byref(cp), dy, dz_next or None, z, mean,
                                                       rstd, gamma, dx, d_residual, dgamma, dbeta,
                                                       workspace, workspace_bytes, stream or None)


def _varlen_c(p: Params, cu_q, cu_k, cu_q_dev: int = 0, cu_k_dev: int = 0):
    """(_CVarlenParams, keep-alive arrays) for host sequence tables and the
    device addresses of their copies."""
    aq = (ctypes.c_int32 * len(cu_q))(*[int(x) for x in cu_q])
    ak = (ctypes.c_int32 * len(cu_k))(*[int(x) for x in cu_k]) if cu_k is not None else None
    vp = _CVarlenParams(p.to_c(), len(cu_q) - 1, ctypes.cast(aq, ctypes.POINTER(ctypes.c_int32)),
                        ctypes.cast(ak, ctypes.POINTER(ctypes.c_int32)) if ak is not None else None,
                        cu_q_dev or None, cu_k_dev or None)
    return vp, (aq, ak)


def attn_core_fwd_varlen(p: Params, cu_q, cu_k, q: int, k: int, v: int, o: int, lse: int, stream: int, *,
                         cu_q_dev: int = 0, cu_k_dev: int = 0) -> int:
    """p supplies h_q, h_kv, d, causal, p_drop, scale, seed, offset, dev_status,
    flags and wait_timeout_ms; cu_q / cu_k are host sequence tables and
    cu_q_dev / cu_k_dev the device addresses of their copies."""
    vp, keep = _varlen_c(p, cu_q, cu_k, cu_q_dev, cu_k_dev)
    return load_library().attn_core_fwd_varlen(ctypes.byref(vp), q, k, v, o, lse, stream or None)


def attn_core_bwd_varlen_workspace_bytes(p: Params, cu_q, cu_k, *, cu_q_dev: int = 0, cu_k_dev: int = 0) -> int:
    vp, keep = _varlen_c(p, cu_q, cu_k, cu_q_dev, cu_k_dev)
    return int(load_library().attn_core_bwd_varlen_workspace_bytes(ctypes.byref(vp)))


def attn_core_bwd_varlen(p: Params, cu_q, cu_k, q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int,
                         dk: int, dv: int, workspace: int, workspace_bytes: int, stream: int, *,
                         cu_q_dev: int = 0, cu_k_dev: int = 0) -> int:
    vp, keep = _varlen_c(p, cu_q, cu_k, cu_q_dev, cu_k_dev)
    return load_library().attn_core_bwd_varlen(ctypes.byref(vp), q, k, v, o, lse, dout, dq, dk, dv, workspace,
                                               workspace_bytes, stream or None)


def _device_tables(cq, ck, device):
    """Device copies of the host sequence tables (kept alive by the caller until
    the kernels that read them are queued: the caching allocator reuses the
    memory only in stream order)."""
    import torch
    tq = torch.tensor(cq, dtype=torch.int32, device=device)
    tk = torch.tensor(ck, dtype=torch.int32, device=device) if ck is not None else None
    return tq, tk, tq.data_ptr(), (tk.data_ptr() if tk is not None else 0)


def attn_core_gelu_fwd(n: int, x: int, y: int, stream: int) -> int:
    return load_library().attn_core_gelu_fwd(int(n), x, y, stream or None)


def attn_core_gelu_bwd(n: int, x: int, dy: int, dx: int, stream: int) -> int:
    return load_library().attn_core_gelu_bwd(int(n), x, dy, dx, stream or None)


# --------------------------------------------------- torch conveniences ---

def _check(t, name, dtype, shape):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream() -> int:
    import torch
    return torch.cuda.current_stream().cuda_stream


def _params_from(q, k, causal, p_drop, seed, offset, scale, **kw) -> Params:
    b, h_q, s, d = q.shape
    return Params(b=b, h_q=h_q, h_kv=k.shape[1], s=s, d=d, causal=causal, p_drop=p_drop,
                  scale=scale, seed=seed, offset=offset, s_kv=k.shape[2], **kw)


def fwd(q, k, v, *, causal: bool = True, p_drop: float = 0.0, seed: int = 0, offset: int = 0,
        scale: float = 0.0, out=None, lse=None, **kw):
    """Forward of the attention core.  Returns (O bf16 [b,h_q,s,d], LSE fp32 [b,h_q,s]).

    K and V may have a different sequence length from Q (s_kv keys,
    cross-attention) when ``causal`` is False."""
    import torch
    p = _params_from(q, k, causal, p_drop, seed, offset, scale, **kw)
    _check(q, "q", torch.bfloat16, (p.b, p.h_q, p.s, p.d))
    _check(k, "k", torch.bfloat16, (p.b, p.h_kv, p.keys, p.d))
    _check(v, "v", torch.bfloat16, (p.b, p.h_kv, p.keys, p.d))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((p.b, p.h_q, p.s), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, (p.b, p.h_q, p.s, p.d))
    _check(lse, "lse", torch.float32, (p.b, p.h_q, p.s))
    rc = attn_core_fwd(p, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       _stream())
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_fwd")
    return out, lse


def bwd_recompute(q, k, v, o, lse, dout, *, causal: bool = True, p_drop: float = 0.0, seed: int = 0,
                  offset: int = 0, scale: float = 0.0, dq=None, dk=None, dv=None, workspace=None,
                  **kw):
    """Recompute-backward.  Returns (dQ, dK, dV), bf16, shaped like Q, K, V."""
    import torch
    p = _params_from(q, k, causal, p_drop, seed, offset, scale, **kw)
    _check(q, "q", torch.bfloat16, (p.b, p.h_q, p.s, p.d))
    _check(k, "k", torch.bfloat16, (p.b, p.h_kv, p.keys, p.d))
    _check(v, "v", torch.bfloat16, (p.b, p.h_kv, p.keys, p.d))
    _check(o, "o", torch.bfloat16, (p.b, p.h_q, p.s, p.d))
    _check(dout, "dout", torch.bfloat16, (p.b, p.h_q, p.s, p.d))
    _check(lse, "lse", torch.float32, (p.b, p.h_q, p.s))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(dq, "dq", torch.bfloat16, (p.b, p.h_q, p.s, p.d))
    _check(dk, "dk", torch.bfloat16, (p.b, p.h_kv, p.keys, p.d))
    _check(dv, "dv", torch.bfloat16, (p.b, p.h_kv, p.keys, p.d))
    ws_bytes = attn_core_bwd_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    rc = attn_core_bwd_recompute(p, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream())
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_bwd_recompute")
    return dq, dk, dv


def stored_bytes(b: int, h_q: int, h_kv: int, s: int, d: int, s_kv: int = 0) -> dict:
    """Activation-byte accounting of one layer shard (see attn_core_bytes)."""
    rc, out = attn_core_stored_bytes(Params(b=b, h_q=h_q, h_kv=h_kv, s=s, d=d, s_kv=s_kv,
                                            causal=not s_kv or s_kv == s))
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_stored_bytes")
    return out


def dropout_add_ln_fwd(x, residual, gamma, beta, *, p_drop: float = 0.0, seed: int = 0, offset: int = 0,
                       eps: float = 1e-5, **kw):
    """z = residual + dropout(x), y = LayerNorm(z).  Returns (z, y, mean, rstd)."""
    import torch
    n, h = x.shape
    p = DalParams(n_rows=n, hidden=h, p_drop=p_drop, eps=eps, seed=seed, offset=offset, **kw)
    _check(x, "x", torch.bfloat16, (n, h))
    _check(residual, "residual", torch.bfloat16, (n, h))
    _check(gamma, "gamma", torch.float32, (h,))
    _check(beta, "beta", torch.float32, (h,))
    z, y = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty(n, dtype=torch.float32, device=x.device)
    rstd = torch.empty(n, dtype=torch.float32, device=x.device)
    rc = attn_core_dropout_add_ln_fwd(p, x.data_ptr(), residual.data_ptr(), gamma.data_ptr(),
                                      beta.data_ptr(), z.data_ptr(), y.data_ptr(), mean.data_ptr(),
                                      rstd.data_ptr(), _stream())
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_dropout_add_ln_fwd")
    return z, y, mean, rstd


def dropout_add_ln_bwd(dy, z, mean, rstd, gamma, *, dz_next=None, p_drop: float = 0.0, seed: int = 0,
                       offset: int = 0, eps: float = 1e-5, workspace=None, **kw):
    """Gradients of dropout_add_ln_fwd.  Returns (dx, d_residual, dgamma, dbeta)."""
    import torch
    n, h = dy.shape
    p = DalParams(n_rows=n, hidden=h, p_drop=p_drop, eps=eps, seed=seed, offset=offset, **kw)
    _check(dy, "dy", torch.bfloat16, (n, h))
    _check(z, "z", torch.bfloat16, (n, h))
    _check(mean, "mean", torch.float32, (n,))
    _check(rstd, "rstd", torch.float32, (n,))
    _check(gamma, "gamma", torch.float32, (h,))
    if dz_next is not None:
        _check(dz_next, "dz_next", torch.bfloat16, (n, h))
    dx, dres = torch.empty_like(dy), torch.empty_like(dy)
    dgamma = torch.empty(h, dtype=torch.float32, device=dy.device)
    dbeta = torch.empty(h, dtype=torch.float32, device=dy.device)
    ws_bytes = attn_core_dropout_add_ln_bwd_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dy.device)
    rc = attn_core_dropout_add_ln_bwd(p, dy.data_ptr(), dz_next.data_ptr() if dz_next is not None else 0,
                                      z.data_ptr(), mean.data_ptr(), rstd.data_ptr(), gamma.data_ptr(),
                                      dx.data_ptr(), dres.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(),
                                      workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                      _stream())
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_dropout_add_ln_bwd")
    return dx, dres, dgamma, dbeta


def gelu_fwd(x, out=None):
    """GeLU (tanh form) of a contiguous bf16 CUDA tensor (numel a multiple of 8)."""
    import torch
    _check(x, "x", torch.bfloat16, tuple(x.shape))
    out = torch.empty_like(x) if out is None else out
    rc = attn_core_gelu_fwd(x.numel(), x.data_ptr(), out.data_ptr(), _stream())
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_gelu_fwd")
    return out


def gelu_bwd(x, dy, out=None):
    """dy * GeLU'(x) for contiguous bf16 CUDA tensors of one shape."""
    import torch
    _check(x, "x", torch.bfloat16, tuple(x.shape))
    _check(dy, "dy", torch.bfloat16, tuple(x.shape))
    out = torch.empty_like(x) if out is None else out
    rc = attn_core_gelu_bwd(x.numel(), x.data_ptr(), dy.data_ptr(), out.data_ptr(), _stream())
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_gelu_bwd")
    return out


def _varlen_params(q, k, causal, p_drop, seed, offset, scale, **kw) -> Params:
    _, h_q, d = q.shape
    return Params(b=1, h_q=h_q, h_kv=k.shape[1], s=1, d=d, causal=causal, p_drop=p_drop, scale=scale,
                  seed=seed, offset=offset, **kw)


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k=None, *, causal: bool = True, p_drop: float = 0.0,
               seed: int = 0, offset: int = 0, scale: float = 0.0, **kw):
    """Forward over a packed batch: q [total_q, h_q, d], k/v [total_k, h_kv, d];
    cu_seqlens_* host sequence tables (lists or CPU tensors; their device
    copies are made here).  The batch is one launch per kernel.  Returns (O,
    LSE [h_q, total_q])."""
    import torch
    p = _varlen_params(q, k, causal, p_drop, seed, offset, scale, **kw)
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k] if cu_seqlens_k is not None else None
    _check(q, "q", torch.bfloat16, (cq[-1], p.h_q, p.d))
    _check(k, "k", torch.bfloat16, ((ck or cq)[-1], p.h_kv, p.d))
    _check(v, "v", torch.bfloat16, ((ck or cq)[-1], p.h_kv, p.d))
    o = torch.empty_like(q)
    lse = torch.empty((p.h_q, cq[-1]), dtype=torch.float32, device=q.device)
    tq, tk, dq_ptr, dk_ptr = _device_tables(cq, ck, q.device)
    rc = attn_core_fwd_varlen(p, cq, ck, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), _stream(), cu_q_dev=dq_ptr, cu_k_dev=dk_ptr)
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_fwd_varlen")
    return o, lse


def bwd_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k=None, *, causal: bool = True,
               p_drop: float = 0.0, seed: int = 0, offset: int = 0, scale: float = 0.0, **kw):
    """Recompute-backward over a packed batch.  Returns (dQ, dK, dV)."""
    import torch
    p = _varlen_params(q, k, causal, p_drop, seed, offset, scale, **kw)
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k] if cu_seqlens_k is not None else None
    _check(o, "o", torch.bfloat16, tuple(q.shape))
    _check(dout, "dout", torch.bfloat16, tuple(q.shape))
    _check(lse, "lse", torch.float32, (p.h_q, cq[-1]))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    tq, tk, dq_ptr, dk_ptr = _device_tables(cq, ck, q.device)
    ws_bytes = attn_core_bwd_varlen_workspace_bytes(p, cq, ck, cu_q_dev=dq_ptr, cu_k_dev=dk_ptr)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    rc = attn_core_bwd_varlen(p, cq, ck, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              ws.data_ptr(), ws.numel(), _stream(), cu_q_dev=dq_ptr, cu_k_dev=dk_ptr)
    if rc != OK:
        raise AttnCoreError(rc, "attn_core_bwd_varlen")
    return dq, dk, dv
