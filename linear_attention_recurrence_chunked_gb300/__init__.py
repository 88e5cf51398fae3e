"""Thin Python binding of the GB300 causal linear-attention library.

Every function here marshals torch tensors into the C ABI of ``include/la.h``
and calls it; all arithmetic runs in the library's CUDA kernels.  There is no
CPU or PyTorch fallback: if the compiled library is missing, importing the
binding's functions raises.

Names follow the C entry points: ``la_based_prefill``, ``la_gdn_prefill``,
``la_decode_step`` (plus the workspace queries and status helpers).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

LA_OK = 0
LA_ERR_INVALID_ARGUMENT = 1
LA_ERR_UNSUPPORTED = 2
LA_ERR_WORKSPACE = 3
LA_ERR_CUDA = 4
LA_ERR_TIMEOUT = 5

LA_DTYPE_F32 = 0
LA_DTYPE_BF16 = 1
LA_VARIANT_TAYLOR = 0
LA_VARIANT_GDN = 1
LA_VARIANT_GATED = 2

TAYLOR_DFEAT = 16
TAYLOR_DV = 64
TAYLOR_D = 1 + TAYLOR_DFEAT + TAYLOR_DFEAT * TAYLOR_DFEAT
GDN_D = 128

_i64 = ctypes.c_int64


class LATensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", _i64), ("stride_h", _i64), ("stride_t", _i64)]


class BasedPrefillArgs(ctypes.Structure):
    _fields_ = [("B", _i64), ("H", _i64), ("N", _i64), ("d_feat", _i64), ("d_v", _i64),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("q", LATensor), ("k", LATensor), ("v", LATensor), ("y", LATensor),
                ("s_in", ctypes.c_void_p), ("z_in", ctypes.c_void_p),
                ("s_out", ctypes.c_void_p), ("z_out", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("decay", ctypes.c_void_p)]


class GdnPrefillArgs(ctypes.Structure):
    _fields_ = [("B", _i64), ("H", _i64), ("N", _i64), ("d_k", _i64), ("d_v", _i64),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("q", LATensor), ("k", LATensor), ("v", LATensor), ("o", LATensor),
                ("alpha", LATensor), ("beta", LATensor),
                ("q_scale", ctypes.c_float),
                ("S_in", ctypes.c_void_p), ("S_out", ctypes.c_void_p)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("S", _i64), ("H", _i64), ("d_k", _i64), ("d_v", _i64),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("state", ctypes.c_void_p), ("z", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("q_scale", ctypes.c_float), ("decay", ctypes.c_void_p)]


EXPORTED = ("la_based_prefill", "la_gdn_prefill", "la_gated_prefill", "la_decode_step", "la_based_prefill_workspace_size",
            "la_gdn_prefill_workspace_size", "la_gdn_prefill_workspace_size_min", "la_gdn_prefill_noalloc", "la_device_status",
            "la_state_rescale", "la_state_gather", "la_swa_decode_step", "la_notebank_scores", "la_notebank_address",
            "la_notebank_route", "la_selftest_bounded_wait", "la_status_string", "la_abi_version",
            "la_last_cuda_error", "la_cuda_error_name")


class NotebankScoresArgs(ctypes.Structure):
    _fields_ = [("L", _i64), ("H", _i64), ("N", _i64), ("d", _i64), ("in_dtype", ctypes.c_int),
                ("k", LATensor), ("chunk", _i64), ("window", _i64),
                ("d_ch", ctypes.c_void_p), ("d_mean", ctypes.c_void_p), ("w", ctypes.c_void_p)]


class NotebankAddressArgs(ctypes.Structure):
    _fields_ = [("L", _i64), ("H", _i64), ("N", _i64), ("d", _i64), ("n_notes", _i64), ("in_dtype", ctypes.c_int),
                ("q", LATensor), ("d_ch", ctypes.c_void_p), ("coords", ctypes.c_void_p), ("spans", ctypes.c_void_p),
                ("t_star", ctypes.c_void_p), ("rho", ctypes.c_void_p)]


class NotebankRouteArgs(ctypes.Structure):
    _fields_ = [("n_notes", _i64), ("J", _i64), ("n_q", _i64), ("R", _i64),
                ("rho", ctypes.c_void_p), ("u", ctypes.c_void_p), ("positions", ctypes.c_void_p),
                ("s", ctypes.c_void_p), ("winner", ctypes.c_void_p), ("votes", ctypes.c_void_p),
                ("top", ctypes.c_void_p)]


class SwaDecodeArgs(ctypes.Structure):
    _fields_ = [("S", _i64), ("H", _i64), ("d", _i64), ("window", _i64),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("scale", ctypes.c_float)]


class LAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {la_status_string(status)} (status {status})"
        if status == LA_ERR_CUDA:
            lib = load_library()
            code = int(lib.la_last_cuda_error())
            msg += f"; CUDA error {code} ({lib.la_cuda_error_name(code).decode()})"
        super().__init__(msg)


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Load the compiled library (build it first with ``_build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built ({p} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp = ctypes.c_void_p
    lib.la_based_prefill.restype = ctypes.c_int
    lib.la_based_prefill.argtypes = [ctypes.POINTER(BasedPrefillArgs), vp, ctypes.c_size_t, vp]
    lib.la_gdn_prefill.restype = ctypes.c_int
    lib.la_gdn_prefill.argtypes = [ctypes.POINTER(GdnPrefillArgs), vp, ctypes.c_size_t, vp]
    lib.la_gated_prefill.restype = ctypes.c_int
    lib.la_gated_prefill.argtypes = [ctypes.POINTER(GdnPrefillArgs), vp, ctypes.c_size_t, vp]
    lib.la_gdn_prefill_noalloc.restype = ctypes.c_int
    lib.la_gdn_prefill_noalloc.argtypes = [ctypes.POINTER(GdnPrefillArgs), vp]
    lib.la_decode_step.restype = ctypes.c_int
    lib.la_decode_step.argtypes = [ctypes.POINTER(DecodeArgs), vp]
    lib.la_based_prefill_workspace_size.restype = ctypes.c_size_t
    lib.la_based_prefill_workspace_size.argtypes = [ctypes.POINTER(BasedPrefillArgs)]
    lib.la_gdn_prefill_workspace_size.restype = ctypes.c_size_t
    lib.la_gdn_prefill_workspace_size.argtypes = [ctypes.POINTER(GdnPrefillArgs)]
    lib.la_gdn_prefill_workspace_size_min.restype = ctypes.c_size_t
    lib.la_gdn_prefill_workspace_size_min.argtypes = [ctypes.POINTER(GdnPrefillArgs)]
    lib.la_swa_decode_step.restype = ctypes.c_int
    lib.la_swa_decode_step.argtypes = [ctypes.POINTER(SwaDecodeArgs), vp]
    lib.la_notebank_scores.restype = ctypes.c_int
    lib.la_notebank_scores.argtypes = [ctypes.POINTER(NotebankScoresArgs), vp]
    lib.la_notebank_address.restype = ctypes.c_int
    lib.la_notebank_address.argtypes = [ctypes.POINTER(NotebankAddressArgs), vp]
    lib.la_notebank_route.restype = ctypes.c_int
    lib.la_notebank_route.argtypes = [ctypes.POINTER(NotebankRouteArgs), vp]
    lib.la_state_rescale.restype = ctypes.c_int
    lib.la_state_rescale.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_float, vp]
    lib.la_state_gather.restype = ctypes.c_int
    lib.la_state_gather.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp]
    lib.la_device_status.restype = ctypes.c_int
    lib.la_device_status.argtypes = [vp, ctypes.c_int]
    lib.la_selftest_bounded_wait.restype = ctypes.c_int
    lib.la_selftest_bounded_wait.argtypes = [ctypes.c_int, ctypes.c_int64, vp]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_status_string.argtypes = [ctypes.c_int]
    lib.la_last_cuda_error.restype = ctypes.c_int
    lib.la_last_cuda_error.argtypes = []
    lib.la_cuda_error_name.restype = ctypes.c_char_p
    lib.la_cuda_error_name.argtypes = [ctypes.c_int]
    lib.la_abi_version.restype = ctypes.c_int
    lib.la_abi_version.argtypes = []
    if path is None:
        _lib = lib
    return lib


def la_status_string(status: int) -> str:
    return load_library().la_status_string(int(status)).decode()


def la_abi_version() -> int:
    return int(load_library().la_abi_version())


# ---------------------------------------------------------------------------
# marshalling helpers


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return LA_DTYPE_F32
    if t == torch.bfloat16:
        return LA_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t}; use float32 or bfloat16")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _view4(t: torch.Tensor) -> LATensor:
    """[B,H,N,d] tensor -> strided view (the d axis must be contiguous)."""
    if t.dim() != 4:
        raise ValueError(f"expected a [B,H,N,d] tensor, got shape {tuple(t.shape)}")
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError("the feature axis must be contiguous")
    return LATensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def _gate3(t: torch.Tensor) -> LATensor:
    """[B,H,N] fp32 gate -> view with its N axis as the token axis."""
    if t.dim() != 3 or t.dtype != torch.float32:
        raise ValueError("alpha/beta must be float32 [B,H,N]")
    return LATensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must live on a CUDA device")


def _workspace(nbytes: int, workspace, device):
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws, nbytes


# ---------------------------------------------------------------------------
# entry points


def _based_args(q, k, v, y, s_in, z_in, s_out, z_out, eps, decay=None):
    B, H, N, F = q.shape
    return BasedPrefillArgs(B, H, N, F, v.shape[-1], _dtype_code(q.dtype), _dtype_code(y.dtype),
                            _view4(q), _view4(k), _view4(v), _view4(y),
                            _ptr(s_in), _ptr(z_in), _ptr(s_out), _ptr(z_out), float(eps), _ptr(decay))


def _check_decay(decay, H):
    if decay is not None and (decay.dtype != torch.float32 or decay.shape != (H,) or not decay.is_contiguous()):
        raise ValueError("decay must be a contiguous float32 tensor of shape [H]")


def la_based_prefill_workspace_size(q, k, v, y=None) -> int:
    y = y if y is not None else v
    a = _based_args(q, k, v, y, None, None, None, None, 0.0)
    return int(load_library().la_based_prefill_workspace_size(ctypes.byref(a)))


def la_based_prefill(q, k, v, y=None, s_in=None, z_in=None, s_out=None, z_out=None, eps: float = 0.0,
                     out_dtype=None, workspace=None, stream=None, decay=None):
    """Chunked Taylor (BASED) prefill.  Returns (y, s_out, z_out).

    q, k: [B,H,N,16], v: [B,H,N,64] (fp32 or bf16); states fp32
    s: [B,H,273,64], z: [B,H,273]; decay: None or fp32 [H], the per-head
    retention lambda (s_i = lambda s_{i-1} + phi(k_i) v_i^T, z likewise)."""
    lib = load_library()
    _check_cuda(q, k, v, y, s_in, z_in, s_out, z_out, decay)
    B, H, N, _ = q.shape
    _check_decay(decay, H)
    dv = v.shape[-1]
    if y is None:
        y = torch.empty((B, H, N, dv), dtype=out_dtype or q.dtype, device=q.device)
    if s_out is None:
        s_out = torch.empty((B, H, TAYLOR_D, dv), dtype=torch.float32, device=q.device)
    if z_out is None:
        z_out = torch.empty((B, H, TAYLOR_D), dtype=torch.float32, device=q.device)
    for name, t in (("s_in", s_in), ("z_in", z_in), ("s_out", s_out), ("z_out", z_out)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 tensor")
    a = _based_args(q, k, v, y, s_in, z_in, s_out, z_out, eps, decay)
    need = int(lib.la_based_prefill_workspace_size(ctypes.byref(a)))
    ws, ws_bytes = _workspace(need, workspace, q.device)
    st = lib.la_based_prefill(ctypes.byref(a), _ptr(ws) if isinstance(ws, torch.Tensor) else ws, ws_bytes,
                              _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_based_prefill")
    return y, s_out, z_out


def _gdn_args(q, k, v, o, alpha, beta, S_in, S_out, q_scale):
    B, H, N, dk = q.shape
    return GdnPrefillArgs(B, H, N, dk, v.shape[-1], _dtype_code(q.dtype), _dtype_code(o.dtype),
                          _view4(q), _view4(k), _view4(v), _view4(o), _gate3(alpha), _gate3(beta),
                          float(q_scale), _ptr(S_in), _ptr(S_out))


def la_gdn_prefill_workspace_size(q, k, v, alpha, beta, o=None) -> int:
    o = o if o is not None else v
    a = _gdn_args(q, k, v, o, alpha, beta, None, None, 1.0)
    return int(load_library().la_gdn_prefill_workspace_size(ctypes.byref(a)))


def la_gdn_prefill_workspace_size_min(q, k, v, alpha, beta, o=None) -> int:
    """Smallest workspace la_gdn_prefill accepts (selects the one-kernel schedule)."""
    o = o if o is not None else v
    a = _gdn_args(q, k, v, o, alpha, beta, None, None, 1.0)
    return int(load_library().la_gdn_prefill_workspace_size_min(ctypes.byref(a)))


def _gdn_family_prefill(fn_name, q, k, v, alpha, beta, o, S_in, S_out, q_scale, out_dtype, workspace, stream):
    lib = load_library()
    _check_cuda(q, k, v, alpha, beta, o, S_in, S_out)
    B, H, N, _ = q.shape
    dv = v.shape[-1]
    if o is None:
        o = torch.empty((B, H, N, dv), dtype=out_dtype or q.dtype, device=q.device)
    if S_out is None:
        S_out = torch.empty((B, H, dv, q.shape[-1]), dtype=torch.float32, device=q.device)
    for name, t in (("S_in", S_in), ("S_out", S_out)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 tensor")
    a = _gdn_args(q, k, v, o, alpha, beta, S_in, S_out, q_scale)
    need = int(lib.la_gdn_prefill_workspace_size(ctypes.byref(a)))
    ws, ws_bytes = _workspace(need, workspace, q.device)
    st = getattr(lib, fn_name)(ctypes.byref(a), _ptr(ws) if isinstance(ws, torch.Tensor) else ws, ws_bytes,
                               _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, fn_name)
    return o, S_out


def la_gdn_prefill(q, k, v, alpha, beta, o=None, S_in=None, S_out=None, q_scale: float = 1.0,
                   out_dtype=None, workspace=None, stream=None):
    """Chunked gated-delta-rule prefill.  Returns (o, S_out).

    q, k, v: [B,H,N,128] (fp32 or bf16); alpha, beta: fp32 [B,H,N];
    S: fp32 [B,H,128,128] (row = value index).  workspace: optional uint8
    device tensor; by default la_gdn_prefill_workspace_size bytes are
    allocated (the records schedule); a smaller one of at least
    la_gdn_prefill_workspace_size_min bytes selects the one-kernel schedule."""
    return _gdn_family_prefill("la_gdn_prefill", q, k, v, alpha, beta, o, S_in, S_out, q_scale, out_dtype,
                               workspace, stream)


def la_gated_prefill(q, k, v, alpha, beta, o=None, S_in=None, S_out=None, q_scale: float = 1.0,
                     out_dtype=None, workspace=None, stream=None):
    """Chunked scalar-gate prefill, S_t = alpha_t S_{t-1} + beta_t v_t k_t^T,
    o_t = S_t (q_scale q_t).  Arguments, workspace and result as la_gdn_prefill."""
    return _gdn_family_prefill("la_gated_prefill", q, k, v, alpha, beta, o, S_in, S_out, q_scale, out_dtype,
                               workspace, stream)


def la_gdn_prefill_noalloc(q, k, v, alpha, beta, o, S_out, S_in=None, q_scale: float = 1.0, stream=None):
    """la_gdn_prefill without a workspace, for callers that cannot allocate:
    the library's fixed 16 MiB device array serves as scratch (see
    include/la.h).  o and S_out must be preallocated by the caller.
    Returns (o, S_out)."""
    lib = load_library()
    _check_cuda(q, k, v, alpha, beta, o, S_in, S_out)
    a = _gdn_args(q, k, v, o, alpha, beta, S_in, S_out, q_scale)
    st = lib.la_gdn_prefill_noalloc(ctypes.byref(a), _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_gdn_prefill_noalloc")
    return o, S_out


def la_decode_step(variant: int, q, k, v, state, z=None, alpha=None, beta=None, out=None,
                   eps: float = 0.0, q_scale: float = 1.0, out_dtype=None, stream=None, decay=None):
    """One decode step, state (and z) updated in place.  Returns out [S,H,d_v].

    GDN and the scalar gate (LA_VARIANT_GATED): q, k, v [S,H,128], alpha, beta
    fp32 [S,H], state fp32 [S,H,128,128].
    Taylor: q, k [S,H,16], v [S,H,64], state fp32 [S,H,273,64], z fp32 [S,H,273];
    decay: None or fp32 [H] per-head retention, as in la_based_prefill."""
    lib = load_library()
    _check_cuda(q, k, v, state, z, alpha, beta, out, decay)
    for name, t in (("q", q), ("k", k), ("v", v), ("state", state), ("z", z), ("alpha", alpha),
                    ("beta", beta), ("out", out)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    S, H, dk = q.shape
    dv = v.shape[-1]
    _check_decay(decay, H)
    if out is None:
        out = torch.empty((S, H, dv), dtype=out_dtype or q.dtype, device=q.device)
    a = DecodeArgs(int(variant), S, H, dk, dv, _dtype_code(q.dtype), _dtype_code(out.dtype),
                   _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(out), _ptr(state), _ptr(z),
                   float(eps), float(q_scale), _ptr(decay))
    st = lib.la_decode_step(ctypes.byref(a), _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_decode_step")
    return out


def _state_split(t, state_dims: int):
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError("states must be contiguous float32 tensors")
    if not 0 <= state_dims <= t.dim():
        raise ValueError("state_dims out of range")
    per = 1
    for d in t.shape[t.dim() - state_dims:]:
        per *= int(d)
    n = t.numel() // per if per else 0
    return n, per


def la_state_rescale(states, lam, state_dims: int = 2, stream=None):
    """S <- lambda S for every state in `states` (its last `state_dims` dims
    form one state: 2 for GDN S or Taylor s, 1 for Taylor z), in place.
    lam: a float, or a float32 device tensor with one factor per state.
    A factor of 0 resets the state to zeros.  Returns `states`."""
    lib = load_library()
    _check_cuda(states, lam if isinstance(lam, torch.Tensor) else None)
    n, per = _state_split(states, state_dims)
    lam_t = lam if isinstance(lam, torch.Tensor) else None
    if lam_t is not None and (lam_t.dtype != torch.float32 or not lam_t.is_contiguous() or lam_t.numel() != n):
        raise ValueError("lam must be a contiguous float32 tensor with one factor per state")
    st = lib.la_state_rescale(_ptr(states), n, per, _ptr(lam_t), 0.0 if lam_t is not None else float(lam),
                              _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_state_rescale")
    return states


def la_state_gather(src, index, state_dims: int = 2, dst=None, stream=None):
    """dst[i] = src[index[i]] over states (the last `state_dims` dims of src
    form one state); index: int64 device tensor.  Copies one state to
    several destinations, reorders, or keeps a branch point.  Returns dst,
    shaped [len(index), *state_shape]."""
    lib = load_library()
    _check_cuda(src, index, dst)
    n_src, per = _state_split(src, state_dims)
    if index.dtype != torch.int64 or not index.is_contiguous():
        raise ValueError("index must be a contiguous int64 tensor")
    shape = tuple(src.shape[src.dim() - state_dims:])
    if dst is None:
        dst = torch.empty((index.numel(), *shape), dtype=torch.float32, device=src.device)
    n_dst, per_d = _state_split(dst, state_dims)
    if per_d != per or n_dst != index.numel():
        raise ValueError("dst must hold len(index) states of the source's shape")
    st = lib.la_state_gather(_ptr(dst), _ptr(src), _ptr(index), n_dst, n_src, per, _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_state_gather")
    return dst


def la_swa_decode_step(q, k, v, k_cache, v_cache, pos, out=None, scale: float | None = None, out_dtype=None,
                       stream=None):
    """One sliding-window softmax-attention decode step (the window layers of
    BASED).  q, k, v: [S,H,d]; k_cache, v_cache: [S,H,window,d] ring buffers
    (token p in slot p % window), updated in place; pos: int64 [S] tokens
    already seen per sequence (not advanced here).  scale defaults to
    1/sqrt(d).  Returns out [S,H,d]."""
    lib = load_library()
    _check_cuda(q, k, v, k_cache, v_cache, pos, out)
    for name, t in (("q", q), ("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache), ("pos", pos),
                    ("out", out)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if pos.dtype != torch.int64:
        raise ValueError("pos must be int64")
    S, H, d = q.shape
    window = k_cache.shape[2]
    if out is None:
        out = torch.empty((S, H, d), dtype=out_dtype or q.dtype, device=q.device)
    a = SwaDecodeArgs(S, H, d, window, _dtype_code(q.dtype), _dtype_code(out.dtype), _ptr(q), _ptr(k), _ptr(v),
                      _ptr(k_cache), _ptr(v_cache), _ptr(pos), _ptr(out),
                      float(scale if scale is not None else d ** -0.5))
    st = lib.la_swa_decode_step(ctypes.byref(a), _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_swa_decode_step")
    return out


NOTE_ADDR_DIMS = 16  # d_rho


def la_notebank_scores(k, chunk: int = 512, window: int = 48, stream=None):
    """NoteBank write-side scores (NoteBank Sec. 2 Eqs. (3), (8)).  k: [L, H, N, d]
    (the L x H channels of one document; fp32 or bf16, d a multiple of 32 up
    to 256).  Returns (d_ch [L,H,N], d_mean [N], w [N - window + 1]) fp32."""
    lib = load_library()
    _check_cuda(k)
    L, H, N, d = k.shape
    d_ch = torch.empty((L, H, N), dtype=torch.float32, device=k.device)
    d_mean = torch.empty((N,), dtype=torch.float32, device=k.device)
    w = torch.empty((max(N - window + 1, 0),), dtype=torch.float32, device=k.device)
    a = NotebankScoresArgs(L, H, N, d, _dtype_code(k.dtype), _view4(k), int(chunk), int(window),
                           _ptr(d_ch), _ptr(d_mean), _ptr(w) if w.numel() else None)
    st = lib.la_notebank_scores(ctypes.byref(a), _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_notebank_scores")
    return d_ch, d_mean, w


def la_notebank_address(d_ch, q, coords, spans, stream=None):
    """NoteBank note addresses (Eqs. (4), (9)): per note span and channel, the
    argmax of d_ch over the span and the query's 16 `coords` there as bf16.
    d_ch [L,H,N] fp32, q [L,H,N,d], coords int32 [L,H,16], spans int64 [n,2]
    (start, length), all on the device.  Returns (t_star int32 [n,L,H],
    rho bf16 [n,L,H,16])."""
    lib = load_library()
    _check_cuda(d_ch, q, coords, spans)
    L, H, N, d = q.shape
    n = spans.shape[0]
    if coords.dtype != torch.int32 or spans.dtype != torch.int64 or not coords.is_contiguous() or not spans.is_contiguous():
        raise ValueError("coords must be contiguous int32 and spans contiguous int64")
    t_star = torch.empty((n, L, H), dtype=torch.int32, device=q.device)
    rho = torch.empty((n, L, H, NOTE_ADDR_DIMS), dtype=torch.bfloat16, device=q.device)
    a = NotebankAddressArgs(L, H, N, d, n, _dtype_code(q.dtype), _view4(q), _ptr(d_ch), _ptr(coords), _ptr(spans),
                            _ptr(t_star), _ptr(rho))
    st = lib.la_notebank_address(ctypes.byref(a), _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_notebank_address")
    return t_star, rho


def la_notebank_route(rho, u, R: int, positions=None, want_scores: bool = False, stream=None):
    """NoteBank routing (Eq. (5)).  rho bf16 [n, J, 16] (notes in insertion
    order), u bf16 [J, n_q, 16] (question features), positions int64 [n] or
    None.  Returns (top int32 [R] in text order, -1 padded, winner int32 [J],
    votes int32 [n], s fp32 [n, J] or None)."""
    lib = load_library()
    _check_cuda(rho, u, positions)
    n, J = rho.shape[0], u.shape[0]
    for name, t in (("rho", rho), ("u", u)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    dev = u.device
    winner = torch.empty((J,), dtype=torch.int32, device=dev)
    votes = torch.empty((n,), dtype=torch.int32, device=dev)
    top = torch.empty((R,), dtype=torch.int32, device=dev)
    s = torch.empty((n, J), dtype=torch.float32, device=dev) if want_scores else None
    a = NotebankRouteArgs(n, J, u.shape[1], int(R), _ptr(rho), _ptr(u), _ptr(positions), _ptr(s), _ptr(winner),
                          _ptr(votes), _ptr(top))
    st = lib.la_notebank_route(ctypes.byref(a), _stream_handle(stream))
    if st != LA_OK:
        raise LAError(st, "la_notebank_route")
    return top, winner, votes, s


def la_device_status(stream=None, clear: bool = True) -> int:
    return int(load_library().la_device_status(_stream_handle(stream), 1 if clear else 0))


def la_selftest_bounded_wait(arrive: bool, limit_ns: int, stream=None) -> int:
    """Launch the bounded-wait self-test (see include/la.h); returns the launch status."""
    return int(load_library().la_selftest_bounded_wait(1 if arrive else 0, int(limit_ns), _stream_handle(stream)))
