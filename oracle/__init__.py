"""fp64 CPU oracle of the causal linear-attention recurrence (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, token by token, double
precision); this module compiles it with gcc and marshals numpy arrays.

Functions follow
  * "History Replays Itself: Unleashing Long-Context Capability in Linear
    Attention" (NoteBank), Sec. 2, Eq. (1) -- the generalised recurrence,
    instantiated with the gated delta rule A_t = alpha_t (I - beta_t k k^T);
  * "BASED：简单线性注意力如何平衡召回能力与生成吞吐" (BASED reading notes),
    Sec. 2.2 (paper Eqs. (1)-(3)) and Sec. 2.3 (paper Eq. (4)) -- the Taylor
    feature map and the s/z normaliser.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

IN_F32 = 0
IN_BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O3, no arch flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O3", "-fPIC", "-shared", "-pthread", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def _declare(lib) -> None:
    i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
    lib.oracle_taylor_dim.restype = i64
    lib.oracle_taylor_dim.argtypes = [i64]
    lib.oracle_taylor_feature.restype = None
    lib.oracle_taylor_feature.argtypes = [vp, i64, vp]
    lib.oracle_taylor.restype = ctypes.c_int
    lib.oracle_taylor.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int, vp, vp, vp,
                                  vp, vp, dp, vp, vp, i64, vp, vp, vp, vp, ctypes.c_int]
    lib.oracle_gdn.restype = ctypes.c_int
    lib.oracle_gdn.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int, vp, vp, vp,
                               vp, vp, dp, vp, vp, i64, vp, vp, ctypes.c_int]
    lib.oracle_gated.restype = ctypes.c_int
    lib.oracle_gated.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int, vp, vp, vp,
                                 vp, vp, dp, vp, vp, i64, vp, vp, ctypes.c_int]


def load_library(path: str):
    """Load a specific compiled oracle (the tests use this to run the pins
    against deliberately broken copies).  Returns the previously loaded one."""
    global _lib
    prev = _lib
    with _lock:
        _lib = None
    lib = ctypes.CDLL(path)
    with _lock:
        _lib = lib
    _declare(lib)
    return prev


def restore_library(prev) -> None:
    global _lib
    with _lock:
        _lib = prev


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _as_input(x):
    """Accept float32 arrays or uint16 arrays holding bf16 bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, IN_F32
    if x.dtype == np.uint16:
        return x, IN_BF16
    raise TypeError(f"oracle inputs must be float32 or uint16 (bf16 bits), got {x.dtype}")


def _samples(t_samples, N):
    if t_samples is None:
        return None, N
    t = np.ascontiguousarray(np.asarray(t_samples, dtype=np.int64))
    return t, int(t.size)


def taylor_dim(dfeat: int) -> int:
    return int(_load().oracle_taylor_dim(dfeat))


def taylor_feature(x) -> np.ndarray:
    """phi(x) = [1, x, vec(x x^T)/sqrt(2)] in fp64 (BASED notes Sec. 2.3)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    D = taylor_dim(x.size)
    out = np.empty(D, dtype=np.float64)
    _load().oracle_taylor_feature(_ptr(x), x.size, _ptr(out))
    return out


def taylor(q, k, v, s_in=None, z_in=None, eps: float = 0.0, t_samples=None,
           want_den: bool = False, nthreads: int | None = None, decay=None):
    """Token-by-token Taylor linear attention with the s/z normaliser.

    q, k: [B,H,N,d'], v: [B,H,N,d_v] (float32 or bf16 bits as uint16).
    decay: None, or the per-head retention lambda ([H] or a scalar): the state
    is scaled by lambda before each write (BASED notes, the decay paragraph
    after Table 7; reading in oracle.c).
    Returns dict(y=[B,H,rows,d_v], s=[B,H,D,d_v], z=[B,H,D], den=[B,H,rows]?).
    """
    q, kind = _as_input(q)
    k, kind_k = _as_input(k)
    v, kind_v = _as_input(v)
    assert kind == kind_k == kind_v, "q, k, v must share one input type"
    B, H, N, df = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3]
    D = taylor_dim(df)
    t, rows = _samples(t_samples, N)
    s_in = None if s_in is None else np.ascontiguousarray(s_in, dtype=np.float64)
    z_in = None if z_in is None else np.ascontiguousarray(z_in, dtype=np.float64)
    if s_in is not None:
        assert s_in.shape == (B, H, D, dv)
    if z_in is not None:
        assert z_in.shape == (B, H, D)
    if decay is not None:
        decay = np.ascontiguousarray(np.broadcast_to(np.asarray(decay, dtype=np.float64), (H,)))
    y = np.zeros((B, H, rows, dv), dtype=np.float64)
    den = np.zeros((B, H, rows), dtype=np.float64) if want_den else None
    s = np.zeros((B, H, D, dv), dtype=np.float64)
    z = np.zeros((B, H, D), dtype=np.float64)
    rc = _load().oracle_taylor(B, H, N, df, dv, kind, _ptr(q), _ptr(k), _ptr(v),
                               _ptr(s_in), _ptr(z_in), float(eps), _ptr(decay), _ptr(t), rows if t is not None else 0,
                               _ptr(y), _ptr(den), _ptr(s), _ptr(z),
                               nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_taylor rejected its arguments (rc={rc})")
    out = {"y": y, "s": s, "z": z}
    if want_den:
        out["den"] = den
    return out


def _gdn_family(fn_name, q, k, v, alpha, beta, S_in=None, q_scale: float = 1.0, t_samples=None,
                nthreads: int | None = None):
    q, kind = _as_input(q)
    k, kind_k = _as_input(k)
    v, kind_v = _as_input(v)
    assert kind == kind_k == kind_v, "q, k, v must share one input type"
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape[:3] == q.shape[:3]
    alpha = np.ascontiguousarray(alpha, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    assert alpha.shape == (B, H, N) and beta.shape == (B, H, N)
    S_in = None if S_in is None else np.ascontiguousarray(S_in, dtype=np.float64)
    if S_in is not None:
        assert S_in.shape == (B, H, dv, dk)
    t, rows = _samples(t_samples, N)
    o = np.zeros((B, H, rows, dv), dtype=np.float64)
    S = np.zeros((B, H, dv, dk), dtype=np.float64)
    rc = getattr(_load(), fn_name)(B, H, N, dk, dv, kind, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(alpha), _ptr(beta), float(q_scale), _ptr(S_in),
                                   _ptr(t), rows if t is not None else 0, _ptr(o), _ptr(S),
                                   nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"{fn_name} rejected its arguments (rc={rc})")
    return {"o": o, "S": S}


def gdn(q, k, v, alpha, beta, S_in=None, q_scale: float = 1.0, t_samples=None,
        nthreads: int | None = None):
    """Token-by-token gated delta rule (NoteBank Sec. 2 Eq. (1),
    A_t = alpha_t (I - beta_t k_t k_t^T)).

    q, k: [B,H,N,d_k], v: [B,H,N,d_v] (float32 or bf16 bits), alpha, beta: [B,H,N] float32.
    Returns dict(o=[B,H,rows,d_v], S=[B,H,d_v,d_k]).
    """
    return _gdn_family("oracle_gdn", q, k, v, alpha, beta, S_in, q_scale, t_samples, nthreads)


def gated(q, k, v, alpha, beta, S_in=None, q_scale: float = 1.0, t_samples=None,
          nthreads: int | None = None):
    """Token-by-token scalar gate (NoteBank Sec. 2 Eq. (1) with A_t = alpha_t I):
    S_t = alpha_t S_{t-1} + beta_t v_t k_t^T, o_t = S_t (q_scale q_t).
    Arguments and result as gdn()."""
    return _gdn_family("oracle_gated", q, k, v, alpha, beta, S_in, q_scale, t_samples, nthreads)


# ---------------------------------------------------------------------------
# State operations between calls.  Each is its plain definition in numpy
# (float32 in, float32 out, one rounding per element exactly as stated).


def state_rescale(states, lam, state_dims: int = 2):
    """NoteBank App. D.1: S <- lambda S per state, lambda in [0, 1]; lambda = 0
    resets (zeros, whatever the state held).  lam: scalar or one per state."""
    x = np.array(states, dtype=np.float32, copy=True)
    lead = x.shape[: x.ndim - state_dims]
    lam = np.broadcast_to(np.asarray(lam, dtype=np.float32), lead)
    for idx in np.ndindex(*lead):
        x[idx] = np.zeros_like(x[idx]) if lam[idx] == 0 else (lam[idx] * x[idx]).astype(np.float32)
    return x


def state_gather(src, index, state_dims: int = 2):
    """NoteBank App. B Alg. 1 (copy(S)): destination i is a copy of source
    state index[i]; src is flattened to [n_states, *state_shape]."""
    src = np.asarray(src, dtype=np.float32)
    shape = src.shape[src.ndim - state_dims:]
    flat = src.reshape((-1,) + shape)
    return np.stack([flat[int(i)].copy() for i in index]) if len(index) else np.zeros((0,) + shape, np.float32)


# ---------------------------------------------------------------------------
# Sliding-window softmax attention (the window layers of BASED: standard
# softmax over the last `window` tokens, BASED notes Sec. 2.4), token by
# token in float64.  Small cases only (plain loops).


def swa(q, k, v, window: int, scale: float, t_samples=None):
    """q, k: [B,H,N,d] (float32 or bf16 bits), v: [B,H,N,d_v].  Returns
    o [B,H,rows,d_v] with o_i = sum_{j=max(0,i-window+1)}^{i}
    softmax_j(scale q_i . k_j) v_j."""
    q = _widen(q)
    k = _widen(k)
    v = _widen(v)
    B, H, N, _ = q.shape
    ts = range(N) if t_samples is None else [int(t) for t in t_samples]
    o = np.zeros((B, H, len(ts), v.shape[-1]))
    for b in range(B):
        for h in range(H):
            for r, i in enumerate(ts):
                lo = max(0, i - window + 1)
                s = np.array([scale * float(np.dot(q[b, h, i], k[b, h, j])) for j in range(lo, i + 1)])
                e = np.exp(s - s.max())
                o[b, h, r] = sum(e[j - lo] * v[b, h, j] for j in range(lo, i + 1)) / e.sum()
    return o


def _widen(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)
