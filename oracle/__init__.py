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


# ---------------------------------------------------------------------------
# NoteBank write side and routing ("History Replays Itself: Unleashing
# Long-Context Capability in Linear Attention", Sec. 2 Eqs. (3)-(5) and
# App. B Eqs. (8)-(9)).  Plain numpy definitions: scores and addresses in
# float64; routing in float32, the precision the pages fix for it (bf16
# addresses and question features converted to fp32, then normalised).
# Readings: a zero vector normalises to zero (so a zero key scores 1); the
# argmaxes take the earliest index on ties; only notes with at least one
# vote are retrieved.


def _unit(x):
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)


def notebank_scores(k, chunk: int, window: int = 48):
    """Distinctiveness of every token in every channel (Eqs. (3), (8)):
    mu_C = unit(mean_{t in C} unit(k_t)) per chunk C of `chunk` tokens
    ([c*chunk, (c+1)*chunk), the last one possibly short) and channel;
    d_t^{l,h} = 1 - <unit(k_t), mu_C(t)>; d_t = mean over the L*H channels;
    w_t = sum_{u=t}^{t+window-1} d_u (the sliding window of App. B.2).
    k: [L, H, N, d] (float32 or bf16 bits).  Returns dict(d_ch [L,H,N],
    d [N], w [N - window + 1])."""
    k = _widen(k)
    L, H, N, _ = k.shape
    kh = _unit(k)
    d_ch = np.zeros((L, H, N))
    for c0 in range(0, N, chunk):
        c1 = min(c0 + chunk, N)
        mu = _unit(kh[:, :, c0:c1].mean(axis=2))
        d_ch[:, :, c0:c1] = 1.0 - np.einsum("lhtd,lhd->lht", kh[:, :, c0:c1], mu)
    d = d_ch.mean(axis=(0, 1))
    w = np.array([d[t:t + window].sum() for t in range(max(N - window + 1, 0))])
    return {"d_ch": d_ch, "d": d, "w": w}


def _round_bf16(x):
    """Round float32 values to bf16 (nearest, ties to even); returned as float64."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def notebank_address(d_ch, q, coords, spans):
    """Note addresses (Eqs. (4), (9)): for note i with token span I_i and
    channel (l,h), t* = argmax_{t in I_i} d_t^{l,h} (earliest on ties) and
    rho_i^{l,h} = P^{l,h} q_{t*}: the query's coordinates coords[l,h, 0..15]
    at t*, stored as bf16.  d_ch: [L,H,N]; q: [L,H,N,d] (float32 or bf16
    bits); coords: [L,H,16]; spans: [n,2] (start, length >= 1).  Returns
    t_star [n,L,H] and rho [n,L,H,16] (the bf16 values as float64)."""
    d_ch = np.asarray(d_ch, dtype=np.float64)
    qf = _widen(q).astype(np.float32)
    L, H, N = d_ch.shape
    spans = np.asarray(spans, dtype=np.int64).reshape(-1, 2)
    n = spans.shape[0]
    t_star = np.zeros((n, L, H), dtype=np.int64)
    rho = np.zeros((n, L, H, coords.shape[-1]))
    for i, (s0, ln) in enumerate(spans):
        for l in range(L):
            for h in range(H):
                seg = d_ch[l, h, s0:s0 + ln]
                t = int(s0 + int(np.argmax(seg)))  # numpy returns the first maximum
                t_star[i, l, h] = t
                rho[i, l, h] = _round_bf16(qf[l, h, t, np.asarray(coords[l, h], dtype=np.int64)])
    return t_star, rho


def notebank_route(rho, u, R: int, positions=None):
    """Routing (Eq. (5)): s_i^{l,h} = max_tau <unit(u_tau^{l,h}), unit(rho_i^{l,h})>
    in float32; each channel votes for argmax_i s_i^{l,h} (earliest on ties);
    V_i = number of votes; the at most R notes with V_i >= 1 and the most
    votes, ties to the earlier-inserted note, returned in text order (by
    `positions`, else insertion order).  rho: [n, J, 16]; u: [J, nq, 16]
    (values of bf16 numbers).  Returns dict(s [n,J], winner [J], votes [n],
    top [<= R])."""
    rho = np.asarray(rho, dtype=np.float32)
    u = np.asarray(u, dtype=np.float32)
    n, J, _ = rho.shape
    rn = (rho / np.linalg.norm(rho, axis=-1, keepdims=True).astype(np.float32)).astype(np.float32)
    un = (u / np.linalg.norm(u, axis=-1, keepdims=True).astype(np.float32)).astype(np.float32)
    s = np.zeros((n, J), dtype=np.float32)
    for j in range(J):
        s[:, j] = np.max(rn[:, j, :] @ un[j].T, axis=1)
    winner = np.array([int(np.argmax(s[:, j])) for j in range(J)], dtype=np.int64)
    votes = np.bincount(winner, minlength=n).astype(np.int64)
    order = sorted((i for i in range(n) if votes[i] >= 1), key=lambda i: (-votes[i], i))[:R]
    pos = np.arange(n) if positions is None else np.asarray(positions)
    top = np.array(sorted(order, key=lambda i: (pos[i], i)), dtype=np.int64)
    return {"s": s, "winner": winner, "votes": votes, "top": top}
