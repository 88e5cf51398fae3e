"""Pins for the fp64 oracle, checked against things other than the oracle itself.

Each test states what fixes the expected value: a closed form the pages give,
brute force of a different formula (the quadratic/attention form, the dense
matrix form of the recurrence), exact rational arithmetic, invariants and
special cases that reduce to textbook results, or dimension facts the pages
print (tests/golden/).  CPU only.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def rel_err(x, ref):
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-300))


def taylor_kernel(q, k):
    """K(q,k) = 1 + q.k + (q.k)^2/2 (BASED notes Sec. 2.3, paper Eq. (4))."""
    t = float(np.dot(q, k))
    return 1.0 + t + 0.5 * t * t


def f32(shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


# --------------------------------------------------------------------------
# Feature map: closed form and dimensions


@pytest.mark.parametrize("df", [1, 2, 4, 16])
def test_feature_inner_product_is_closed_form_kernel(df):
    for _ in range(20):
        q = rng.standard_normal(df)
        k = rng.standard_normal(df)
        got = float(np.dot(oracle.taylor_feature(q), oracle.taylor_feature(k)))
        assert got == pytest.approx(taylor_kernel(q, k), rel=1e-13, abs=1e-13)


def test_feature_dims_match_pages():
    g = json.load(open(os.path.join(GOLDEN, "taylor_feature_dims.json")))
    assert oracle.taylor_dim(16) == g["full_outer_product"]["16"]
    phi = oracle.taylor_feature(rng.standard_normal(16))
    assert phi.size == 273
    assert 273 <= g["hardware_padded_multiple_of_64"]["16"] and g["hardware_padded_multiple_of_64"]["16"] % 64 == 0
    # The full map repeats each cross term twice; the number of distinct
    # monomials is the compact dimension the pages print.
    for df_s, compact in g["compact_symmetric"].items():
        if not df_s.isdigit():
            continue
        df = int(df_s)
        x = rng.standard_normal(df) + 3.0  # generic point: distinct monomials have distinct values
        phi = oracle.taylor_feature(x)
        assert phi.size == 1 + df + df * df
        assert len(np.unique(np.round(phi, 12))) == compact


def test_feature_layout_row_major_and_constant_term():
    x = np.arange(1, 5, dtype=np.float64)
    phi = oracle.taylor_feature(x)
    assert phi[0] == 1.0
    assert np.array_equal(phi[1:5], x)
    quad = phi[5:].reshape(4, 4)
    assert np.allclose(quad, np.outer(x, x) / math.sqrt(2.0), rtol=0, atol=1e-15)


def test_denominator_positivity_identity():
    # 1 + t + t^2/2 = ((t+1)^2 + 1)/2 >= 1/2  (BASED notes Sec. 2.3)
    for t in np.linspace(-10, 10, 101):
        assert 1 + t + t * t / 2 == pytest.approx(((t + 1) ** 2 + 1) / 2, rel=1e-14)
        assert 1 + t + t * t / 2 >= 0.5


# --------------------------------------------------------------------------
# Taylor recurrence vs the quadratic (attention) form


def quadratic_form(q, k, v):
    """y_i = sum_{j<=i} K(q_i,k_j) v_j / sum_{j<=i} K(q_i,k_j), by brute force."""
    B, H, N, _ = q.shape
    y = np.zeros(v.shape, dtype=np.float64)
    den = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                w = np.array([taylor_kernel(q[b, h, i].astype(np.float64), k[b, h, j].astype(np.float64))
                              for j in range(i + 1)])
                y[b, h, i] = w @ v[b, h, : i + 1].astype(np.float64) / w.sum()
                den[b, h, i] = w.sum()
    return y, den


@pytest.mark.parametrize("df,dv,N", [(4, 5, 37), (16, 8, 40)])
def test_taylor_equals_quadratic_form(df, dv, N):
    q = f32((1, 2, N, df), 1 / math.sqrt(df))
    k = f32((1, 2, N, df), 1 / math.sqrt(df))
    v = f32((1, 2, N, dv))
    out = oracle.taylor(q, k, v, want_den=True, nthreads=2)
    y_ref, den_ref = quadratic_form(q, k, v)
    assert rel_err(out["y"], y_ref) < 1e-12
    assert rel_err(out["den"], den_ref) < 1e-12


def test_taylor_exact_rational_example():
    """Dyadic inputs, exact Fraction arithmetic of the quadratic form."""
    q = np.array([[0.5, -0.25], [1.0, 0.75], [-0.5, 0.5], [0.25, 0.125]], dtype=np.float32)
    k = np.array([[0.25, 0.5], [-1.0, 0.5], [0.75, -0.25], [0.5, 0.5]], dtype=np.float32)
    v = np.array([[1.0, -2.0], [0.5, 3.0], [-1.5, 0.25], [2.0, 1.0]], dtype=np.float32)
    out = oracle.taylor(q[None, None], k[None, None], v[None, None])

    def K(a, b):
        t = sum(Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b))
        return 1 + t + t * t / 2

    for i in range(4):
        w = [K(q[i], k[j]) for j in range(i + 1)]
        for c in range(2):
            exact = sum(wj * Fraction(float(v[j, c])) for j, wj in enumerate(w)) / sum(w)
            assert out["y"][0, 0, i, c] == pytest.approx(float(exact), rel=1e-15, abs=1e-15)


def test_taylor_state_invariants():
    df, dv, N = 16, 8, 50
    q = f32((2, 2, N, df), 0.25)
    k = f32((2, 2, N, df), 0.25)
    v = f32((2, 2, N, dv))
    out = oracle.taylor(q, k, v, want_den=True)
    s, z = out["s"], out["z"]
    kd, vd = k.astype(np.float64), v.astype(np.float64)
    # constant row: z[0] = N, s[0] = sum v
    assert np.all(z[..., 0] == N)
    assert np.allclose(s[..., 0, :], vd.sum(axis=2), rtol=1e-13, atol=1e-12)
    # linear rows: sum k v^T
    assert np.allclose(s[..., 1:1 + df, :], np.einsum("bhna,bhnc->bhac", kd, vd), rtol=1e-12, atol=1e-12)
    # quadratic rows, row-major (a,b): sum k_a k_b v / sqrt 2 ; symmetric bit-for-bit
    quad = s[..., 1 + df:, :].reshape(2, 2, df, df, dv)
    ref = np.einsum("xhna,xhnm,xhnc->xhamc", kd, kd, vd) / math.sqrt(2.0)
    assert np.allclose(quad, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(quad, np.swapaxes(quad, 2, 3))
    # z rows: sum of features
    assert np.allclose(z[..., 1:1 + df], kd.sum(axis=2), rtol=1e-12, atol=1e-12)
    # denominator >= i/2 for the 1-based prefix length i
    i = np.arange(1, N + 1)
    assert np.all(out["den"] >= i / 2 - 1e-12)


def test_taylor_zero_query_is_running_mean():
    df, dv, N = 16, 6, 30
    q = np.zeros((1, 1, N, df), np.float32)
    k = f32((1, 1, N, df), 0.25)
    v = f32((1, 1, N, dv))
    y = oracle.taylor(q, k, v)["y"][0, 0]
    ref = np.cumsum(v[0, 0].astype(np.float64), axis=0) / np.arange(1, N + 1)[:, None]
    assert rel_err(y, ref) < 1e-13


def test_taylor_split_resume_and_samples():
    df, dv, N = 16, 8, 45
    q = f32((1, 3, N, df), 0.25)
    k = f32((1, 3, N, df), 0.25)
    v = f32((1, 3, N, dv))
    full = oracle.taylor(q, k, v)
    a = oracle.taylor(q[:, :, :17], k[:, :, :17], v[:, :, :17])
    b = oracle.taylor(q[:, :, 17:], k[:, :, 17:], v[:, :, 17:], s_in=a["s"], z_in=a["z"])
    assert rel_err(np.concatenate([a["y"], b["y"]], axis=2), full["y"]) < 1e-13
    assert rel_err(b["s"], full["s"]) < 1e-13 and rel_err(b["z"], full["z"]) < 1e-13
    t = [0, 5, 17, 44]
    smp = oracle.taylor(q, k, v, t_samples=t)
    assert np.array_equal(smp["y"], full["y"][:, :, t])


# --------------------------------------------------------------------------
# Taylor with a fixed per-head decay (BASED notes, the decay paragraph after
# Table 7; reading: s_i = lambda s_{i-1} + phi(k_i) v_i^T, z likewise)


def decayed_quadratic_form(q, k, v, lam, s0_probe=None):
    """y_i = sum_{j<=i} lam^(i-j) K(q_i,k_j) v_j / sum_{j<=i} lam^(i-j) K(q_i,k_j), by brute force."""
    B, H, N, _ = q.shape
    y = np.zeros(v.shape, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                w = np.array([lam[h] ** (i - j) * taylor_kernel(q[b, h, i].astype(np.float64),
                                                               k[b, h, j].astype(np.float64))
                              for j in range(i + 1)])
                y[b, h, i] = w @ v[b, h, : i + 1].astype(np.float64) / w.sum()
    return y


def test_taylor_decay_one_is_undecayed():
    q, k, v = f32((1, 2, 30, 16), 0.25), f32((1, 2, 30, 16), 0.25), f32((1, 2, 30, 8))
    a = oracle.taylor(q, k, v)
    b = oracle.taylor(q, k, v, decay=np.ones(2))
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["s"], b["s"]) and np.array_equal(a["z"], b["z"])


@pytest.mark.parametrize("df,dv,N", [(4, 5, 33), (16, 8, 40)])
def test_taylor_decay_equals_weighted_quadratic_form(df, dv, N):
    q = f32((1, 3, N, df), 1 / math.sqrt(df))
    k = f32((1, 3, N, df), 1 / math.sqrt(df))
    v = f32((1, 3, N, dv))
    lam = np.array([0.9, 0.5, 0.99])
    out = oracle.taylor(q, k, v, decay=lam, nthreads=2)
    assert rel_err(out["y"], decayed_quadratic_form(q, k, v, lam)) < 1e-12
    # the final state read by a probe x: phi(x)^T s_N = sum_j lam^(N-1-j) K(x, k_j) v_j
    x = rng.standard_normal(df) / math.sqrt(df)
    phx = oracle.taylor_feature(x)
    for h in range(3):
        w = np.array([lam[h] ** (N - 1 - j) * taylor_kernel(x, k[0, h, j].astype(np.float64)) for j in range(N)])
        assert rel_err(phx @ out["s"][0, h], w @ v[0, h].astype(np.float64)) < 1e-12
        assert phx @ out["z"][0, h] == pytest.approx(w.sum(), rel=1e-12)


def test_taylor_decay_zero_keeps_only_the_current_token():
    q, k, v = f32((1, 1, 12, 16), 0.25), f32((1, 1, 12, 16), 0.25), f32((1, 1, 12, 6))
    s0 = rng.standard_normal((1, 1, 273, 6))
    z0 = np.abs(rng.standard_normal((1, 1, 273)))
    y = oracle.taylor(q, k, v, s_in=s0, z_in=z0, decay=0.0)["y"][0, 0]
    assert rel_err(y, v[0, 0].astype(np.float64)) < 1e-13


def test_taylor_decay_split_resume_with_state():
    df, dv, N = 16, 8, 41
    q, k, v = f32((1, 2, N, df), 0.25), f32((1, 2, N, df), 0.25), f32((1, 2, N, dv))
    lam = np.array([0.95, 0.7])
    s0 = rng.standard_normal((1, 2, 273, dv)) * 0.1
    z0 = np.abs(rng.standard_normal((1, 2, 273))) * 0.1
    full = oracle.taylor(q, k, v, s_in=s0, z_in=z0, decay=lam)
    a = oracle.taylor(q[:, :, :19], k[:, :, :19], v[:, :, :19], s_in=s0, z_in=z0, decay=lam)
    b = oracle.taylor(q[:, :, 19:], k[:, :, 19:], v[:, :, 19:], s_in=a["s"], z_in=a["z"], decay=lam)
    assert rel_err(np.concatenate([a["y"], b["y"]], axis=2), full["y"]) < 1e-13
    assert rel_err(b["s"], full["s"]) < 1e-13 and rel_err(b["z"], full["z"]) < 1e-13
    # the recurrence is linear in (s0, v): with v = 0 the incoming state's share of s_N is lam^N s0
    zero_v = oracle.taylor(q, k, np.zeros_like(v), s_in=s0, z_in=z0, decay=lam)
    no_s0 = oracle.taylor(q, k, np.zeros_like(v), decay=lam)
    for h in range(2):
        assert rel_err(zero_v["s"][0, h] - no_s0["s"][0, h], lam[h] ** N * s0[0, h]) < 1e-12


def test_bf16_bits_decode_like_float32():
    x = f32((1, 1, 20, 16), 0.25)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)           # truncate to bf16
    xr = (bits.astype(np.uint32) << 16).view(np.float32)          # the same values as fp32
    v = f32((1, 1, 20, 4))
    vbits = (v.view(np.uint32) >> 16).astype(np.uint16)
    vr = (vbits.astype(np.uint32) << 16).view(np.float32)
    a = oracle.taylor(bits, bits, vbits)
    b = oracle.taylor(xr, xr, vr)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["s"], b["s"])


# --------------------------------------------------------------------------
# Gated delta rule


def dense_eq1(q, k, v, alpha, beta, S0):
    """S_t = S_{t-1} A_t + beta_t v_t k_t^T with A_t = alpha_t (I - beta_t k_t k_t^T)
    formed as a dense d_k x d_k matrix; o_t = S_t q_t (NoteBank Sec. 2 Eq. (1))."""
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, N, dv))
    S_out = np.zeros((B, H, dv, dk))
    I = np.eye(dk)
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for t in range(N):
                kt = k[b, h, t].astype(np.float64)
                A = float(alpha[b, h, t]) * (I - float(beta[b, h, t]) * np.outer(kt, kt))
                S = S @ A + float(beta[b, h, t]) * np.outer(v[b, h, t].astype(np.float64), kt)
                o[b, h, t] = S @ q[b, h, t].astype(np.float64)
            S_out[b, h] = S
    return o, S_out


def gdn_rand(B, H, N, dk, dv):
    q = f32((B, H, N, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = f32((B, H, N, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = f32((B, H, N, dv))
    beta = (1 / (1 + np.exp(-rng.standard_normal((B, H, N))))).astype(np.float32)
    alpha = np.exp(-rng.uniform(0.001, 0.1, (B, H, N))).astype(np.float32)
    return q.astype(np.float32), k.astype(np.float32), v, alpha, beta


@pytest.mark.parametrize("dk,dv,N", [(6, 5, 23), (8, 8, 31)])
def test_gdn_equals_dense_matrix_form(dk, dv, N):
    q, k, v, alpha, beta = gdn_rand(2, 2, N, dk, dv)
    S0 = rng.standard_normal((2, 2, dv, dk))
    out = oracle.gdn(q, k, v, alpha, beta, S_in=S0)
    o_ref, S_ref = dense_eq1(q, k, v, alpha, beta, S0)
    assert rel_err(out["o"], o_ref) < 1e-12
    assert rel_err(out["S"], S_ref) < 1e-12


def test_gdn_reduces_to_additive_for_orthogonal_keys():
    """alpha = 1, beta = 1 and each key orthogonal to all earlier keys:
    A_t acts as I on the state, so S_t = sum_{j<=t} v_j k_j^T (additive
    linear attention, NoteBank Sec. 2)."""
    dk, dv, N = 16, 7, 12
    # rows of a 16x16 Sylvester Hadamard matrix / 4: entries +-1/4, exactly
    # orthonormal in binary floating point; random order and signs
    had = np.array([[1.0]])
    while had.shape[0] < dk:
        had = np.block([[had, had], [had, -had]])
    rows = rng.permutation(dk)[:N]
    signs = rng.choice([-1.0, 1.0], N)
    k = (had[rows] * signs[:, None] / 4.0).astype(np.float32)[None, None]
    q = f32((1, 1, N, dk))
    v = f32((1, 1, N, dv))
    ones = np.ones((1, 1, N), np.float32)
    out = oracle.gdn(q, k, v, ones, ones)
    kd, vd, qd = k[0, 0].astype(np.float64), v[0, 0].astype(np.float64), q[0, 0].astype(np.float64)
    S = np.zeros((dv, dk))
    for t in range(N):
        S = S + np.outer(vd[t], kd[t])
        assert np.allclose(out["o"][0, 0, t], S @ qd[t], rtol=1e-10, atol=1e-10)
    assert np.allclose(out["S"][0, 0], S, rtol=1e-10, atol=1e-10)


def test_gdn_beta_zero_pure_decay():
    dk, dv, N = 8, 4, 20
    q, k, v, alpha, _ = gdn_rand(1, 2, N, dk, dv)
    S0 = rng.standard_normal((1, 2, dv, dk))
    out = oracle.gdn(q, k, v, alpha, np.zeros_like(alpha), S_in=S0)
    g = np.cumprod(alpha.astype(np.float64), axis=-1)
    for h in range(2):
        for t in range(N):
            assert np.allclose(out["o"][0, h, t], g[0, h, t] * (S0[0, h] @ q[0, h, t]), rtol=1e-12, atol=1e-12)
        assert np.allclose(out["S"][0, h], g[0, h, -1] * S0[0, h], rtol=1e-12, atol=1e-14)
    # alpha = 1, beta = 0: the state never changes
    one = np.ones_like(alpha)
    out = oracle.gdn(q, k, v, one, np.zeros_like(alpha), S_in=S0)
    assert np.array_equal(out["S"], S0)


def test_gdn_overwrite_property_unit_keys():
    """||k_t|| = 1 exactly => S_t k_t = alpha_t (1 - beta_t) S_{t-1} k_t + beta_t v_t;
    with beta = 1 the key reads back exactly its value (delta-rule overwrite)."""
    dk, dv, N = 16, 5, 25
    k = np.zeros((1, 1, N, dk), np.float32)
    for t in range(N):  # four entries of +-1/2: unit norm in exact arithmetic
        idx = rng.choice(dk, 4, replace=False)
        k[0, 0, t, idx] = rng.choice([-0.5, 0.5], 4)
    q = f32((1, 1, N, dk))
    v = f32((1, 1, N, dv))
    alpha = np.exp(-rng.uniform(0.001, 0.1, (1, 1, N))).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((1, 1, N))))).astype(np.float32)
    S_prev = np.zeros((dv, dk))
    for t in range(N):
        o = oracle.gdn(q[:, :, : t + 1], k[:, :, : t + 1], v[:, :, : t + 1], alpha[:, :, : t + 1], beta[:, :, : t + 1])
        S_t = o["S"][0, 0]
        kt = k[0, 0, t].astype(np.float64)
        lhs = S_t @ kt
        rhs = float(alpha[0, 0, t]) * (1 - float(beta[0, 0, t])) * (S_prev @ kt) + float(beta[0, 0, t]) * v[0, 0, t].astype(np.float64)
        assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
        S_prev = S_t
    ones = np.ones((1, 1, N), np.float32)
    o = oracle.gdn(q, k, v, ones, ones)
    # last key reads back the last value exactly
    assert np.allclose(o["S"][0, 0] @ k[0, 0, -1].astype(np.float64), v[0, 0, -1], rtol=1e-13, atol=1e-13)


def test_gdn_q_scale_split_and_samples():
    dk, dv, N = 8, 6, 40
    q, k, v, alpha, beta = gdn_rand(1, 3, N, dk, dv)
    full = oracle.gdn(q, k, v, alpha, beta)
    half = oracle.gdn(q, k, v, alpha, beta, q_scale=0.5)
    assert rel_err(half["o"], 0.5 * full["o"]) < 1e-14
    a = oracle.gdn(q[:, :, :13], k[:, :, :13], v[:, :, :13], alpha[:, :, :13], beta[:, :, :13])
    b = oracle.gdn(q[:, :, 13:], k[:, :, 13:], v[:, :, 13:], alpha[:, :, 13:], beta[:, :, 13:], S_in=a["S"])
    assert rel_err(np.concatenate([a["o"], b["o"]], axis=2), full["o"]) < 1e-13
    assert rel_err(b["S"], full["S"]) < 1e-13
    t = [3, 13, 39]
    smp = oracle.gdn(q, k, v, alpha, beta, t_samples=t)
    assert np.array_equal(smp["o"], full["o"][:, :, t])


# --------------------------------------------------------------------------
# Scalar gate, A_t = alpha_t I (the gated family of NoteBank Sec. 2)


def gated_closed_form(q, k, v, alpha, beta, S0, q_scale=1.0):
    """Unrolled scalar-gate recurrence, written as explicit sums:
    S_t = (prod_{m<=t} alpha_m) S_0 + sum_{j<=t} (prod_{j<m<=t} alpha_m) beta_j v_j k_j^T,
    o_t = S_t (q_scale q_t)."""
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, N, dv))
    S_out = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            a = alpha[b, h].astype(np.float64)
            for t in range(N):
                S = np.prod(a[: t + 1]) * S0[b, h]
                for j in range(t + 1):
                    S = S + np.prod(a[j + 1: t + 1]) * float(beta[b, h, j]) * np.outer(
                        v[b, h, j].astype(np.float64), k[b, h, j].astype(np.float64))
                o[b, h, t] = S @ (q_scale * q[b, h, t].astype(np.float64))
                if t == N - 1:
                    S_out[b, h] = S
    return o, S_out


@pytest.mark.parametrize("dk,dv,N", [(6, 5, 17), (8, 8, 25)])
def test_gated_equals_closed_form(dk, dv, N):
    q, k, v, alpha, beta = gdn_rand(2, 2, N, dk, dv)
    S0 = rng.standard_normal((2, 2, dv, dk))
    out = oracle.gated(q, k, v, alpha, beta, S_in=S0, q_scale=0.75)
    o_ref, S_ref = gated_closed_form(q, k, v, alpha, beta, S0, q_scale=0.75)
    assert rel_err(out["o"], o_ref) < 1e-12
    assert rel_err(out["S"], S_ref) < 1e-12


def test_gated_equals_delta_rule_for_orthogonal_keys():
    """Each key orthogonal to every earlier key and S_0 = 0: S_{t-1} k_t = 0,
    so the delta rule's erase term vanishes and the gated delta rule (pinned
    above against the dense Eq. (1)) equals the scalar gate, for any alpha, beta."""
    dk, dv, N = 16, 6, 14
    had = np.array([[1.0]])
    while had.shape[0] < dk:
        had = np.block([[had, had], [had, -had]])
    rows = rng.permutation(dk)[:N]
    k = (had[rows] * rng.choice([-1.0, 1.0], N)[:, None] / 4.0).astype(np.float32)[None, None]
    q = f32((1, 1, N, dk))
    v = f32((1, 1, N, dv))
    alpha = np.exp(-rng.uniform(0.001, 0.1, (1, 1, N))).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((1, 1, N))))).astype(np.float32)
    a = oracle.gated(q, k, v, alpha, beta)
    b = oracle.gdn(q, k, v, alpha, beta)
    assert rel_err(a["o"], b["o"]) < 1e-12
    assert rel_err(a["S"], b["S"]) < 1e-12


def test_gated_additive_special_case():
    """alpha = beta = 1 is standard additive linear attention (NoteBank Sec. 2):
    o_t = sum_{j<=t} (k_j . q_t) v_j."""
    dk, dv, N = 5, 4, 19
    q, k, v, _, _ = gdn_rand(1, 1, N, dk, dv)
    ones = np.ones((1, 1, N), np.float32)
    out = oracle.gated(q, k, v, ones, ones)
    kd, vd, qd = k[0, 0].astype(np.float64), v[0, 0].astype(np.float64), q[0, 0].astype(np.float64)
    for t in range(N):
        ref = sum((kd[j] @ qd[t]) * vd[j] for j in range(t + 1))
        assert np.allclose(out["o"][0, 0, t], ref, rtol=1e-12, atol=1e-12)


def test_gated_split_resume():
    dk, dv, N = 8, 6, 33
    q, k, v, alpha, beta = gdn_rand(1, 2, N, dk, dv)
    full = oracle.gated(q, k, v, alpha, beta)
    a = oracle.gated(q[:, :, :10], k[:, :, :10], v[:, :, :10], alpha[:, :, :10], beta[:, :, :10])
    b = oracle.gated(q[:, :, 10:], k[:, :, 10:], v[:, :, 10:], alpha[:, :, 10:], beta[:, :, 10:], S_in=a["S"])
    assert rel_err(np.concatenate([a["o"], b["o"]], axis=2), full["o"]) < 1e-13
    assert rel_err(b["S"], full["S"]) < 1e-13


# --------------------------------------------------------------------------
# State operations (NoteBank App. D.1 rescale/reset; App. B Alg. 1 copy)


def test_state_rescale_definition_and_reset():
    S = rng.standard_normal((3, 2, 5, 4)).astype(np.float32)
    assert np.array_equal(oracle.state_rescale(S, 1.0), S)
    bad = S.copy()
    bad[0, 1, 2, 3] = np.nan
    bad[2, 0, 0, 0] = np.inf
    assert np.array_equal(oracle.state_rescale(bad, 0.0), np.zeros_like(S))  # a reset, whatever was stored
    lam = np.array([[0.5, 0.25], [1.0, 0.0], [0.75, 0.125]], np.float32)
    out = oracle.state_rescale(S, lam)
    for b in range(3):
        for h in range(2):
            assert np.array_equal(out[b, h], S[b, h] * lam[b, h])
    # powers of two compose exactly
    assert np.array_equal(oracle.state_rescale(oracle.state_rescale(S, 0.5), 0.25), oracle.state_rescale(S, 0.125))


def test_state_rescale_feeds_the_recurrence_linearly():
    """The recurrence is affine in its entry state, so replaying from
    lambda S_0 gives o(0) + lambda (o(S_0) - o(0)) for both the gated delta
    rule and the scalar gate (each pinned above to its definition)."""
    dk, dv, N = 8, 6, 21
    q, k, v, alpha, beta = gdn_rand(1, 2, N, dk, dv)
    S0 = rng.standard_normal((1, 2, dv, dk)).astype(np.float32)
    lam = 0.25  # a power of two: lambda S_0 is exact in float32
    for fn in (oracle.gdn, oracle.gated):
        base = fn(q, k, v, alpha, beta)
        full = fn(q, k, v, alpha, beta, S_in=S0)
        resc = fn(q, k, v, alpha, beta, S_in=oracle.state_rescale(S0, lam))
        assert rel_err(resc["o"], base["o"] + lam * (full["o"] - base["o"])) < 1e-12
        assert rel_err(resc["S"], base["S"] + lam * (full["S"] - base["S"])) < 1e-12


def test_state_gather_copies_and_branches():
    src = rng.standard_normal((4, 3, 7)).astype(np.float32)
    idx = [2, 0, 2, 3, 2]
    out = oracle.state_gather(src, idx, state_dims=1)
    flat = src.reshape(-1, 7)
    for i, j in enumerate(idx):
        assert np.array_equal(out[i], flat[j])
    assert oracle.state_gather(src, [], state_dims=1).shape == (0, 7)


# --------------------------------------------------------------------------
# Sliding-window softmax attention (BASED notes Sec. 2.4)


def masked_softmax_attention(q, k, v, scale, mask):
    """Row-wise softmax of the masked score matrix, then times V (the matrix
    form of attention; mask[i, j] True keeps key j for query i)."""
    sc = scale * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
    sc = np.where(mask, sc, -np.inf)
    sc = sc - sc.max(axis=-1, keepdims=True)
    p = np.exp(sc)
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("bhij,bhjd->bhid", p, v.astype(np.float64))


@pytest.mark.parametrize("window", [1, 2, 5, 16])
def test_swa_equals_banded_matrix_softmax(window):
    N, d = 23, 6
    q, k, v = f32((2, 2, N, d)), f32((2, 2, N, d)), f32((2, 2, N, 5))
    i, j = np.arange(N)[:, None], np.arange(N)[None, :]
    band = (j <= i) & (j > i - window)
    ref = masked_softmax_attention(q, k, v, 0.4, band)
    assert rel_err(oracle.swa(q, k, v, window, 0.4), ref) < 1e-12


def test_swa_special_cases():
    N, d = 17, 4
    q, k, v = f32((1, 1, N, d)), f32((1, 1, N, d)), f32((1, 1, N, 3))
    # a window at least N long is plain causal softmax attention
    i, j = np.arange(N)[:, None], np.arange(N)[None, :]
    assert rel_err(oracle.swa(q, k, v, N + 3, 0.5), masked_softmax_attention(q, k, v, 0.5, j <= i)) < 1e-12
    # window 1: each token reads its own value
    assert np.allclose(oracle.swa(q, k, v, 1, 0.5), v.astype(np.float64), rtol=0, atol=0)
    # equal keys: the mean of the window's values
    ke = np.repeat(k[:, :, :1], N, axis=2)
    o = oracle.swa(q, ke, v, 4, 0.5)
    for t in range(N):
        assert np.allclose(o[0, 0, t], v[0, 0, max(0, t - 3): t + 1].astype(np.float64).mean(axis=0), atol=1e-14)


def test_gdn_state_size_arithmetic():
    g = json.load(open(os.path.join(GOLDEN, "state_size.json")))
    q, k, v, alpha, beta = gdn_rand(1, 1, 2, 4, 3)
    S = oracle.gdn(q, k, v, alpha, beta)["S"]
    assert S.shape[-2:] == (3, 4)  # d_v x d_k
    assert g["J"] * g["d_v"] * g["d_k"] * g["bytes_per_element"] == g["MiB"] * 2 ** 20


def test_rejects_bad_samples():
    q, k, v, alpha, beta = gdn_rand(1, 1, 5, 4, 3)
    with pytest.raises(ValueError):
        oracle.gdn(q, k, v, alpha, beta, t_samples=[3, 1])
    with pytest.raises(ValueError):
        oracle.taylor(q, k, v[..., :3], t_samples=[7])


def test_empty_sequence_passes_state_through():
    q = np.zeros((1, 2, 0, 16), np.float32)
    v = np.zeros((1, 2, 0, 8), np.float32)
    s0 = rng.standard_normal((1, 2, 273, 8))
    z0 = rng.standard_normal((1, 2, 273))
    out = oracle.taylor(q, q, v, s_in=s0, z_in=z0)
    assert np.array_equal(out["s"], s0) and np.array_equal(out["z"], z0)
    S0 = rng.standard_normal((1, 2, 8, 16))
    out = oracle.gdn(q, q, v, np.zeros((1, 2, 0), np.float32), np.zeros((1, 2, 0), np.float32), S_in=S0)
    assert np.array_equal(out["S"], S0)


# --------------------------------------------------------------------------
# NoteBank write side and routing (NoteBank Sec. 2 Eqs. (3)-(5), App. B
# Eqs. (8)-(9))


def test_notebank_scores_hand_example():
    # keys (1,0), (0,1), (1,1): unit keys e1, e2, (e1+e2)/sqrt2; their mean points along (1,1),
    # so mu = (1,1)/sqrt2 and d = 1 - 1/sqrt2, 1 - 1/sqrt2, 0
    k = np.array([[[[1, 0], [0, 1], [1, 1]]]], dtype=np.float32)
    r = oracle.notebank_scores(k, chunk=3, window=2)
    a = 1 - 1 / math.sqrt(2)
    assert np.allclose(r["d_ch"][0, 0], [a, a, 0.0], rtol=0, atol=1e-15)
    assert np.allclose(r["w"], [2 * a, a], rtol=0, atol=1e-15)


def test_notebank_scores_identities():
    L, H, N, d, C = 2, 3, 70, 8, 32
    k = f32((L, H, N, d))
    r = oracle.notebank_scores(k, chunk=C, window=5)
    # per chunk and channel: mean_t (1 - d_t) = <mean_t unit(k_t), mu> = |mean_t unit(k_t)|
    kh = k / np.linalg.norm(k.astype(np.float64), axis=-1, keepdims=True)
    for c0 in range(0, N, C):
        c1 = min(c0 + C, N)
        m = np.linalg.norm(kh[:, :, c0:c1].mean(axis=2), axis=-1)
        assert np.allclose((1 - r["d_ch"][:, :, c0:c1]).mean(axis=2), m, rtol=1e-12, atol=1e-12)
    assert np.all(r["d_ch"] >= -1e-12) and np.all(r["d_ch"] <= 2 + 1e-12)
    assert np.allclose(r["d"], r["d_ch"].mean(axis=(0, 1)), rtol=0, atol=0)
    cs = np.concatenate([[0.0], np.cumsum(r["d"])])
    assert np.allclose(r["w"], cs[5:] - cs[:-5], rtol=1e-12, atol=1e-12)
    # positive rescaling of any key changes nothing; parallel keys are not distinctive
    k2 = k * (0.5 + rng.random((L, H, N, 1))).astype(np.float32)
    assert np.allclose(oracle.notebank_scores(k2, chunk=C, window=5)["d_ch"], r["d_ch"], atol=1e-6)
    par = np.broadcast_to(k[:, :, :1], k.shape) * (1 + rng.random((L, H, N, 1))).astype(np.float32)
    assert np.allclose(oracle.notebank_scores(par, chunk=C)["d_ch"], 0.0, atol=1e-7)


def test_notebank_address_argmax_and_gather():
    L, H, N, d = 1, 2, 40, 32
    d_ch = rng.random((L, H, N))
    d_ch[0, 0, 12] = d_ch[0, 0, 17] = 5.0      # tie inside the span: the earlier token wins
    d_ch[0, 1, 30] = 9.0                       # outside the span: ignored
    q = f32((L, H, N, d))
    coords = np.stack([rng.permutation(d)[:16] for _ in range(L * H)]).reshape(L, H, 16)
    t_star, rho = oracle.notebank_address(d_ch, q, coords, [(10, 15)])
    assert t_star[0, 0, 0] == 12
    assert t_star[0, 0, 1] == 10 + int(np.argmax(d_ch[0, 1, 10:25]))
    for h in range(H):
        vals = q[0, h, t_star[0, 0, h], coords[0, h]]
        assert np.all(np.abs(rho[0, 0, h] - vals) <= np.abs(vals) * 2.0 ** -8)   # one bf16 rounding
        assert np.array_equal(rho[0, 0, h], oracle._round_bf16(vals))


def test_notebank_route_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "notebank_vote_example.json")))
    names = g["notes"]
    J = len(g["channel_winners"])
    # note i's address in channel j is e_j if note i should win channel j, else e_(j+1); the question
    # feature of channel j is e_j: the winner has cosine 1, the other note 0
    rho = np.zeros((len(names), J, 16), np.float32)
    for j, w in enumerate(g["channel_winners"]):
        for i, nm in enumerate(names):
            rho[i, j, j if nm == w else j + 1] = 1.0
    u = np.zeros((J, 1, 16), np.float32)
    for j in range(J):
        u[j, 0, j] = 1.0
    # A was written after B in the text: the replay order must follow the text, not the votes
    r = oracle.notebank_route(rho, u, R=g["R"], positions=[500, 100])
    assert [names[i] for i in r["winner"]] == g["channel_winners"]
    assert {names[i]: int(r["votes"][i]) for i in range(len(names))} == g["votes"]
    assert sorted(names[i] for i in r["top"]) == sorted(g["retrieved"])
    assert [names[i] for i in r["top"]] == ["B", "A"]
    assert [names[i] for i in oracle.notebank_route(rho, u, R=1, positions=[500, 100])["top"]] == ["A"]


def test_notebank_route_ties_scaling_and_max_over_question():
    n, J, nq = 6, 4, 5
    rho = f32((n, J, 16))
    u = f32((J, nq, 16))
    r = oracle.notebank_route(rho, u, R=3)
    # cosine: positive rescaling of addresses or question features changes nothing
    r2 = oracle.notebank_route(rho * 3.0, u * 0.25, R=3)
    assert np.allclose(r2["s"], r["s"], atol=1e-6) and np.array_equal(r2["winner"], r["winner"])
    # max over question tokens: each s equals the best single-token cosine
    for i in range(n):
        for j in range(J):
            best = max(float(np.dot(rho[i, j], u[j, t]) / np.linalg.norm(rho[i, j]) / np.linalg.norm(u[j, t]))
                       for t in range(nq))
            assert r["s"][i, j] == pytest.approx(best, abs=1e-6)
    assert r["votes"].sum() == J
    # a duplicate of the winning note inserted later never takes its vote (ties go to the earlier note)
    w0 = int(r["winner"][0])
    dup = np.concatenate([rho, rho[w0:w0 + 1]], axis=0)
    assert oracle.notebank_route(dup, u, R=3)["winner"][0] == w0
    # equal votes: the earlier-inserted note is retrieved first
    rho2 = np.zeros((3, 2, 16), np.float32)
    u2 = np.zeros((2, 1, 16), np.float32)
    rho2[0, 0, 0] = rho2[2, 1, 1] = 1.0
    rho2[1, :, 5] = rho2[0, 1, 5] = rho2[2, 0, 5] = 1.0
    u2[0, 0, 0] = u2[1, 0, 1] = 1.0
    r3 = oracle.notebank_route(rho2, u2, R=1)
    assert list(r3["votes"]) == [1, 0, 1] and list(r3["top"]) == [0]


def test_round_bf16_ties_to_even():
    """Exact halfway cases of float32 -> bf16 go to the even mantissa (the rounding the GPU's
    conversions use); values just off the halfway point go to the nearer neighbour."""
    ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    cases = [
        (1.0 + ulp / 2, 1.0),                  # halfway between 1 and 1 + ulp: even is 1
        (1.0 + 3 * ulp / 2, 1.0 + 2 * ulp),    # halfway between 1 + ulp and 1 + 2 ulp: even is 1 + 2 ulp
        (-(1.0 + ulp / 2), -1.0),
        (-(1.0 + 3 * ulp / 2), -(1.0 + 2 * ulp)),
        (1.0 + ulp / 2 + 2.0 ** -23, 1.0 + ulp),  # one float32 ulp above halfway: up
        (1.0 + ulp / 2 - 2.0 ** -23, 1.0),        # one below: down
        (3.0 + 2.0 ** -7, 3.0),                # spacing 2^-6 in [2, 4): halfway to 3 + 2^-6, 3 is even
        (0.0, 0.0),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    assert np.array_equal(x.astype(np.float64), np.array([c[0] for c in cases]))  # exact in float32
    assert np.array_equal(oracle._round_bf16(x), np.array([c[1] for c in cases]))
