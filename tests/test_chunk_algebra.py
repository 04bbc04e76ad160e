"""CPU checks of the chunked scan's algebra and of its tensor-core operand split.

The tensor-core scans regroup the delta-rule recurrence in chunks of C positions (the
WY/UT form; fm_kernel_ssm.m names a chunked prefill path built on per-chunk cumulative
sums of g and keeps the sequential scan as its reference, without the algebra). Here
that regrouping is written out in numpy float64, with plain dense linear algebra, and
compared with the oracle's sequential recurrence: per chunk with gam_t = g_0 + .. + g_t,

    A[t][s] = beta_t exp(gam_t - gam_s) (k_t . k_s)             (s < t)
    (I + A) W = diag(beta exp(gam)) K,   (I + A) Ut = diag(beta) V
    U = Ut - W S,   y_t = scale (exp(gam_t) q_t . S + sum_{s<=t} exp(gam_t - gam_s) (q_t . k_s) u_s)
    S' = exp(gam_last) S + sum_s exp(gam_last - gam_s) k_s u_s^T

with S as the [dk][dv] matrix. The regrouping is exact, so the two agree to float64
rounding. The operand splits of the tensor-core products are checked against their
error bounds: x = hi + lo with hi = bf16(x), lo = bf16(x - hi) (nearest, ties to even)
and hi*hi + hi*lo + lo*hi, the 3xBF16 products the chunked scans issue, and the tf32
form of the same split. Nothing here runs on a GPU.
"""
import math

import numpy as np
import pytest

import oracle

C = 32


def chunked_scan(state, q, k, v, g, beta, scale, chunk=C):
    """The WY/UT regrouping, fp64. state [N][H][S(j)][S(i)] (the library's transposed
    layout) is updated in place; returns y [N][T][H][S]."""
    N, T, Hk, S = q.shape
    H = v.shape[2]
    y = np.zeros(v.shape)
    for n in range(N):
        for h in range(H):
            kh = h % Hk
            Sm = state[n, h].T.copy()  # [dk][dv]
            for t0 in range(0, T, chunk):
                t1 = min(T, t0 + chunk)
                K, Q, V = k[n, t0:t1, kh], q[n, t0:t1, kh], v[n, t0:t1, h]
                gam = np.cumsum(g[n, t0:t1, h])
                bet = beta[n, t0:t1, h]
                L = t1 - t0
                dec = np.exp(gam[:, None] - gam[None, :])  # exp(gam_t - gam_s)
                A = np.tril(bet[:, None] * dec * (K @ K.T), -1)
                IA = np.eye(L) + A
                W = np.linalg.solve(IA, (bet * np.exp(gam))[:, None] * K)
                Ut = np.linalg.solve(IA, bet[:, None] * V)
                U = Ut - W @ Sm
                M = np.tril(dec * (Q @ K.T))
                y[n, t0:t1, h] = scale * (np.exp(gam)[:, None] * (Q @ Sm) + M @ U)
                Sm = np.exp(gam[-1]) * Sm + (np.exp(gam[-1] - gam)[:, None] * K).T @ U
            state[n, h] = Sm.T
    return y


def inputs(r, N, T, Hk, H, S, g_lo=-0.5):
    q = r.normal(size=(N, T, Hk, S))
    k = r.normal(size=(N, T, Hk, S))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return dict(q=q, k=k, v=r.normal(size=(N, T, H, S)),
                g=r.uniform(g_lo, -0.001, size=(N, T, H)),
                beta=1 / (1 + np.exp(-r.normal(size=(N, T, H)))))


@pytest.mark.parametrize("N,T,Hk,H,S", [(1, 1, 1, 1, 8), (2, 31, 1, 2, 8), (1, 32, 2, 2, 16),
                                        (2, 33, 2, 4, 16), (1, 100, 1, 3, 32)])
def test_chunked_regrouping_equals_sequential_oracle(N, T, Hk, H, S):
    r = np.random.default_rng(T * 7 + H)
    x = inputs(r, N, T, Hk, H, S)
    st0 = r.normal(0, 0.1, size=(N, H, S, S))
    scale = 1 / math.sqrt(S)
    st_seq = st0.copy()
    y_seq, _ = oracle.recurrence(st_seq, scale=scale, **x)
    st_chk = st0.copy()
    y_chk = chunked_scan(st_chk, scale=scale, **x)
    np.testing.assert_allclose(y_chk, y_seq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(st_chk, st_seq, rtol=0, atol=1e-11)


def test_chunk_length_does_not_matter():
    """Chunks of 8, 32 or the whole sequence give the same result (the regrouping is
    exact for any chunk length, including the ragged last chunk)."""
    r = np.random.default_rng(3)
    x = inputs(r, 1, 45, 1, 2, 8, g_lo=-2.0)
    st0 = r.normal(0, 0.1, size=(1, 2, 8, 8))
    outs = []
    for c in (8, 32, 45):
        st = st0.copy()
        outs.append((chunked_scan(st, scale=0.3, chunk=c, **x), st))
    for y, st in outs[1:]:
        np.testing.assert_allclose(y, outs[0][0], rtol=0, atol=1e-11)
        np.testing.assert_allclose(st, outs[0][1], rtol=0, atol=1e-11)


def test_dropping_a_term_is_caught():
    """The comparison is sharp enough to see a plausible slip: the decay of the carried
    state left out of the readout changes y well beyond the tolerance above."""
    r = np.random.default_rng(11)
    x = inputs(r, 1, 40, 1, 1, 8)
    st0 = r.normal(0, 0.1, size=(1, 1, 8, 8))
    st_seq = st0.copy()
    y_seq, _ = oracle.recurrence(st_seq, scale=0.35, **x)
    x_bad = dict(x)
    x_bad["g"] = np.zeros_like(x["g"])  # as if exp(gam) were dropped everywhere
    y_bad = chunked_scan(st0.copy(), scale=0.35, **x_bad)
    assert np.abs(y_bad - y_seq).max() > 1e-3


# ---------------------------------------------------------------- the operand split

def split_hl(x):
    """hi: x with the low 13 mantissa bits cleared; lo = x - hi (exact in fp32)."""
    x = np.asarray(x, np.float32)
    hi = (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    return hi, (x - hi).astype(np.float32)


def tf32_trunc(x):
    return (np.asarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)


def test_split_is_exact_and_lo_small():
    r = np.random.default_rng(5)
    x = (r.normal(size=100000) * np.exp(r.uniform(-20, 20, size=100000))).astype(np.float32)
    hi, lo = split_hl(x)
    assert np.all(tf32_trunc(hi) == hi)  # hi is a tf32 value
    np.testing.assert_array_equal(hi.astype(np.float64) + lo.astype(np.float64), x.astype(np.float64))
    nz = x != 0
    assert np.all(np.abs(lo[nz]) < np.abs(x[nz]) * 2.0 ** -10)


def test_three_pass_product_error_bound():
    """hi*hi + hi*lo' + lo'*hi with lo' = tf32(lo) (what the tensor core reads) is within
    a few units of 2^-20 of the exact product; one tf32 pass is ~2^-10 off."""
    r = np.random.default_rng(6)
    a = r.normal(size=20000).astype(np.float32)
    b = r.normal(size=20000).astype(np.float32)
    ah, al = split_hl(a)
    bh, bl = split_hl(b)
    al, bl = tf32_trunc(al).astype(np.float64), tf32_trunc(bl).astype(np.float64)
    ah, bh = ah.astype(np.float64), bh.astype(np.float64)
    exact = a.astype(np.float64) * b.astype(np.float64)
    three = ah * bh + ah * bl + al * bh
    one = tf32_trunc(a).astype(np.float64) * tf32_trunc(b).astype(np.float64)
    rel3 = np.abs(three - exact) / np.abs(exact)
    rel1 = np.abs(one - exact) / np.abs(exact)
    assert rel3.max() < 4 * 2.0 ** -20
    assert rel1.max() > 2.0 ** -12


# ---------------------------------------------------------------- why three passes

def _tf32(x):
    return tf32_trunc(x).astype(np.float64)


def _products(a, b, passes):
    """a @ b as the tensor core forms it from fp32 operands read at tf32 precision: one
    pass (hi * hi) or the three-pass split (hi * hi + hi * lo + lo * hi)."""
    ah, bh = _tf32(a), _tf32(b)
    if passes == 1:
        return ah @ bh
    al, bl = _tf32(a - ah), _tf32(b - bh)
    return ah @ bh + ah @ bl + al @ bh


def chunked_scan_tf32(state, q, k, v, g, beta, scale, passes, chunk=C, products=None):
    """The regrouping above with the four state-dependent products (W S, (Gam q) S, M U
    and the state update) taken as the tensor cores take them (`products(a, b, passes)`,
    tf32 by default); the chunk-local work (Gram products, solves) stays exact, as it is
    not on the tensor cores."""
    prod = products or _products
    N, T, Hk, S = q.shape
    H = v.shape[2]
    y = np.zeros(v.shape)
    for n in range(N):
        for h in range(H):
            kh = h % Hk
            Sm = state[n, h].T.copy()
            for t0 in range(0, T, chunk):
                t1 = min(T, t0 + chunk)
                K, Q, V = k[n, t0:t1, kh], q[n, t0:t1, kh], v[n, t0:t1, h]
                gam = np.cumsum(g[n, t0:t1, h])
                bet = beta[n, t0:t1, h]
                dec = np.exp(gam[:, None] - gam[None, :])
                IA = np.eye(t1 - t0) + np.tril(bet[:, None] * dec * (K @ K.T), -1)
                W = np.linalg.solve(IA, (bet * np.exp(gam))[:, None] * K)
                Ut = np.linalg.solve(IA, bet[:, None] * V)
                U = Ut - prod(W, Sm, passes)
                M = np.tril(dec * (Q @ K.T))
                y[n, t0:t1, h] = scale * (prod(np.exp(gam)[:, None] * Q, Sm, passes) +
                                          prod(M, U, passes))
                Sm = np.exp(gam[-1]) * Sm + prod((np.exp(gam[-1] - gam)[:, None] * K).T,
                                                 U, passes)
            state[n, h] = Sm.T
    return y


def test_one_tf32_pass_misses_the_long_scan_bound_three_passes_meet_it():
    """The precision choice of the tensor-core scans: over 1024 positions at S = 128 (the
    prefill scan's distributions), tf32 operands in one pass put y and the state well
    past the long-scan bound (max |err| <= 2e-3 RMS of the exact scan); the hi / lo split
    in three passes stays two orders of magnitude inside it."""
    r = np.random.default_rng(21)
    x = inputs(r, 1, 1024, 1, 2, 128)
    st0 = r.normal(0, 0.1, size=(1, 2, 128, 128))
    scale = 1 / math.sqrt(128)
    st_ref = st0.copy()
    y_ref, _ = oracle.recurrence(st_ref, scale=scale, **x)

    def rel(a, b):
        return np.abs(a - b).max() / math.sqrt(np.mean(b * b))
    st1 = st0.copy()
    y1 = chunked_scan_tf32(st1, scale=scale, passes=1, **x)
    st3 = st0.copy()
    y3 = chunked_scan_tf32(st3, scale=scale, passes=3, **x)
    assert rel(y1, y_ref) > 2e-3 and rel(st1, st_ref) > 2e-3
    assert rel(y3, y_ref) < 2e-5 and rel(st3, st_ref) < 2e-5


# ---------------------------------------------------------------- the bf16 split

def bf16_rn(x):
    """Nearest bf16 value (ties to even) of float32 x, as float64."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def split_bf16(x):
    """hi = bf16(x), lo = bf16(x - hi), with x - hi formed in float32 (it is exact)."""
    x = np.asarray(x, np.float32)
    hi = bf16_rn(x)
    return hi, bf16_rn((x - hi.astype(np.float32)).astype(np.float32))


def test_bf16_split_residual_is_exact_and_small():
    r = np.random.default_rng(8)
    x = (r.normal(size=100000) * np.exp(r.uniform(-20, 20, size=100000))).astype(np.float32)
    hi = bf16_rn(x)
    res = x.astype(np.float64) - hi
    assert np.all(res.astype(np.float32).astype(np.float64) == res)  # exact in float32
    nz = x != 0
    assert np.all(np.abs(res[nz]) <= np.abs(x[nz]) * 2.0 ** -8)
    hi, lo = split_bf16(x)
    assert np.all(np.abs(x[nz] - hi[nz] - lo[nz]) <= np.abs(x[nz]) * 2.0 ** -16)


def test_three_pass_bf16_product_error_bound():
    """hi*hi + hi*lo + lo*hi is within 3 * 2^-16 (relative) of the exact product; one bf16
    pass is ~2^-8 off."""
    r = np.random.default_rng(9)
    a = r.normal(size=50000).astype(np.float32)
    b = r.normal(size=50000).astype(np.float32)
    ah, al = split_bf16(a)
    bh, bl = split_bf16(b)
    exact = a.astype(np.float64) * b.astype(np.float64)
    rel3 = np.abs(ah * bh + ah * bl + al * bh - exact) / np.abs(exact)
    rel1 = np.abs(ah * bh - exact) / np.abs(exact)
    assert rel3.max() < 3 * 2.0 ** -16
    assert rel1.max() > 2.0 ** -9


def _products_bf16(a, b, passes):
    """a @ b from bf16 operand parts: one pass (hi * hi) or three (hi*hi + hi*lo + lo*hi)."""
    ah, al = split_bf16(a)
    bh, bl = split_bf16(b)
    if passes == 1:
        return ah @ bh
    return ah @ bh + ah @ bl + al @ bh


def test_one_bf16_pass_misses_the_long_scan_bound_three_passes_meet_it():
    """The precision of the chunked scans' 3xBF16 products: over 1024 positions at S = 128,
    one bf16 pass puts y and the state far past the long-scan bound (max |err| <= 2e-3 RMS
    of the exact scan); the three-pass split stays an order of magnitude inside it
    (1.2e-4 and 1.4e-4 of RMS here)."""
    r = np.random.default_rng(21)
    x = inputs(r, 1, 1024, 1, 2, 128)
    st0 = r.normal(0, 0.1, size=(1, 2, 128, 128))
    scale = 1 / math.sqrt(128)
    st_ref = st0.copy()
    y_ref, _ = oracle.recurrence(st_ref, scale=scale, **x)

    def rel(a, b):
        return np.abs(a - b).max() / math.sqrt(np.mean(b * b))
    st1 = st0.copy()
    y1 = chunked_scan_tf32(st1, scale=scale, passes=1, products=_products_bf16, **x)
    st3 = st0.copy()
    y3 = chunked_scan_tf32(st3, scale=scale, passes=3, products=_products_bf16, **x)
    assert rel(y1, y_ref) > 2e-3 and rel(st1, st_ref) > 2e-3
    assert rel(y3, y_ref) < 3e-4 and rel(st3, st_ref) < 3e-4
