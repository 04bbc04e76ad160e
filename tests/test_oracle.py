"""Pins for the CPU oracle: closed forms, invariants and independent formulations.

Each pin checks the oracle against something other than itself: a value fixed
by the mathematics, a library routine (numpy / scipy) that computes the same
quantity another way, or the dense-matrix form of the recurrence. The pins are
chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in any oracle function fails at least one of them
(tests/test_oracle_mutants.py checks exactly that).
"""
import math

import numpy as np
import pytest
from scipy.special import expit

import oracle

PRECS = ("f32", "f64")
TOL = {"f32": 2e-6, "f64": 1e-13}


def rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- scalar functions

@pytest.mark.parametrize("prec", PRECS)
def test_softplus_closed_forms(prec):
    # softplus(0) = ln 2 exactly (log1p(exp(0)) = log 2).
    assert oracle.softplus(0.0, prec) == pytest.approx(math.log(2.0), rel=TOL[prec])
    # Above the guard the value is the argument itself.
    for v in (20.5, 31.0, 100.0, 1e4):
        assert oracle.softplus(v, prec) == pytest.approx(v, rel=1e-7)
    # Continuity at the guard: softplus(20) - 20 = log1p(exp(-20)) < 2.1e-9.
    assert abs(oracle.softplus(20.0, "f64") - 20.0) < 2.1e-9
    assert abs(oracle.softplus(20.0, "f64") - 20.0 - math.log1p(math.exp(-20.0))) < 1e-12
    # Far below zero softplus(v) = exp(v) to first order.
    assert oracle.softplus(-30.0, prec) == pytest.approx(math.exp(-30.0), rel=1e-6)
    # Against numpy's logaddexp(0, v) = log(1 + e^v) across the range.
    for v in np.linspace(-15, 19.9, 41):
        assert oracle.softplus(v, prec) == pytest.approx(np.logaddexp(0.0, v), rel=TOL[prec] * 4,
                                                         abs=1e-30)


@pytest.mark.parametrize("prec", PRECS)
def test_silu_sigmoid_closed_forms(prec):
    assert oracle.silu(0.0, prec) == 0.0
    assert oracle.silu(1.0, prec) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=TOL[prec])
    for x in np.linspace(-8, 8, 33):
        # silu(x) - silu(-x) = x, and silu(x) = x * expit(x).
        assert oracle.silu(x, prec) - oracle.silu(-x, prec) == pytest.approx(x, abs=4 * TOL[prec])
        assert oracle.silu(x, prec) == pytest.approx(x * expit(x), rel=4 * TOL[prec], abs=1e-30)
    b = np.linspace(-6, 6, 25)
    s = oracle.sigmoid(b, prec)
    assert s[12] == 0.5
    np.testing.assert_allclose(s + s[::-1], 1.0, rtol=0, atol=4 * TOL[prec])
    np.testing.assert_allclose(s, expit(b), rtol=4 * TOL[prec])


@pytest.mark.parametrize("prec", PRECS)
def test_decay_gate(prec):
    r = rng(1)
    rows, H = 5, 6
    alpha = r.normal(0, 3, (rows, H))
    dt = r.normal(0, 1, H)
    a = -np.exp(r.uniform(-1, 1, H))
    g = oracle.decay_gate(alpha, dt, a, prec)
    want = a[None, :] * np.logaddexp(0.0, alpha + dt[None, :])
    np.testing.assert_allclose(g, want, rtol=8 * TOL[prec])
    # a = -1, dt = 0 gives g = -softplus(alpha); its inverse alpha = log(expm1(-g))
    # reproduces a target log-decay.
    target = np.linspace(-2.0, -0.01, 12).reshape(2, 6)
    g2 = oracle.decay_gate(np.log(np.expm1(-target)), np.zeros(6), -np.ones(6), prec)
    np.testing.assert_allclose(g2, target, rtol=16 * TOL[prec])
    assert np.all(g <= 0)


# ---------------------------------------------------------------- conv1d + SiLU

@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("K", [2, 3, 4, 6])
def test_conv_impulse_response(prec, K):
    """Zero history, a unit impulse on channel c at t=0: the pre-activation at
    t = 0..K-1 is w[c][K-1], w[c][K-2], ..., w[c][0], then zero; other channels
    stay zero. Pins tap order, the raw-input roll and channel independence."""
    r = rng(2)
    C, T = 7, K + 3
    w = r.normal(0, 0.5, (C, K))
    dt = np.float32 if prec == "f32" else np.float64
    for c in (0, 3, 6):
        qkv = np.zeros((1, T, C))
        qkv[0, 0, c] = 1.0
        cs = np.zeros((1, C, K - 1), dtype=dt)
        pre, _ = oracle.conv1d_silu_seq(qkv, w, cs, apply_silu=False, prec=prec)
        want = np.zeros((T, C))
        want[:K, c] = w[c, ::-1]
        np.testing.assert_allclose(pre[0], want, rtol=TOL[prec], atol=0)
        out, _ = oracle.conv1d_silu_seq(qkv, w, np.zeros((1, C, K - 1), dtype=dt), prec=prec)
        np.testing.assert_allclose(out[0], want * expit(want), rtol=4 * TOL[prec], atol=1e-30)


@pytest.mark.parametrize("prec", PRECS)
def test_conv_matches_correlate(prec):
    """Against numpy's correlate over [history, inputs]; the state ends holding the
    last K-1 RAW inputs."""
    r = rng(3)
    N, T, C, K = 2, 9, 5, 4
    qkv = r.normal(0, 1, (N, T, C))
    w = r.normal(0, 0.5, (C, K))
    dt = np.float32 if prec == "f32" else np.float64
    hist0 = r.normal(0, 1, (N, C, K - 1)).astype(dt)
    cs = hist0.copy()
    pre, skipped = oracle.conv1d_silu_seq(qkv, w, cs, apply_silu=False, prec=prec)
    assert skipped == 0
    for n in range(N):
        for c in range(C):
            xp = np.concatenate([hist0[n, c].astype(np.float64), qkv[n, :, c]])
            want = np.correlate(xp, w[c], mode="valid")
            np.testing.assert_allclose(pre[n, :, c], want, rtol=0, atol=8 * TOL[prec])
    np.testing.assert_array_equal(cs, np.transpose(qkv[:, -(K - 1):, :], (0, 2, 1)).astype(dt))


@pytest.mark.parametrize("prec", PRECS)
def test_conv_scan_equals_single_steps(prec):
    r = rng(4)
    N, T, C, K = 2, 6, 8, 4
    qkv = r.normal(0, 1, (N, T, C))
    w = r.normal(0, 0.5, (C, K))
    dt = np.float32 if prec == "f32" else np.float64
    cs_a = r.normal(0, 1, (N, C, K - 1)).astype(dt)
    cs_b = cs_a.copy()
    out_a, _ = oracle.conv1d_silu_seq(qkv, w, cs_a, prec=prec)
    for t in range(T):
        out_t, _ = oracle.conv1d_silu_seq(qkv[:, t:t + 1], w, cs_b, prec=prec)
        np.testing.assert_array_equal(out_t[:, 0], out_a[:, t])
    np.testing.assert_array_equal(cs_a, cs_b)


# ---------------------------------------------------------------- L2 norm, gated norm

@pytest.mark.parametrize("prec", PRECS)
def test_l2norm(prec):
    r = rng(5)
    x = r.normal(0, 1, (6, 32))
    x[2] = 0.0
    out = oracle.l2norm(x, 1e-6, prec)
    nrm = np.linalg.norm(out, axis=1)
    np.testing.assert_allclose(nrm[[0, 1, 3, 4, 5]], 1.0, rtol=4 * TOL[prec])
    np.testing.assert_array_equal(out[2], 0.0)
    np.testing.assert_allclose(out, x / np.maximum(np.linalg.norm(x, axis=1, keepdims=True), 1e-6),
                               rtol=4 * TOL[prec], atol=1e-30)
    # Below eps the divisor is eps itself.
    tiny = np.full((1, 4), 1e-9)
    np.testing.assert_allclose(oracle.l2norm(tiny, 1e-6, prec), tiny / 1e-6, rtol=4 * TOL[prec])


@pytest.mark.parametrize("prec", PRECS)
def test_gated_norm(prec):
    r = rng(6)
    rows, D, eps = 5, 32, 1e-6
    y = r.normal(0, 1, (rows, D))
    z = r.normal(0, 1, (rows, D))
    w = r.normal(1, 0.1, D)
    out = oracle.gated_norm(y, w, z, eps, prec)
    want = y / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps) * w * (z * expit(z))
    np.testing.assert_allclose(out, want, rtol=16 * TOL[prec], atol=1e-30)
    # The weight is shared by every row: identical (y, z) rows give identical outputs.
    y[3], z[3] = y[1], z[1]
    out = oracle.gated_norm(y, w, z, eps, prec)
    np.testing.assert_array_equal(out[3], out[1])
    # Scale invariance with eps = 0, and the constant-row closed form.
    out1 = oracle.gated_norm(y, w, z, 0.0, prec)
    out2 = oracle.gated_norm(7.5 * y, w, z, 0.0, prec)
    np.testing.assert_allclose(out1, out2, rtol=16 * TOL[prec])
    c = -0.37
    yc = np.full((1, D), c)
    zc = np.full((1, D), 30.0)  # silu(30) = 30 to double precision
    got = oracle.gated_norm(yc, np.ones(D), zc, eps, prec)
    np.testing.assert_allclose(got, c / math.sqrt(c * c + eps) * 30.0, rtol=16 * TOL[prec])


# ---------------------------------------------------------------- recurrence

def _unit(r, shape):
    x = r.normal(0, 1, shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rec_inputs(r, N, T, Hk, H, S, g_lo=-2.0, g_hi=-0.01):
    return dict(q=_unit(r, (N, T, Hk, S)), k=_unit(r, (N, T, Hk, S)),
                v=r.normal(0, 1, (N, T, H, S)), g=r.uniform(g_lo, g_hi, (N, T, H)),
                beta=expit(r.normal(0, 1, (N, T, H))))


def _dense_reference(state_t, q, k, v, g, beta, scale, Hk):
    """Dense-matrix form of the recurrence, fp64:
        S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,  y_t = scale S_t^T q_t
    with S_h[i][j] = state[h][j][i] (the transposed storage)."""
    N, T, H, S = v.shape
    Sm = np.transpose(state_t, (0, 1, 3, 2)).astype(np.float64).copy()  # [N][H][i][j]
    y = np.zeros((N, T, H, S))
    eye = np.eye(S)
    for n in range(N):
        for t in range(T):
            for h in range(H):
                kk, qq = k[n, t, h % Hk], q[n, t, h % Hk]
                Sm[n, h] = (np.exp(g[n, t, h]) * (eye - beta[n, t, h] * np.outer(kk, kk)) @ Sm[n, h]
                            + beta[n, t, h] * np.outer(kk, v[n, t, h]))
                y[n, t, h] = scale * Sm[n, h].T @ qq
    return np.transpose(Sm, (0, 1, 3, 2)), y


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("Hk,H", [(1, 1), (1, 2), (2, 4)])
def test_recurrence_bruteforce_dense(prec, Hk, H):
    r = rng(7)
    N, T, S = 2, 16, 4
    x = _rec_inputs(r, N, T, Hk, H, S)
    st0 = r.normal(0, 0.1, (N, H, S, S))
    scale = 1 / math.sqrt(S)
    want_state, want_y = _dense_reference(st0, scale=scale, Hk=Hk, **x)
    dt = np.float32 if prec == "f32" else np.float64
    st = st0.astype(dt)
    y, skipped = oracle.recurrence(st, scale=scale, prec=prec, **x)
    assert skipped == 0
    tol = 1e-12 if prec == "f64" else 2e-5
    np.testing.assert_allclose(y, want_y, rtol=0, atol=tol * (1 + np.abs(want_y).max()))
    np.testing.assert_allclose(st, want_state, rtol=0, atol=tol * (1 + np.abs(want_state).max()))


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_identity_step(prec):
    """beta = 0 and g = 0 leave the state unchanged and read out y = scale S^T q."""
    r = rng(8)
    N, T, Hk, H, S = 1, 3, 2, 4, 32
    x = _rec_inputs(r, N, T, Hk, H, S)
    x["beta"][:] = 0.0
    x["g"][:] = 0.0
    dt = np.float32 if prec == "f32" else np.float64
    st0 = r.normal(0, 0.1, (N, H, S, S)).astype(dt)
    st = st0.copy()
    y, _ = oracle.recurrence(st, scale=0.25, prec=prec, **x)
    np.testing.assert_array_equal(st, st0)
    for t in range(T):
        for h in range(H):
            want = 0.25 * st0[0, h].astype(np.float64) @ x["q"][0, t, h % Hk]
            np.testing.assert_allclose(y[0, t, h], want, rtol=0, atol=8 * TOL[prec])


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_delta_rule_exact_write(prec):
    """beta = 1, exp(g) = 1 and a unit k: after the write S^T k = v exactly."""
    r = rng(9)
    N, Hk, H, S = 1, 2, 4, 32
    x = _rec_inputs(r, N, 1, Hk, H, S)
    x["beta"][:] = 1.0
    x["g"][:] = 0.0
    dt = np.float32 if prec == "f32" else np.float64
    st = r.normal(0, 0.1, (N, H, S, S)).astype(dt)
    oracle.recurrence(st, scale=1.0, prec=prec, **x)
    for h in range(H):
        sk = st[0, h].astype(np.float64) @ x["k"][0, 0, h % Hk]  # row j dotted with k = (S^T k)_j
        np.testing.assert_allclose(sk, x["v"][0, 0, h], rtol=0,
                                   atol=1e-12 if prec == "f64" else 1e-5)


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_decay_closed_form(prec):
    """beta = 0: S_T = exp(sum_t g_t) S_0."""
    r = rng(10)
    N, T, Hk, H, S = 2, 8, 1, 2, 32
    x = _rec_inputs(r, N, T, Hk, H, S)
    x["beta"][:] = 0.0
    dt = np.float32 if prec == "f32" else np.float64
    st0 = r.normal(0, 0.1, (N, H, S, S))
    st = st0.astype(dt)
    oracle.recurrence(st, scale=1.0, prec=prec, **x)
    want = np.exp(x["g"].sum(axis=1))[:, :, None, None] * st0
    np.testing.assert_allclose(st, want, rtol=1e-12 if prec == "f64" else 2e-6, atol=1e-30)


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_single_token_from_zero(prec):
    """From a zero state one token gives S = beta k v^T and y = scale beta (q.k) v."""
    r = rng(11)
    N, Hk, H, S = 2, 2, 4, 32
    x = _rec_inputs(r, N, 1, Hk, H, S)
    dt = np.float32 if prec == "f32" else np.float64
    st = np.zeros((N, H, S, S), dtype=dt)
    scale = 1 / math.sqrt(S)
    y, _ = oracle.recurrence(st, scale=scale, prec=prec, **x)
    for n in range(N):
        for h in range(H):
            kk, qq, vv, b = x["k"][n, 0, h % Hk], x["q"][n, 0, h % Hk], x["v"][n, 0, h], x["beta"][n, 0, h]
            np.testing.assert_allclose(st[n, h], b * np.outer(vv, kk), rtol=0, atol=8 * TOL[prec])
            np.testing.assert_allclose(y[n, 0, h], scale * b * (qq @ kk) * vv, rtol=0,
                                       atol=16 * TOL[prec])


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_t4_identity(prec):
    """y_j = scale (sum_i e^g r_i q_i + delta_j (k.q)) with delta_j = (v_j - e^g r.k) beta,
    r the state row before the token: the read-after-write output via the
    factorised two-sum form."""
    r = rng(12)
    N, Hk, H, S = 1, 2, 4, 32
    x = _rec_inputs(r, N, 1, Hk, H, S)
    dt = np.float32 if prec == "f32" else np.float64
    st0 = r.normal(0, 0.1, (N, H, S, S))
    st = st0.astype(dt)
    scale = 1 / math.sqrt(S)
    y, _ = oracle.recurrence(st, scale=scale, prec=prec, **x)
    for h in range(H):
        kk, qq = x["k"][0, 0, h % Hk], x["q"][0, 0, h % Hk]
        e = np.exp(x["g"][0, 0, h])
        rows = st0[0, h]
        delta = (x["v"][0, 0, h] - e * rows @ kk) * x["beta"][0, 0, h]
        want = scale * (e * rows @ qq + delta * (kk @ qq))
        np.testing.assert_allclose(y[0, 0, h], want, rtol=0, atol=1e-13 if prec == "f64" else 1e-6)


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_gqa_tiled_mapping(prec):
    """v-head vh reads k-head vh % Hk: identical to Hk = H with q, k tiled
    [k0, k1, k0, k1], and different from the blocked repeat [k0, k0, k1, k1]."""
    r = rng(13)
    N, T, Hk, H, S = 1, 4, 2, 4, 32
    x = _rec_inputs(r, N, T, Hk, H, S)
    dt = np.float32 if prec == "f32" else np.float64
    st0 = r.normal(0, 0.1, (N, H, S, S)).astype(dt)
    st_a, st_b, st_c = st0.copy(), st0.copy(), st0.copy()
    y_a, _ = oracle.recurrence(st_a, scale=0.5, prec=prec, **x)
    tiled = dict(x, q=np.tile(x["q"], (1, 1, 2, 1)), k=np.tile(x["k"], (1, 1, 2, 1)))
    y_b, _ = oracle.recurrence(st_b, scale=0.5, prec=prec, **tiled)
    np.testing.assert_array_equal(y_a, y_b)
    np.testing.assert_array_equal(st_a, st_b)
    blocked = dict(x, q=np.repeat(x["q"], 2, axis=2), k=np.repeat(x["k"], 2, axis=2))
    y_c, _ = oracle.recurrence(st_c, scale=0.5, prec=prec, **blocked)
    assert not np.array_equal(y_a, y_c)


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_scan_equals_steps_and_split(prec):
    r = rng(14)
    N, T, Hk, H, S = 2, 10, 1, 2, 32
    x = _rec_inputs(r, N, T, Hk, H, S)
    dt = np.float32 if prec == "f32" else np.float64
    st0 = r.normal(0, 0.1, (N, H, S, S)).astype(dt)
    st_a, st_b, st_c = st0.copy(), st0.copy(), st0.copy()
    y_a, _ = oracle.recurrence(st_a, scale=0.5, prec=prec, **x)
    for t in range(T):
        y_t, _ = oracle.recurrence(st_b, scale=0.5, prec=prec,
                                   **{k_: v_[:, t:t + 1] for k_, v_ in x.items()})
        np.testing.assert_array_equal(y_t[:, 0], y_a[:, t])
    np.testing.assert_array_equal(st_a, st_b)
    for lo, hi in ((0, 4), (4, T)):
        y_c, _ = oracle.recurrence(st_c, scale=0.5, prec=prec,
                                   **{k_: v_[:, lo:hi] for k_, v_ in x.items()})
        np.testing.assert_array_equal(y_c, y_a[:, lo:hi])
    np.testing.assert_array_equal(st_a, st_c)


@pytest.mark.parametrize("prec", PRECS)
def test_recurrence_slots(prec):
    """Sequence n uses slot slots[n]; untouched slots stay bit-identical; an
    out-of-range slot is skipped, counted and writes nothing."""
    r = rng(15)
    N, T, Hk, H, S, P = 4, 2, 1, 2, 32, 6
    x = _rec_inputs(r, N, T, Hk, H, S)
    dt = np.float32 if prec == "f32" else np.float64
    pool0 = r.normal(0, 0.1, (P, H, S, S)).astype(dt)
    slots = np.array([4, 0, 9, 2], dtype=np.int32)
    pool = pool0.copy()
    y, skipped = oracle.recurrence(pool, scale=0.5, slots=slots, prec=prec, **x)
    assert skipped == 1
    np.testing.assert_array_equal(y[2], 0.0)
    for s in (1, 3, 5):
        np.testing.assert_array_equal(pool[s], pool0[s])
    for n, s in ((0, 4), (1, 0), (3, 2)):
        alone = pool0[s:s + 1].copy()
        y1, _ = oracle.recurrence(alone, scale=0.5, prec=prec,
                                  **{k_: v_[n:n + 1] for k_, v_ in x.items()})
        np.testing.assert_array_equal(pool[s], alone[0])
        np.testing.assert_array_equal(y[n], y1[0])
    slots[0] = -1
    pool = pool0.copy()
    _, skipped = oracle.recurrence(pool, scale=0.5, slots=slots, prec=prec, **x)
    assert skipped == 2
    np.testing.assert_array_equal(pool[4], pool0[4])


def test_oracle_precisions_agree():
    r = rng(16)
    N, T, Hk, H, S = 1, 16, 2, 4, 32
    x = _rec_inputs(r, N, T, Hk, H, S)
    st0 = r.normal(0, 0.1, (N, H, S, S))
    st32, st64 = st0.astype(np.float32), st0.astype(np.float64)
    y32, _ = oracle.recurrence(st32, scale=0.25, prec="f32", **x)
    y64, _ = oracle.recurrence(st64, scale=0.25, prec="f64", **x)
    np.testing.assert_allclose(y32, y64, rtol=0, atol=1e-5)
    np.testing.assert_allclose(st32, st64, rtol=0, atol=1e-5)


# ---------------------------------------------------------------- whole block

def _block_reference(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, Hk, scale,
                     l2_eps, norm_eps):
    """Independent fp64 restatement of one decode token of the block, built from
    library routines: np.correlate for the conv, expit for SiLU and the sigmoid,
    logaddexp for softplus, np.linalg.norm, the dense-matrix recurrence."""
    N, C = qkv.shape
    P, H, S, _ = state.shape
    K = conv_w.shape[1]
    key = Hk * S
    cs = conv_state.astype(np.float64).copy()
    st = state.astype(np.float64).copy()
    out = np.zeros((N, H, S))
    for n in range(N):
        pre = np.array([np.correlate(np.append(cs[n, c], qkv[n, c]), conv_w[c], "valid")[0]
                        for c in range(C)])
        xo = pre * expit(pre)
        cs[n] = np.concatenate([cs[n][:, 1:], qkv[n][:, None]], axis=1)
        qh = xo[:key].reshape(Hk, S)
        kh = xo[key:2 * key].reshape(Hk, S)
        qh = qh / np.maximum(np.linalg.norm(qh, axis=1, keepdims=True), l2_eps)
        kh = kh / np.maximum(np.linalg.norm(kh, axis=1, keepdims=True), l2_eps)
        v = xo[2 * key:].reshape(H, S)
        g = a * np.logaddexp(0.0, alpha[n] + dt)
        beta = expit(b[n])
        new_st, y = _dense_reference(st[n:n + 1], qh[None, None], kh[None, None], v[None, None],
                                     g[None, None], beta[None, None], scale, Hk)
        st[n] = new_st[0]
        yy = y[0, 0]
        out[n] = yy / np.sqrt(np.mean(yy * yy, axis=1, keepdims=True) + norm_eps) * norm_w \
            * (z[n] * expit(z[n]))
    return out, cs, st


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("Hk,H,S", [(2, 4, 8), (1, 1, 4), (2, 2, 8)])
def test_block_decode_against_independent_form(prec, Hk, H, S):
    r = rng(17)
    N, K = 3, 4
    C = 2 * Hk * S + H * S
    qkv = r.normal(0, 1, (N, C))
    conv_w = r.normal(0, 0.5, (C, K))
    cs0 = r.normal(0, 1, (N, C, K - 1))
    alpha = r.normal(0, 2, (N, H))
    b = r.normal(0, 1, (N, H))
    dt_ = r.normal(0, 0.5, H)
    a = -np.exp(r.uniform(-0.5, 0.5, H))
    z = r.normal(0, 1, (N, H, S))
    nw = r.normal(1, 0.1, S)
    st0 = r.normal(0, 0.1, (N, H, S, S))
    scale = 1 / math.sqrt(S)
    want_out, want_cs, want_st = _block_reference(qkv, conv_w, cs0, alpha, b, dt_, a, z, nw, st0,
                                                  Hk, scale, 1e-6, 1e-6)
    dty = np.float32 if prec == "f32" else np.float64
    cs, st = cs0.astype(dty), st0.astype(dty)
    out, skipped = oracle.block_decode(qkv, conv_w, cs, alpha, b, dt_, a, z, nw, st, Hk, scale,
                                       1e-6, 1e-6, prec=prec)
    assert skipped == 0
    tol = 1e-11 if prec == "f64" else 5e-5
    np.testing.assert_allclose(out, want_out, rtol=0, atol=tol * (1 + np.abs(want_out).max()))
    np.testing.assert_allclose(st, want_st, rtol=0, atol=tol)
    np.testing.assert_array_equal(cs, want_cs.astype(dty))
