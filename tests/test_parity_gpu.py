"""GPU parity: every entry point of libgdn.so against the CPU oracle.

All inputs come from the seeded generators; the oracle (double build) and the
GPU see the same float32 arrays. Tolerances are the ones stated for the method:
  - one step (single token, or the first of a chain): elementwise
    |gpu - ref| <= 1e-4 + 1e-4 * |ref| for y/out and the state;
  - after a long chain or scan: max |gpu - ref| <= 2e-3 * RMS(ref), per tensor.
Within the GPU library, the scan and repeated decode calls (and the scan split in
two) must agree bit for bit; the fused block with a whole head per CTA must
equal the unfused pipeline bit for bit.
"""
import numpy as np
import pytest

import oracle
from gated_deltanet_linear_scan_gb300 import inputs as I
from tests.oracle_units import prefill_4x4096

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ helpers

def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def assert_step(gpu, ref, name):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, name
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    err = np.abs(gpu - ref)
    bound = 1e-4 + 1e-4 * np.abs(ref)
    worst = np.max(err - bound)
    assert worst <= 0, f"{name}: elementwise bound exceeded by {worst:.3e} (max err {err.max():.3e})"


def assert_rms(gpu, ref, name, rel=2e-3):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    rms = np.sqrt(np.mean(ref * ref))
    err = np.max(np.abs(gpu - ref))
    assert err <= rel * rms, f"{name}: max err {err:.3e} > {rel} * RMS {rms:.3e}"


@pytest.fixture(scope="module", autouse=True)
def lib(cuda_lib):
    yield cuda_lib
    cuda_lib.gdn_device_error()  # no bounded wait gave up during the module


# ------------------------------------------------------------------ small steps

def test_decay_gate_and_beta(lib):
    r = np.random.default_rng(100)
    rows, H = 37, 32
    alpha = r.normal(0, 6, (rows, H)).astype(np.float32)
    alpha[0, :4] = [25.0, 20.0, 19.99, -40.0]  # both sides of the guard at 20
    dt = r.normal(0, 0.5, H).astype(np.float32)
    a = (-np.exp(r.uniform(-1, 1, H))).astype(np.float32)
    g = torch.empty(rows, H, device="cuda")
    lib.gdn_decay_gate(dev(alpha), dev(dt), dev(a), g, H, rows)
    assert_step(host(g), oracle.decay_gate(alpha, dt, a), "g")
    b = r.normal(0, 3, 1001).astype(np.float32)
    beta = dev(b)
    lib.gdn_beta_sigmoid(beta, beta, b.size)  # in place
    assert_step(host(beta), oracle.sigmoid(b), "beta")


@pytest.mark.parametrize("K", [2, 3, 4, 5, 8])
# T = 65 and 150 cross the scan's 64-position blocks, with a ragged last block
# C = 250 runs the one-channel-a-thread form (a channel count not divisible by 4)
@pytest.mark.parametrize("C,T", [(256, 1), (256, 21), (8192, 3), (256, 65), (512, 150), (250, 70)])
def test_conv1d_silu(lib, K, C, T):
    r = np.random.default_rng(101 + K)
    N, P = 3, 5
    slots = np.array([4, 0, 2], dtype=np.int32)
    qkv = r.normal(0, 1, (N, T, C)).astype(np.float32)
    w = r.normal(0, 0.5, (C, K)).astype(np.float32)
    cs0 = r.normal(0, 1, (P, C, K - 1)).astype(np.float32)
    cs = dev(cs0)
    out = torch.zeros(N, T, C, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gdn_conv1d_silu_seq(dev(qkv), dev(w), cs, out, N, T, C, K, slots=dev(slots), pool=P,
                            err_count=err)
    cs_ref = f64(cs0)
    out_ref, skipped = oracle.conv1d_silu_seq(qkv, w, cs_ref, slots=slots, pool=P)
    assert skipped == 0 and host(err)[0] == 0
    assert_step(host(out), out_ref, "conv out")
    assert_step(host(cs), cs_ref, "conv_state")
    for s in (1, 3):
        np.testing.assert_array_equal(host(cs)[s], cs0[s])
    # the scan equals T single-token calls, bit for bit
    cs2 = dev(cs0)
    for t in range(T):
        o1 = torch.zeros(N, C, device="cuda")
        lib.gdn_conv1d_silu(dev(qkv[:, t]), dev(w), cs2, o1, N, C, K, slots=dev(slots), pool=P)
        np.testing.assert_array_equal(host(o1), host(out)[:, t])
    np.testing.assert_array_equal(host(cs2), host(cs))


def test_conv1d_silu_channel_grouping_same_bits(lib):
    """Four channels a thread (16-byte accesses) and one channel a thread (the form for
    rows that are not 16-byte aligned) give the same bits: the same inputs, and outputs
    one float past a 16-byte boundary, against the aligned call."""
    r = np.random.default_rng(106)
    N, T, C, K = 2, 150, 512, 4
    qkv = r.normal(0, 1, (N, T, C)).astype(np.float32)
    w = dev(r.normal(0, 0.5, (C, K)).astype(np.float32))
    cs0 = r.normal(0, 1, (N, C, K - 1)).astype(np.float32)
    cs_a, out_a = dev(cs0), torch.zeros(N, T, C, device="cuda")
    lib.gdn_conv1d_silu_seq(dev(qkv), w, cs_a, out_a, N, T, C, K)
    qb = torch.zeros(qkv.size + 1, device="cuda")
    qb[1:] = dev(qkv).reshape(-1)
    ob = torch.zeros(out_a.numel() + 1, device="cuda")
    cs_b = dev(cs0)
    lib.gdn_conv1d_silu_seq(qb[1:].view(N, T, C), w, cs_b, ob[1:].view(N, T, C), N, T, C, K)
    assert torch.equal(ob[1:].view(N, T, C), out_a)
    assert torch.equal(cs_b, cs_a)


def test_conv1d_silu_invalid_slot(lib):
    r = np.random.default_rng(102)
    N, C, K, P = 3, 256, 4, 4
    slots = np.array([1, 7, -2], dtype=np.int32)
    qkv = r.normal(0, 1, (N, C)).astype(np.float32)
    w = r.normal(0, 0.5, (C, K)).astype(np.float32)
    cs0 = r.normal(0, 1, (P, C, K - 1)).astype(np.float32)
    cs = dev(cs0)
    out = torch.full((N, C), 7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gdn_conv1d_silu(dev(qkv), dev(w), cs, out, N, C, K, slots=dev(slots), pool=P,
                        err_count=err)
    assert host(err)[0] == 2
    o = host(out)
    assert np.all(o[1:] == 7.0)
    np.testing.assert_array_equal(host(cs)[[0, 2, 3]], cs0[[0, 2, 3]])


# SiLU's argument over its whole range. It covers values near zero, values whose result
# is x itself, and values below about -88, where exp(-x) overflows and the divisor passes
# 2^126. The arguments go through the conv (the current tap alone with weight 1, so the
# pre-activation is the input) and through the gated norm's gate.
SILU_ARGS = np.array([0.0, -0.0, 1e-30, -1e-30, 1e-3, -1e-3, 0.5, -0.5, 1.0, -1.0, 5.0, -5.0,
                      10.0, -10.0, 20.0, -20.0, 50.0, -50.0, 87.0, -87.0, 88.5, -88.5, 89.0,
                      -89.0, 100.0, -100.0, 1000.0, -1000.0, 3e38, -3e38], dtype=np.float32)


def test_silu_argument_range(lib):
    C, T, K = 256, 3, 2
    qkv = np.stack([np.resize(np.roll(SILU_ARGS, 7 * t), C) for t in range(T)])[None]
    w = np.tile(np.array([0.0, 1.0], dtype=np.float32), (C, 1))
    cs0 = np.zeros((1, C, K - 1), dtype=np.float32)
    out = torch.zeros(1, T, C, device="cuda")
    lib.gdn_conv1d_silu_seq(dev(qkv), dev(w), dev(cs0), out, 1, T, C, K)
    ref, _ = oracle.conv1d_silu_seq(qkv, w, f64(cs0))
    got = host(out)
    assert_step(got, ref, "silu through the conv")
    assert np.all(np.abs(got[qkv <= -100.0]) <= 1e-30)
    # the fast exponential and division stay within 1e-5 relative where |x| <= 20 (the
    # range a conv output takes): far inside the one-step bound
    mid = np.abs(qkv) <= 20.0
    assert np.all(np.abs(got[mid] - ref[mid]) <= 1e-5 * np.abs(ref[mid]) + 1e-37)

    # the gate's arguments up to 1000 in magnitude: with z = 3e38 the gated output
    # y w silu(z) / rms is beyond fp32's range whatever SiLU returns
    D, rows = 128, 8
    zargs = SILU_ARGS[np.abs(SILU_ARGS) <= 1000.0]
    z = np.stack([np.resize(np.roll(zargs, 3 * i), D) for i in range(rows)])
    y = np.random.default_rng(105).normal(0, 1, (rows, D)).astype(np.float32)
    nw = np.ones(D, dtype=np.float32)
    o = torch.empty(rows, D, device="cuda")
    lib.gdn_gated_norm(dev(y), dev(nw), dev(z), o, rows, D, 1e-6)
    assert_step(host(o), oracle.gated_norm(y, nw, z, 1e-6), "silu through the gated norm")


@pytest.mark.parametrize("Hk,H,S", [(2, 4, 32), (16, 32, 128), (1, 2, 64), (2, 4, 256)])
def test_qkv_split_norm(lib, Hk, H, S):
    r = np.random.default_rng(103)
    rows = 5
    C = 2 * Hk * S + H * S
    x = r.normal(0, 1, (rows, C)).astype(np.float32)
    x[2, :S] = 0.0  # a zero q head: maps to zeros
    q = torch.empty(rows, Hk, S, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty(rows, H, S, device="cuda")
    lib.gdn_qkv_split_norm(dev(x), q, k, v, rows, Hk, H, S, 1e-6)
    key = Hk * S
    assert_step(host(q), oracle.l2norm(x[:, :key].reshape(rows, Hk, S), 1e-6), "q")
    assert_step(host(k), oracle.l2norm(x[:, key:2 * key].reshape(rows, Hk, S), 1e-6), "k")
    np.testing.assert_array_equal(host(v), x[:, 2 * key:].reshape(rows, H, S))


@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_gated_norm(lib, D):
    r = np.random.default_rng(104)
    rows = 67
    y = r.normal(0, 1, (rows, D)).astype(np.float32)
    z = r.normal(0, 1, (rows, D)).astype(np.float32)
    w = r.normal(1, 0.1, D).astype(np.float32)
    out = torch.empty(rows, D, device="cuda")
    lib.gdn_gated_norm(dev(y), dev(w), dev(z), out, rows, D, 1e-6)
    assert_step(host(out), oracle.gated_norm(y, w, z, 1e-6), "gated norm")
    yt = dev(y)
    lib.gdn_gated_norm(yt, dev(w), dev(z), yt, rows, D, 1e-6)  # in place
    np.testing.assert_array_equal(host(yt), host(out))


# ------------------------------------------------------------------ recurrence

def rec_case(Hk, H, S, N, T, seed, pool=None):
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=S, n_seqs=N, n_tokens=T,
                       pool=pool, cid=200 + seed)
    x = I.recurrence_batch(cfg)
    st0 = I.state_pool(cfg)
    return cfg, x, st0


def run_decode(lib, cfg, x, st, t, slots=None, pool=None, err=None):
    N, H, S = cfg.n_seqs, cfg.n_v_heads, cfg.state_size
    y = torch.zeros(N, H, S, device="cuda")
    lib.gdn_recurrence_decode(st, dev(x["q"][:, t]), dev(x["k"][:, t]), dev(x["v"][:, t]),
                              dev(x["g"][:, t]), dev(x["beta"][:, t]), y, N, cfg.n_k_heads, H, S,
                              cfg.scale, slots=slots, pool=pool, err_count=err)
    return y


@pytest.mark.parametrize("Hk,H,S", [(2, 4, 32), (16, 32, 128), (1, 1, 64), (4, 16, 256),
                                    (8, 8, 128)])
def test_recurrence_decode(lib, Hk, H, S):
    cfg, x, st0 = rec_case(Hk, H, S, N=3, T=1, seed=S + H)
    st = dev(st0)
    y = run_decode(lib, cfg, x, st, 0)
    st_ref = f64(st0)
    y_ref, _ = oracle.recurrence(st_ref, x["q"][:, :1], x["k"][:, :1], x["v"][:, :1],
                                 x["g"][:, :1], x["beta"][:, :1], cfg.scale)
    assert_step(host(y), y_ref[:, 0], "y")
    assert_step(host(st), st_ref, "state")


def test_recurrence_decode_slots(lib):
    cfg, x, _ = rec_case(2, 4, 128, N=4, T=1, seed=7, pool=9)
    pool0 = I.state_pool(cfg)
    slots = np.array([5, 0, 11, 3], dtype=np.int32)  # 11 is out of range
    st = dev(pool0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = run_decode(lib, cfg, x, st, 0, slots=dev(slots), pool=9, err=err)
    assert host(err)[0] == 1
    st_ref = f64(pool0)
    y_ref, skipped = oracle.recurrence(st_ref, x["q"][:, :1], x["k"][:, :1], x["v"][:, :1],
                                       x["g"][:, :1], x["beta"][:, :1], cfg.scale, slots=slots,
                                       pool=9)
    assert skipped == 1
    got = host(st)
    for s in (1, 2, 4, 6, 7, 8):
        np.testing.assert_array_equal(got[s], pool0[s])  # untouched slots keep their bits
    assert_step(got, st_ref, "state pool")
    yy = host(y)
    assert np.all(yy[2] == 0.0)
    assert_step(yy[[0, 1, 3]], y_ref[[0, 1, 3], 0], "y")


def run_scan(lib, cfg, x, st, lo, hi, slots=None, pool=None, err=None):
    N, H, S = cfg.n_seqs, cfg.n_v_heads, cfg.state_size
    T = hi - lo
    y = torch.zeros(N, T, H, S, device="cuda")
    sl = lambda a: dev(a[:, lo:hi])  # noqa: E731
    lib.gdn_recurrence_scan(st, sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]), y,
                            N, T, cfg.n_k_heads, H, S, cfg.scale, slots=slots, pool=pool,
                            err_count=err)
    return y


@pytest.mark.parametrize("Hk,H,S,T", [(2, 4, 32, 16), (2, 4, 128, 37), (1, 2, 64, 5),
                                      (2, 4, 256, 33), (1, 2, 64, 50)])
def test_recurrence_scan(lib, Hk, H, S, T):
    cfg, x, st0 = rec_case(Hk, H, S, N=2, T=T, seed=T + S)
    st = dev(st0)
    y = run_scan(lib, cfg, x, st, 0, T)
    st_ref = f64(st0)
    y_ref, _ = oracle.recurrence(st_ref, x["q"], x["k"], x["v"], x["g"], x["beta"], cfg.scale)
    assert_step(host(y), y_ref, "y")
    assert_step(host(st), st_ref, "final state")
    # T decode calls agree with the scan bit for bit, and so does a split scan.
    st_d = dev(st0)
    for t in range(T):
        yd = run_decode(lib, cfg, x, st_d, t)
        np.testing.assert_array_equal(host(yd), host(y)[:, t])
    np.testing.assert_array_equal(host(st_d), host(st))
    st_s = dev(st0)
    cut = T // 2
    y1 = run_scan(lib, cfg, x, st_s, 0, cut)
    y2 = run_scan(lib, cfg, x, st_s, cut, T)
    np.testing.assert_array_equal(np.concatenate([host(y1), host(y2)], axis=1), host(y))
    np.testing.assert_array_equal(host(st_s), host(st))


def test_recurrence_scan_slots(lib):
    cfg, x, _ = rec_case(2, 4, 128, N=3, T=20, seed=3, pool=5)
    pool0 = I.state_pool(cfg)
    slots = np.array([4, -1, 1], dtype=np.int32)
    st = dev(pool0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = run_scan(lib, cfg, x, st, 0, 20, slots=dev(slots), pool=5, err=err)
    assert host(err)[0] == 1
    st_ref = f64(pool0)
    y_ref, _ = oracle.recurrence(st_ref, x["q"], x["k"], x["v"], x["g"], x["beta"], cfg.scale,
                                 slots=slots, pool=5)
    got = host(st)
    for s in (0, 2, 3):
        np.testing.assert_array_equal(got[s], pool0[s])
    assert_step(got, st_ref, "state pool")
    assert_step(host(y)[[0, 2]], y_ref[[0, 2]], "y")


@pytest.mark.slow
def test_recurrence_scan_prefill_4x4096(lib):
    """The long-scan workload at full size (N=4, T=4096, H=32, Hk=16, S=128), in the
    launch the bench times: every (sequence, v-head) unit against the oracle, y and the
    final state under the long-scan bound, the first token under the one-step bound."""
    cfg, x, st0, refs = prefill_4x4096()
    st = dev(st0)
    y = run_scan(lib, cfg, x, st, 0, cfg.n_tokens)
    yh, sth = host(y), host(st)
    assert len(refs) == cfg.n_seqs * cfg.n_v_heads
    for (n, vh), (y_ref, s_ref) in refs.items():
        assert_step(yh[n, :1, vh], y_ref[:1], f"y token 0 ({n},{vh})")
        assert_rms(yh[n, :, vh], y_ref, f"y ({n},{vh})")
        assert_rms(sth[n, vh], s_ref, f"final state ({n},{vh})")


@pytest.mark.parametrize("Hk,H,S", [(2, 4, 32), (16, 32, 128), (4, 16, 256), (1, 2, 64)])
def test_recurrence_decode_2pass(lib, Hk, H, S):
    """Factorised readout: the state is the plain decode's bit for bit, y matches the
    oracle within the one-step bound."""
    cfg, x, st0 = rec_case(Hk, H, S, N=3, T=1, seed=S + H + 7)
    N = cfg.n_seqs
    st_a, st_b = dev(st0), dev(st0)
    y_a = run_decode(lib, cfg, x, st_a, 0)
    y_b = torch.zeros(N, H, S, device="cuda")
    lib.gdn_recurrence_decode_2pass(st_b, dev(x["q"][:, 0]), dev(x["k"][:, 0]), dev(x["v"][:, 0]),
                                    dev(x["g"][:, 0]), dev(x["beta"][:, 0]), y_b, N, Hk, H, S,
                                    cfg.scale)
    assert torch.equal(st_a, st_b)
    st_ref = f64(st0)
    y_ref, _ = oracle.recurrence(st_ref, x["q"][:, :1], x["k"][:, :1], x["v"][:, :1],
                                 x["g"][:, :1], x["beta"][:, :1], cfg.scale)
    assert_step(host(y_b), y_ref[:, 0], "y (2-pass)")
    assert_step(host(y_a), host(y_b), "y plain vs 2-pass")


@pytest.mark.parametrize("S,T", [(128, 37), (32, 16), (64, 20), (256, 7)])
def test_recurrence_scan_snapshots(lib, S, T):
    """snaps[t] is the state after token t: equal bit for bit to t+1 decode calls,
    and restoring snaps[M-1] then scanning the rest reproduces the full scan."""
    cfg, x, st0 = rec_case(2, 4, S, N=2, T=T, seed=S + T + 11)
    N, H = cfg.n_seqs, cfg.n_v_heads
    st_full = dev(st0)
    y_full = run_scan(lib, cfg, x, st_full, 0, T)
    st = dev(st0)
    y = torch.zeros(N, T, H, S, device="cuda")
    snaps = torch.zeros(N, T, H, S, S, device="cuda")
    lib.gdn_recurrence_scan_snapshots(st, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]),
                                      dev(x["beta"]), y, snaps, N, T, cfg.n_k_heads, H, S,
                                      cfg.scale)
    assert torch.equal(y, y_full) and torch.equal(st, st_full)
    assert torch.equal(snaps[:, T - 1], st)
    st_d = dev(st0)
    for t in range(T):
        run_decode(lib, cfg, x, st_d, t)
        assert torch.equal(snaps[:, t], st_d), f"snapshot {t}"
    st_ref = f64(st0)
    oracle.recurrence(st_ref, scale=cfg.scale, **{k_: v_[:, :5] for k_, v_ in x.items()})
    assert_step(host(snaps[:, 4]), st_ref, "snapshot 4 vs oracle")
    M = T // 3  # accept M tokens, roll back the rest, resume
    st_r = snaps[:, M - 1].contiguous().clone()
    y_r = run_scan(lib, cfg, x, st_r, M, T)
    assert torch.equal(y_r, y_full[:, M:]) and torch.equal(st_r, st_full)


def test_snapshot_restore(lib):
    """Rollback after a verification scan: restoring each sequence to the snapshots after
    its accepted count equals scanning (and conv-scanning) only that prefix, bit for bit;
    slots route; an out-of-range count leaves its slots as the scans left them and is
    counted once; slots no sequence uses keep their bits."""
    S, T, C, K = 128, 9, 256, 4
    cfg, x, pool0 = rec_case(2, 4, S, N=4, T=T, seed=77, pool=6)
    N, H, Hk = cfg.n_seqs, cfg.n_v_heads, cfg.n_k_heads
    slots = np.array([5, 0, 3, 2], dtype=np.int32)
    accepted = np.array([1, T, 4, 0], dtype=np.int32)
    r = np.random.default_rng(78)
    qkv = r.normal(0, 1, (N, T, C)).astype(np.float32)
    w = r.normal(0, 0.5, (C, K)).astype(np.float32)
    cs0 = r.normal(0, 1, (6, C, K - 1)).astype(np.float32)
    d_slots = dev(slots)
    st, cs = dev(pool0), dev(cs0)
    y = torch.zeros(N, T, H, S, device="cuda")
    snaps = torch.zeros(N, T, H, S, S, device="cuda")
    lib.gdn_recurrence_scan_snapshots(st, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]),
                                      dev(x["beta"]), y, snaps, N, T, Hk, H, S, cfg.scale,
                                      slots=d_slots, pool=6)
    out = torch.zeros(N, T, C, device="cuda")
    csnaps = torch.zeros(N, T, C, K - 1, device="cuda")
    lib.gdn_conv1d_silu_seq_snapshots(dev(qkv), dev(w), cs, out, csnaps, N, T, C, K,
                                      slots=d_slots, pool=6)
    after_st, after_cs = host(st), host(cs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gdn_snapshot_restore(st, snaps, dev(accepted), N, T, H, S, conv_state=cs,
                             conv_snaps=csnaps, conv_dim=C, conv_kernel=K, slots=d_slots,
                             pool=6, err_count=err)
    assert host(err)[0] == 1
    got_st, got_cs = host(st), host(cs)
    for n in range(N):
        sl, m = slots[n], accepted[n]
        if not 1 <= m <= T:
            np.testing.assert_array_equal(got_st[sl], after_st[sl])
            np.testing.assert_array_equal(got_cs[sl], after_cs[sl])
            continue
        st_ref = dev(pool0[sl:sl + 1])
        lib.gdn_recurrence_scan(st_ref, *(dev(x[k_][n:n + 1, :m]) for k_ in
                                          ("q", "k", "v", "g", "beta")),
                                torch.zeros(1, m, H, S, device="cuda"), 1, m, Hk, H, S, cfg.scale)
        np.testing.assert_array_equal(got_st[sl], host(st_ref)[0], f"state of sequence {n}")
        cs_ref = dev(cs0[sl:sl + 1])
        lib.gdn_conv1d_silu_seq(dev(qkv[n:n + 1, :m]), dev(w), cs_ref,
                                torch.zeros(1, m, C, device="cuda"), 1, m, C, K)
        np.testing.assert_array_equal(got_cs[sl], host(cs_ref)[0], f"conv of sequence {n}")
    for sl in (1, 4):  # no sequence uses these slots
        np.testing.assert_array_equal(got_st[sl], pool0[sl])
        np.testing.assert_array_equal(got_cs[sl], cs0[sl])


@pytest.mark.slow
def test_recurrence_scan_snapshots_speculative_verify_size(lib):
    """The speculative-verification workload at full size (64 sequences x 4 draft tokens,
    Hk=16, H=32, S=128, the launch the bench times): the last snapshot is the final state
    bit for bit, and sampled (sequence, v-head) units match the oracle token by token in
    y and in every snapshot."""
    cfg = I.get_config(3, n_tokens=4)
    N, T, Hk, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    x = I.recurrence_batch(cfg)
    st0 = I.state_pool(cfg)
    st = dev(st0)
    y = torch.zeros(N, T, H, S, device="cuda")
    snaps = torch.zeros(N, T, H, S, S, device="cuda")
    lib.gdn_recurrence_scan_snapshots(st, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]),
                                      dev(x["beta"]), y, snaps, N, T, Hk, H, S, cfg.scale)
    assert torch.equal(snaps[:, T - 1], st)
    for n, vh in ((0, 0), (17, 5), (40, 22), (63, 31)):
        kh = vh % Hk
        unit = {"q": x["q"][n:n + 1, :, kh:kh + 1], "k": x["k"][n:n + 1, :, kh:kh + 1],
                "v": x["v"][n:n + 1, :, vh:vh + 1], "g": x["g"][n:n + 1, :, vh:vh + 1],
                "beta": x["beta"][n:n + 1, :, vh:vh + 1]}
        got_y = host(y[n, :, vh])
        got_s = host(snaps[n, :, vh])
        for t in range(T):
            s_ref = f64(st0[n:n + 1, vh:vh + 1])
            y_ref, _ = oracle.recurrence(s_ref, scale=cfg.scale,
                                         **{k_: v_[:, :t + 1] for k_, v_ in unit.items()})
            assert_step(got_y[t], y_ref[0, t, 0], f"y ({n},{vh}) token {t}")
            assert_step(got_s[t], s_ref[0, 0], f"snapshot ({n},{vh}) token {t}")


@pytest.mark.parametrize("T", [9, 130])
def test_conv1d_silu_seq_snapshots(lib, T):
    r = np.random.default_rng(105)
    N, C, K = 2, 256, 4
    qkv = r.normal(0, 1, (N, T, C)).astype(np.float32)
    w = r.normal(0, 0.5, (C, K)).astype(np.float32)
    cs0 = r.normal(0, 1, (N, C, K - 1)).astype(np.float32)
    cs = dev(cs0)
    out = torch.zeros(N, T, C, device="cuda")
    snaps = torch.zeros(N, T, C, K - 1, device="cuda")
    lib.gdn_conv1d_silu_seq_snapshots(dev(qkv), dev(w), cs, out, snaps, N, T, C, K)
    cs2 = dev(cs0)
    out2 = torch.zeros(N, T, C, device="cuda")
    lib.gdn_conv1d_silu_seq(dev(qkv), dev(w), cs2, out2, N, T, C, K)
    assert torch.equal(out, out2) and torch.equal(cs, cs2)
    cs3 = dev(cs0)
    for t in range(T):
        o1 = torch.zeros(N, C, device="cuda")
        lib.gdn_conv1d_silu(dev(qkv[:, t]), dev(w), cs3, o1, N, C, K)
        assert torch.equal(snaps[:, t], cs3), f"conv snapshot {t}"
    ref = f64(cs0)
    oracle.conv1d_silu_seq(qkv[:, :3], w, ref)
    assert_step(host(snaps[:, 2]), ref, "conv snapshot 2 vs oracle")


# ------------------------------------------------------------------ fused block

class BlockRun:
    """Chained decode steps of the fused block on the GPU, with the oracle
    following a subset of sequences in lockstep."""

    def __init__(self, lib, cfg, sample):
        self.lib, self.cfg, self.sample = lib, cfg, list(sample)
        st = I.block_static(cfg)
        self.static = st
        self.slots = I.slots(cfg)
        P = cfg.pool_size
        self.state0 = I.state_pool(cfg)
        self.conv0 = I.conv_state_pool(cfg)
        self.state = dev(self.state0)
        self.conv = dev(self.conv0)
        self.d_static = {k: dev(v) for k, v in st.items()}
        self.d_slots = dev(self.slots) if self.slots is not None else None
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ids = [self.slot_of(n) for n in self.sample]
        self.ref_state = f64(self.state0[ids])
        self.ref_conv = f64(self.conv0[ids])
        self.P = P

    def slot_of(self, n):
        return int(self.slots[n]) if self.slots is not None else n

    def step(self, step):
        cfg = self.cfg
        a = I.block_step(cfg, step)
        out = torch.zeros(cfg.n_seqs, cfg.n_v_heads, cfg.state_size, device="cuda")
        self.lib.gdn_block_decode(
            dev(a["qkv"]), self.d_static["conv_w"], self.conv, dev(a["alpha"]), dev(a["b"]),
            self.d_static["dt"], self.d_static["a"], dev(a["z"]), self.d_static["norm_w"],
            self.state, out, cfg.n_seqs, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size,
            cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps, slots=self.d_slots, pool=self.P,
            err_count=self.err)
        s = self.sample
        ref, skipped = oracle.block_decode(
            a["qkv"][s], self.static["conv_w"], self.ref_conv, a["alpha"][s], a["b"][s],
            self.static["dt"], self.static["a"], a["z"][s], self.static["norm_w"],
            self.ref_state, cfg.n_k_heads, cfg.scale, cfg.eps, cfg.eps)
        assert skipped == 0
        return host(out), ref


def check_block_chain(lib, cfg, sample, steps):
    """Chained fused-block steps: after the first step out, state and conv_state of the
    sampled sequences meet the one-step elementwise bound, after the last the long-chain
    RMS bound."""
    run = BlockRun(lib, cfg, sample)
    ids = [run.slot_of(n) for n in sample]
    for step in range(steps):
        out, ref = run.step(step)
        if step == 0:
            assert_step(out[sample], ref, "out, first step")
            assert_step(host(run.state[ids]), run.ref_state, "state, first step")
            assert_step(host(run.conv[ids]), run.ref_conv, "conv_state, first step")
    assert_rms(out[sample], ref, f"out after {steps} steps")
    assert_rms(host(run.state[ids]), run.ref_state, f"state after {steps} steps")
    assert_rms(host(run.conv[ids]), run.ref_conv, f"conv_state after {steps} steps")
    assert host(run.err)[0] == 0
    return run


def test_block_decode_tiny_chain(lib):
    """The tiny workload (N=1, Hk=2, H=4, S=32), 16 chained steps, every step checked."""
    cfg = I.get_config(0)
    run = BlockRun(lib, cfg, [0])
    for step in range(cfg.steps):
        out, ref = run.step(step)
        assert_step(out, ref, f"out step {step}")
    assert_step(host(run.state), run.ref_state, "state")
    assert_step(host(run.conv), run.ref_conv, "conv_state")


@pytest.mark.parametrize("Hk,H,S,N", [(1, 1, 64, 2), (2, 8, 128, 3), (4, 4, 256, 2),
                                      (1, 2, 32, 5), (2, 16, 128, 2)])  # GQA up to 8
def test_block_decode_shapes(lib, Hk, H, S, N):
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=S, n_seqs=N, cid=300 + S + H)
    check_block_chain(lib, cfg, list(range(N)), steps=3)


@pytest.mark.parametrize("Hk,H,S,N", [(16, 32, 128, 20), (8, 16, 64, 40), (16, 16, 128, 20),
                                      (4, 16, 128, 80), (2, 16, 128, 160)])  # GQA up to 8
def test_block_decode_persistent_shapes(lib, Hk, H, S, N):
    """At least two (sequence, k-head) groups per SM: the persistent form runs."""
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=S, n_seqs=N, cid=500 + S + H + N)
    check_block_chain(lib, cfg, [0, N // 2, N - 1], steps=3)


def test_block_decode_persistent_invalid_slot(lib):
    cfg = I.get_config(3, n_seqs=20, pool=24, cid=600)
    run = BlockRun(lib, cfg, [0])
    slots = np.arange(20, dtype=np.int32) + 2
    slots[7] = 99  # out of range: skipped, counted, untouched
    run.slots, run.d_slots = slots, dev(slots)
    a = I.block_step(cfg, 0)
    out = torch.full((20, cfg.n_v_heads, cfg.state_size), 5.0, device="cuda")
    lib.gdn_block_decode(dev(a["qkv"]), run.d_static["conv_w"], run.conv, dev(a["alpha"]),
                         dev(a["b"]), run.d_static["dt"], run.d_static["a"], dev(a["z"]),
                         run.d_static["norm_w"], run.state, out, 20, cfg.n_k_heads, cfg.n_v_heads,
                         cfg.state_size, 4, cfg.scale, cfg.eps, cfg.eps, slots=run.d_slots,
                         pool=24, err_count=run.err)
    assert host(run.err)[0] == 1
    o = host(out)
    assert np.all(o[7] == 5.0) and np.all(np.isfinite(o))
    st, cv = host(run.state), host(run.conv)
    for sl in (0, 1, 9):  # slot 9 belonged to the skipped sequence
        np.testing.assert_array_equal(st[sl], run.state0[sl])
        np.testing.assert_array_equal(cv[sl], run.conv0[sl])
    # a valid sequence matches the oracle
    ref_st = f64(run.state0[slots[3]:slots[3] + 1])
    ref_cv = f64(run.conv0[slots[3]:slots[3] + 1])
    ref, _ = oracle.block_decode(a["qkv"][3:4], run.static["conv_w"], ref_cv, a["alpha"][3:4],
                                 a["b"][3:4], run.static["dt"], run.static["a"], a["z"][3:4],
                                 run.static["norm_w"], ref_st, cfg.n_k_heads, cfg.scale, cfg.eps,
                                 cfg.eps)
    assert_step(o[3:4], ref, "out")
    assert_step(st[slots[3]:slots[3] + 1], ref_st, "state")


@pytest.mark.slow
def test_block_decode_single_seq_1000(lib):
    """Single-sequence decode at the verified shape, 1000 chained steps."""
    cfg = I.get_config(1)
    check_block_chain(lib, cfg, [0], steps=cfg.steps)


@pytest.mark.slow
def test_block_decode_batched_64(lib):
    """Batched decode, 64 sequences, 200 chained steps; sampled sequences checked."""
    cfg = I.get_config(3)
    check_block_chain(lib, cfg, [0, 37, 63], steps=cfg.steps)


@pytest.mark.slow
def test_block_decode_serving_pool(lib):
    """256 active slots of a 512-slot pool, 50 steps: sampled active slots match the
    oracle and every untouched slot keeps its bits."""
    cfg = I.get_config(4)
    run = check_block_chain(lib, cfg, [0, 101, 255], steps=cfg.steps)
    active = set(int(s) for s in run.slots)
    untouched = torch.tensor(sorted(set(range(cfg.pool_size)) - active), device="cuda")
    init_state = dev(run.state0)
    init_conv = dev(run.conv0)
    assert torch.equal(run.state.index_select(0, untouched), init_state.index_select(0, untouched))
    assert torch.equal(run.conv.index_select(0, untouched), init_conv.index_select(0, untouched))


def test_block_decode_invalid_slot(lib):
    cfg = I.get_config(0, n_seqs=3, pool=4, cid=400)
    run = BlockRun(lib, cfg, [0])
    run.slots = np.array([2, 9, 0], dtype=np.int32)
    run.d_slots = dev(run.slots)
    a = I.block_step(cfg, 0)
    out = torch.full((3, cfg.n_v_heads, cfg.state_size), 5.0, device="cuda")
    lib.gdn_block_decode(dev(a["qkv"]), run.d_static["conv_w"], run.conv, dev(a["alpha"]),
                         dev(a["b"]), run.d_static["dt"], run.d_static["a"], dev(a["z"]),
                         run.d_static["norm_w"], run.state, out, 3, cfg.n_k_heads, cfg.n_v_heads,
                         cfg.state_size, 4, cfg.scale, cfg.eps, cfg.eps, slots=run.d_slots,
                         pool=4, err_count=run.err)
    assert host(run.err)[0] == 1
    assert np.all(host(out)[1] == 5.0)
    np.testing.assert_array_equal(host(run.state)[[1, 3]], run.state0[[1, 3]])
    np.testing.assert_array_equal(host(run.conv)[[1, 3]], run.conv0[[1, 3]])


def test_block_equals_unfused_pipeline(lib):
    """With a whole head per CTA (64 sequences), the fused block and the chain of
    standalone kernels give the same bits."""
    cfg = I.get_config(3)
    N, Hk, H, S, C = cfg.n_seqs, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size, cfg.conv_dim
    st = I.block_static(cfg)
    a = I.block_step(cfg, 0)
    state0 = dev(np.random.default_rng(5).normal(0, 0.1, (N, H, S, S)).astype(np.float32))
    conv0 = dev(np.random.default_rng(6).normal(0, 1, (N, C, 3)).astype(np.float32))
    d = {k: dev(v) for k, v in {**st, **a}.items()}
    # fused
    st_f, cv_f = state0.clone(), conv0.clone()
    out_f = torch.empty(N, H, S, device="cuda")
    lib.gdn_block_decode(d["qkv"], d["conv_w"], cv_f, d["alpha"], d["b"], d["dt"], d["a"], d["z"],
                         d["norm_w"], st_f, out_f, N, Hk, H, S, 4, cfg.scale, cfg.eps, cfg.eps)
    # unfused
    st_u, cv_u = state0.clone(), conv0.clone()
    conv_out = torch.empty(N, C, device="cuda")
    lib.gdn_conv1d_silu(d["qkv"], d["conv_w"], cv_u, conv_out, N, C, 4)
    q = torch.empty(N, Hk, S, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty(N, H, S, device="cuda")
    lib.gdn_qkv_split_norm(conv_out, q, k, v, N, Hk, H, S, cfg.eps)
    g = torch.empty(N, H, device="cuda")
    lib.gdn_decay_gate(d["alpha"], d["dt"], d["a"], g, H, N)
    beta = torch.empty(N, H, device="cuda")
    lib.gdn_beta_sigmoid(d["b"], beta, N * H)
    y = torch.empty(N, H, S, device="cuda")
    lib.gdn_recurrence_decode(st_u, q, k, v, g, beta, y, N, Hk, H, S, cfg.scale)
    out_u = torch.empty_like(y)
    lib.gdn_gated_norm(y, d["norm_w"], d["z"], out_u, N * H, S, cfg.eps)
    torch.cuda.synchronize()
    assert torch.equal(cv_f, cv_u)
    assert torch.equal(st_f, st_u)
    assert torch.equal(out_f, out_u)


# ------------------------------------------------------------------ prefill block

def run_prefill(lib, cfg, T, seqs_in, state, conv, slots=None, pool=None, err=None, out=None):
    N, H, S = len(seqs_in[0]["qkv"]), cfg.n_v_heads, cfg.state_size
    st = I.block_static(cfg)
    stack = {key: np.stack([a[key] for a in seqs_in], axis=1) for key in ("qkv", "alpha", "b", "z")}
    out = torch.zeros(N, T, H, S, device="cuda") if out is None else out
    nbytes = lib.gdn_block_prefill_workspace_size(N, T, cfg.n_k_heads, H, S)
    ws = torch.empty(nbytes // 4, device="cuda")
    lib.gdn_block_prefill(dev(stack["qkv"]), dev(st["conv_w"]), conv, dev(stack["alpha"]),
                          dev(stack["b"]), dev(st["dt"]), dev(st["a"]), dev(stack["z"]),
                          dev(st["norm_w"]), state, out, N, T, cfg.n_k_heads, H, S,
                          cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps, ws, slots=slots,
                          pool=pool, err_count=err)
    return out, stack


@pytest.mark.parametrize("Hk,H,S,N,T", [(2, 4, 32, 1, 16), (2, 4, 128, 2, 37), (16, 32, 128, 3, 20)])
def test_block_prefill(lib, Hk, H, S, N, T):
    """The prefill block equals T single-token steps of the block (oracle), and the
    GPU's own T decode calls, within the stated bounds."""
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=S, n_seqs=N, cid=700 + S + T)
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    state, conv = dev(st0), dev(cs0)
    out, stack = run_prefill(lib, cfg, T, steps, state, conv)
    got = host(out)
    stat = I.block_static(cfg)
    ref_st, ref_cs = f64(st0), f64(cs0)
    ref = np.zeros(got.shape)
    for t in range(T):
        a = steps[t]
        ref[:, t], _ = oracle.block_decode(a["qkv"], stat["conv_w"], ref_cs, a["alpha"], a["b"],
                                           stat["dt"], stat["a"], a["z"], stat["norm_w"], ref_st,
                                           cfg.n_k_heads, cfg.scale, cfg.eps, cfg.eps)
    assert_step(got[:, 0], ref[:, 0], "out token 0")
    assert_rms(got, ref, "out")
    assert_rms(host(state), ref_st, "state")
    assert_rms(host(conv), ref_cs, "conv_state")
    # against T calls of the GPU's fused decode
    st_d, cs_d = dev(st0), dev(cs0)
    dd = {k_: dev(v_) for k_, v_ in stat.items()}
    for t in range(T):
        a = steps[t]
        o = torch.empty(N, H, S, device="cuda")
        lib.gdn_block_decode(dev(a["qkv"]), dd["conv_w"], cs_d, dev(a["alpha"]), dev(a["b"]),
                             dd["dt"], dd["a"], dev(a["z"]), dd["norm_w"], st_d, o, N, Hk, H, S,
                             4, cfg.scale, cfg.eps, cfg.eps)
        assert_step(got[:, t], host(o), f"prefill vs decode, token {t}")


def test_block_prefill_snapshots(lib):
    """The prefill block keeping snapshots: out, state and conv history are gdn_block_prefill's
    bit for bit; snaps[t] and conv_snaps[t] are the state and conv history the block leaves
    after the first t + 1 positions (bit for bit); slots route; gdn_snapshot_restore then
    rolls every sequence back to its own accepted count."""
    cfg = I.get_config(0, n_k_heads=2, n_v_heads=4, state_size=128, n_seqs=3, pool=5, cid=905)
    N, Hk, H, S, K, T = 3, 2, 4, 128, cfg.conv_kernel, 7
    C = (2 * Hk + H) * S
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    slots = dev(np.array([4, 0, 2], dtype=np.int32))
    # without snapshots
    state_r, conv_r = dev(st0), dev(cs0)
    out_r, stack = run_prefill(lib, cfg, T, steps, state_r, conv_r, slots=slots, pool=5)
    # with them
    stat = {k_: dev(v_) for k_, v_ in I.block_static(cfg).items()}
    state, conv = dev(st0), dev(cs0)
    out = torch.zeros(N, T, H, S, device="cuda")
    snaps = torch.zeros(N, T, H, S, S, device="cuda")
    csnaps = torch.zeros(N, T, C, K - 1, device="cuda")
    ws = torch.empty(lib.gdn_block_prefill_workspace_size(N, T, Hk, H, S) // 4, device="cuda")
    lib.gdn_block_prefill_snapshots(dev(stack["qkv"]), stat["conv_w"], conv, dev(stack["alpha"]),
                                    dev(stack["b"]), stat["dt"], stat["a"], dev(stack["z"]),
                                    stat["norm_w"], state, out, snaps, csnaps, N, T, Hk, H, S, K,
                                    cfg.scale, cfg.eps, cfg.eps, ws, slots=slots, pool=5)
    assert torch.equal(out, out_r) and torch.equal(state, state_r) and torch.equal(conv, conv_r)
    sl = [4, 0, 2]
    for t in range(T):
        st_p, cs_p = dev(st0), dev(cs0)
        run_prefill(lib, cfg, t + 1, steps[:t + 1], st_p, cs_p, slots=slots, pool=5)
        for n in range(N):
            assert torch.equal(snaps[n, t], st_p[sl[n]]), f"state snapshot {t}, sequence {n}"
            assert torch.equal(csnaps[n, t], cs_p[sl[n]]), f"conv snapshot {t}, sequence {n}"
    accepted = np.array([2, T, 5], dtype=np.int32)
    lib.gdn_snapshot_restore(state, snaps, dev(accepted), N, T, H, S, conv_state=conv,
                             conv_snaps=csnaps, conv_dim=C, conv_kernel=K, slots=slots, pool=5)
    for n in range(N):
        assert torch.equal(state[sl[n]], snaps[n, accepted[n] - 1])
        assert torch.equal(conv[sl[n]], csnaps[n, accepted[n] - 1])
    for s_ in (1, 3):  # slots no sequence uses
        np.testing.assert_array_equal(host(state)[s_], st0[s_])
        np.testing.assert_array_equal(host(conv)[s_], cs0[s_])


def test_block_prefill_invalid_slot(lib):
    cfg = I.get_config(0, n_seqs=3, pool=4, cid=800)
    T = 12
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    state, conv = dev(st0), dev(cs0)
    slots = np.array([3, 6, 0], dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((3, T, cfg.n_v_heads, cfg.state_size), 9.0, device="cuda")
    run_prefill(lib, cfg, T, steps, state, conv, slots=dev(slots), pool=4, err=err, out=out)
    assert host(err)[0] == 1
    o = host(out)
    assert np.all(o[1] == 9.0) and np.all(np.isfinite(o))
    for sl in (1, 2):
        np.testing.assert_array_equal(host(state)[sl], st0[sl])
        np.testing.assert_array_equal(host(conv)[sl], cs0[sl])


@pytest.mark.slow
def test_block_prefill_4_sequences_512_tokens(lib):
    """Full-width heads (Hk=16, H=32, S=128), 4 sequences x 512 tokens; one sampled
    sequence checked against the oracle."""
    cfg = I.get_config(2)
    T = 512
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    state, conv = dev(st0), dev(cs0)
    out, _ = run_prefill(lib, cfg, T, steps, state, conv)
    got = host(out)
    stat = I.block_static(cfg)
    n = 2
    ref_st, ref_cs = f64(st0[n:n + 1]), f64(cs0[n:n + 1])
    ref = np.zeros((T,) + got.shape[2:])
    for t in range(T):
        a = steps[t]
        r, _ = oracle.block_decode(a["qkv"][n:n + 1], stat["conv_w"], ref_cs, a["alpha"][n:n + 1],
                                   a["b"][n:n + 1], stat["dt"], stat["a"], a["z"][n:n + 1],
                                   stat["norm_w"], ref_st, cfg.n_k_heads, cfg.scale, cfg.eps,
                                   cfg.eps)
        ref[t] = r[0]
    assert_step(got[n, 0], ref[0], "out token 0")
    assert_rms(got[n], ref, "out")
    assert_rms(host(state)[n], ref_st[0], "state")
