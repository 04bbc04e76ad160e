"""GPU parity of the chunked tensor-core scan (gdn_recurrence_scan_chunked).

The chunked form regroups the recurrence exactly, so it is held to the oracle's
long-scan bound: max |gpu - ref| <= 2e-3 * RMS(ref) for y and for the final
state, per tensor (ref = the fp64 oracle). Cases cover one position, a chunk
minus one, exactly one chunk, one more, several chunks with a ragged tail, GQA
ratios 1, 2 and 4, slot routing with a skipped sequence, and the 4 x 4096 prefill
workload at full size; then the prefill block built on it (gdn_block_prefill_chunked)
against the oracle's block steps and against the sequential-scan prefill block.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402
from tests.oracle_units import prefill_4x4096  # noqa: E402

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def f64(x):
    return np.array(x, dtype=np.float64)


def assert_rms(gpu, ref, name, rel=2e-3):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    rms = np.sqrt(np.mean(ref * ref))
    err = np.max(np.abs(gpu - ref))
    assert err <= rel * rms, f"{name}: max err {err:.3e} > {rel} * RMS {rms:.3e}"
    return err / rms


@pytest.fixture(scope="module", autouse=True)
def lib(cuda_lib):
    yield cuda_lib
    cuda_lib.gdn_device_error()  # raises if a bounded wait gave up during the module


def case(Hk, H, N, T, seed, pool=None):
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=128, n_seqs=N, n_tokens=T,
                       pool=pool, cid=300 + seed)
    return cfg, I.recurrence_batch(cfg), I.state_pool(cfg)


def run_chunked(lib, cfg, x, st, slots=None, pool=None, err=None):
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    y = torch.zeros(N, T, H, S, device="cuda")
    lib.gdn_recurrence_scan_chunked(st, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]),
                                    dev(x["beta"]), y, N, T, cfg.n_k_heads, H, S, cfg.scale,
                                    slots=slots, pool=pool, err_count=err)
    return y


@pytest.mark.parametrize("Hk,H,N,T", [(2, 4, 2, 1), (2, 4, 2, 31), (1, 2, 1, 32), (2, 4, 1, 33),
                                      (2, 4, 2, 100), (4, 4, 1, 64), (2, 8, 2, 200)])
def test_chunked_scan_vs_oracle(lib, Hk, H, N, T):
    cfg, x, st0 = case(Hk, H, N, T, seed=T + H)
    st = dev(st0)
    y = run_chunked(lib, cfg, x, st)
    st_ref = f64(st0)
    y_ref, _ = oracle.recurrence(st_ref, x["q"], x["k"], x["v"], x["g"], x["beta"], cfg.scale)
    assert_rms(host(y), y_ref, "y")
    assert_rms(host(st), st_ref, "final state")
    # each (sequence, v-head) unit on its own scale, too
    yh = host(y)
    for n in range(N):
        for vh in range(H):
            assert_rms(yh[n, :, vh], y_ref[n, :, vh], f"y ({n},{vh})")


def test_chunked_scan_matches_sequential_scan(lib):
    """Against the library's sequential scan (itself bit-identical to decode steps)."""
    cfg, x, st0 = case(2, 4, 2, 160, seed=5)
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    st_c, st_s = dev(st0), dev(st0)
    y_c = run_chunked(lib, cfg, x, st_c)
    y_s = torch.zeros(N, T, H, S, device="cuda")
    lib.gdn_recurrence_scan(st_s, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]),
                            dev(x["beta"]), y_s, N, T, cfg.n_k_heads, H, S, cfg.scale)
    assert_rms(host(y_c), host(y_s), "y vs sequential")
    assert_rms(host(st_c), host(st_s), "state vs sequential")


def test_chunked_scan_slots(lib):
    cfg, x, _ = case(2, 4, 3, 70, seed=9, pool=5)
    pool0 = I.state_pool(cfg)
    slots = np.array([4, -1, 1], dtype=np.int32)
    st = dev(pool0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = run_chunked(lib, cfg, x, st, slots=dev(slots), pool=5, err=err)
    assert host(err)[0] == 1
    st_ref = f64(pool0)
    y_ref, skipped = oracle.recurrence(st_ref, x["q"], x["k"], x["v"], x["g"], x["beta"],
                                       cfg.scale, slots=slots, pool=5)
    assert skipped == 1
    got = host(st)
    for s in (0, 2, 3):
        np.testing.assert_array_equal(got[s], pool0[s])  # untouched slots keep their bits
    for s in (1, 4):
        assert_rms(got[s], st_ref[s], f"state slot {s}")
    yh = host(y)
    assert np.all(yh[1] == 0.0)  # nothing written for the skipped sequence
    assert_rms(yh[[0, 2]], y_ref[[0, 2]], "y")


@pytest.mark.slow
def test_chunked_scan_prefill_4x4096(lib):
    """The prefill workload at full size (N=4, T=4096, Hk=16, H=32, S=128): every
    output against the sequential GPU scan and every (sequence, v-head) unit against
    the oracle, under the long-scan bound."""
    cfg = I.get_config(2)
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    x = I.recurrence_batch(cfg)
    st0 = I.state_pool(cfg)
    st_c, st_s = dev(st0), dev(st0)
    y_c = run_chunked(lib, cfg, x, st_c)
    y_s = torch.zeros(N, T, H, S, device="cuda")
    lib.gdn_recurrence_scan(st_s, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]),
                            dev(x["beta"]), y_s, N, T, cfg.n_k_heads, H, S, cfg.scale)
    yh, sth = host(y_c), host(st_c)
    assert_rms(yh, host(y_s), "y vs sequential")
    assert_rms(sth, host(st_s), "state vs sequential")
    _, _, _, refs = prefill_4x4096()
    assert len(refs) == N * H
    for (n, vh), (y_ref, s_ref) in refs.items():  # every unit against the oracle
        assert_rms(yh[n, :, vh], y_ref, f"y ({n},{vh})")
        assert_rms(sth[n, vh], s_ref, f"final state ({n},{vh})")


# ------------------------------------------------------------------ prefill block

def run_block_prefill(lib, cfg, T, steps, state, conv, chunked, slots=None, pool=None,
                      err=None, ws_bytes=None):
    """ws_bytes: the workspace size (None = the minimum, gdn_block_prefill_workspace_size)."""
    N, H, S = len(steps[0]["qkv"]), cfg.n_v_heads, cfg.state_size
    st = I.block_static(cfg)
    stack = {key: np.stack([a[key] for a in steps], axis=1) for key in ("qkv", "alpha", "b", "z")}
    out = torch.zeros(N, T, H, S, device="cuda")
    if ws_bytes is None:
        ws_bytes = lib.gdn_block_prefill_workspace_size(N, T, cfg.n_k_heads, H, S)
    ws = torch.full(((ws_bytes + 3) // 4,), float("nan"), device="cuda")
    fn = lib.gdn_block_prefill_chunked if chunked else lib.gdn_block_prefill
    fn(dev(stack["qkv"]), dev(st["conv_w"]), conv, dev(stack["alpha"]), dev(stack["b"]),
       dev(st["dt"]), dev(st["a"]), dev(stack["z"]), dev(st["norm_w"]), state, out, N, T,
       cfg.n_k_heads, H, S, cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps, ws, slots=slots,
       pool=pool, err_count=err)
    return out


def oracle_block_chain(cfg, steps, st0, cs0, seqs):
    stat = I.block_static(cfg)
    ref_st, ref_cs = f64(st0[seqs]), f64(cs0[seqs])
    outs = []
    for a in steps:
        r, _ = oracle.block_decode(a["qkv"][seqs], stat["conv_w"], ref_cs, a["alpha"][seqs],
                                   a["b"][seqs], stat["dt"], stat["a"], a["z"][seqs],
                                   stat["norm_w"], ref_st, cfg.n_k_heads, cfg.scale, cfg.eps,
                                   cfg.eps)
        outs.append(r)
    return np.stack(outs, axis=1), ref_st, ref_cs


@pytest.mark.parametrize("Hk,H,N,T", [(2, 4, 2, 45), (16, 32, 2, 70)])
def test_block_prefill_chunked(lib, Hk, H, N, T):
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=128, n_seqs=N, cid=900 + T)
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    state, conv = dev(st0), dev(cs0)
    out = run_block_prefill(lib, cfg, T, steps, state, conv, chunked=True)
    ref, ref_st, ref_cs = oracle_block_chain(cfg, steps, st0, cs0, list(range(N)))
    assert_rms(host(out), ref, "out")
    assert_rms(host(state), ref_st, "state")
    assert_rms(host(conv), ref_cs, "conv_state")
    # against the sequential-scan prefill block
    state2, conv2 = dev(st0), dev(cs0)
    out2 = run_block_prefill(lib, cfg, T, steps, state2, conv2, chunked=False)
    assert_rms(host(out), host(out2), "out vs sequential prefill")
    assert torch.equal(conv, conv2)  # the conv scan is shared: bit for bit


def test_block_prefill_chunked_two_phase_workspace(lib):
    """A workspace with room for the two-phase scan (all chunks, or 3 at a time) gives
    the bits of the minimum workspace (the one-kernel scan)."""
    cfg = I.get_config(0, n_k_heads=2, n_v_heads=4, state_size=128, n_seqs=2, cid=960)
    T = 150
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    N, H, S = 2, cfg.n_v_heads, cfg.state_size
    base = lib.gdn_block_prefill_workspace_size(N, T, cfg.n_k_heads, H, S)
    full = lib.gdn_block_prefill_chunked_workspace_size(N, T, cfg.n_k_heads, H, S)
    assert full > base
    results = []
    for nbytes in (base, full, (base + 15) // 16 * 16 + 3 * N * H * 36 * 1024):
        state, conv = dev(st0), dev(cs0)
        out = run_block_prefill(lib, cfg, T, steps, state, conv, chunked=True, ws_bytes=nbytes)
        results.append((out, state, conv))
    for out, state, conv in results[1:]:
        assert torch.equal(out, results[0][0])
        assert torch.equal(state, results[0][1])
        assert torch.equal(conv, results[0][2])


def test_block_prefill_chunked_invalid_slot(lib):
    cfg = I.get_config(0, n_k_heads=2, n_v_heads=4, state_size=128, n_seqs=3, pool=4, cid=950)
    T = 40
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    state, conv = dev(st0), dev(cs0)
    slots = np.array([3, 6, 0], dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_block_prefill(lib, cfg, T, steps, state, conv, chunked=True, slots=dev(slots),
                            pool=4, err=err)
    assert host(err)[0] == 1
    assert np.all(host(out)[1] == 0.0)
    for sl in (1, 2):
        np.testing.assert_array_equal(host(state)[sl], st0[sl])
        np.testing.assert_array_equal(host(conv)[sl], cs0[sl])


@pytest.mark.slow
def test_block_prefill_chunked_4_sequences_512_tokens(lib):
    """Full-width heads (Hk=16, H=32, S=128), 4 sequences x 512 tokens; one sampled
    sequence against the oracle, all of them against the sequential-scan block."""
    cfg = I.get_config(2)
    T = 512
    steps = [I.block_step(cfg, t) for t in range(T)]
    st0, cs0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    state, conv = dev(st0), dev(cs0)
    out = run_block_prefill(lib, cfg, T, steps, state, conv, chunked=True)
    got = host(out)
    n = 1
    ref, ref_st, _ = oracle_block_chain(cfg, steps, st0, cs0, [n])
    assert_rms(got[n], ref[0], "out")
    assert_rms(host(state)[n], ref_st[0], "state")
    state2, conv2 = dev(st0), dev(cs0)
    out2 = run_block_prefill(lib, cfg, T, steps, state2, conv2, chunked=False)
    assert_rms(got, host(out2), "out vs sequential prefill")
    assert_rms(host(state), host(state2), "state vs sequential prefill")
