"""GPU parity of the two-phase chunked scan (gdn_recurrence_scan_chunked_ws and its
phases, gdn_chunked_prepare / gdn_chunked_advance).

It runs the arithmetic of the one-kernel chunked scan in the same order, so its y and
final state must equal that form's bit for bit, whatever the workspace size (one
wave, or waves of 1 and 3 chunks with the state passing through its fp32 home in
between) and however the phases are called. It is also held directly to the oracle's
long-scan bound (max |gpu - ref| <= 2e-3 * RMS(ref) per tensor), including at the full
4 x 4096 prefill size on sampled units.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402
from tests.oracle_units import prefill_4x4096  # noqa: E402

pytestmark = pytest.mark.gpu

BLK = 36 * 1024  # workspace bytes per (chunk, sequence, v-head)


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


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
    cuda_lib.gdn_device_error()  # raises if a bounded wait gave up during the module


def case(Hk, H, N, T, seed, pool=None):
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=128, n_seqs=N, n_tokens=T,
                       pool=pool, cid=700 + seed)
    return cfg, I.recurrence_batch(cfg), I.state_pool(cfg)


def run(lib, cfg, x, st, form, ws_chunks=None, slots=None, pool=None, err=None):
    """form 'fused' (one kernel) or 'ws' (two phases; ws_chunks = chunks per wave, None =
    the whole call in one wave)."""
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    y = torch.zeros(N, T, H, S, device="cuda")
    args = (st, dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["g"]), dev(x["beta"]), y, N, T,
            cfg.n_k_heads, H, S, cfg.scale)
    if form == "fused":
        lib.gdn_recurrence_scan_chunked(*args, slots=slots, pool=pool, err_count=err)
    else:
        nbytes = (lib.gdn_recurrence_scan_chunked_ws_size(N, T, H, S) if ws_chunks is None
                  else ws_chunks * N * H * BLK)
        ws = torch.full((nbytes // 4,), float("nan"), device="cuda")  # contents must not matter
        lib.gdn_recurrence_scan_chunked_ws(*args, ws, slots=slots, pool=pool, err_count=err)
    return y


# GQA ratios 1, 2, 3, 4 and 5 (odd ratios reuse the two v-row buffers of the chunk
# preparation unevenly), single positions, ragged and exact chunk ends
CASES = [(2, 4, 2, 1), (2, 4, 2, 31), (1, 2, 1, 32), (2, 4, 1, 33), (2, 4, 2, 100),
         (4, 4, 1, 64), (2, 8, 2, 200), (1, 1, 3, 97), (1, 3, 2, 70), (2, 10, 1, 45)]


@pytest.mark.parametrize("Hk,H,N,T", CASES)
def test_ws_equals_one_kernel_form(lib, Hk, H, N, T):
    cfg, x, st0 = case(Hk, H, N, T, seed=T + 3 * H)
    st_f, st_w = dev(st0), dev(st0)
    y_f = run(lib, cfg, x, st_f, "fused")
    y_w = run(lib, cfg, x, st_w, "ws")
    assert torch.equal(y_w, y_f)
    assert torch.equal(st_w, st_f)


@pytest.mark.parametrize("chunks", [1, 3])
def test_ws_waves_equal_one_wave(lib, chunks):
    cfg, x, st0 = case(2, 4, 2, 230, seed=41)
    st_1, st_w = dev(st0), dev(st0)
    y_1 = run(lib, cfg, x, st_1, "ws")
    y_w = run(lib, cfg, x, st_w, "ws", ws_chunks=chunks)
    assert torch.equal(y_w, y_1)
    assert torch.equal(st_w, st_1)


@pytest.mark.parametrize("Hk,H,N,T", [(2, 4, 2, 75), (2, 8, 1, 160)])
def test_ws_vs_oracle(lib, Hk, H, N, T):
    cfg, x, st0 = case(Hk, H, N, T, seed=11 + T)
    st = dev(st0)
    y = run(lib, cfg, x, st, "ws", ws_chunks=2)
    st_ref = np.array(st0, dtype=np.float64)
    y_ref, _ = oracle.recurrence(st_ref, x["q"], x["k"], x["v"], x["g"], x["beta"], cfg.scale)
    yh = host(y)
    assert_rms(yh, y_ref, "y")
    assert_rms(host(st), st_ref, "final state")
    for n in range(N):
        for vh in range(H):
            assert_rms(yh[n, :, vh], y_ref[n, :, vh], f"y ({n},{vh})")


def test_ws_slots_counted_once(lib):
    """A skipped sequence is counted once however many waves run; untouched slots keep
    their bits; routed slots equal the one-kernel form's."""
    cfg, x, _ = case(2, 4, 3, 70, seed=9, pool=5)
    pool0 = I.state_pool(cfg)
    slots = dev(np.array([4, -1, 1], dtype=np.int32))
    st_w, st_f = dev(pool0), dev(pool0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_w = run(lib, cfg, x, st_w, "ws", ws_chunks=1, slots=slots, pool=5, err=err)
    y_f = run(lib, cfg, x, st_f, "fused", slots=slots, pool=5)
    assert host(err)[0] == 1
    got = host(st_w)
    for s in (0, 2, 3):
        np.testing.assert_array_equal(got[s], pool0[s])
    assert torch.equal(st_w, st_f)
    assert torch.equal(y_w, y_f)
    assert np.all(host(y_w)[1] == 0.0)


@pytest.mark.slow
def test_ws_prefill_4x4096(lib):
    """The prefill workload at full size: bit for bit the one-kernel form, in one wave
    and in waves of 16 chunks; every (sequence, v-head) unit against the oracle."""
    cfg = I.get_config(2)
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    x = I.recurrence_batch(cfg)
    st0 = I.state_pool(cfg)
    st_w, st_f, st_v = dev(st0), dev(st0), dev(st0)
    y_w = run(lib, cfg, x, st_w, "ws")
    y_f = run(lib, cfg, x, st_f, "fused")
    assert torch.equal(y_w, y_f)
    assert torch.equal(st_w, st_f)
    y_v = run(lib, cfg, x, st_v, "ws", ws_chunks=16)
    assert torch.equal(y_v, y_w)
    assert torch.equal(st_v, st_w)
    del y_f, y_v
    yh, sth = host(y_w), host(st_w)
    _, _, _, refs = prefill_4x4096()
    assert len(refs) == N * H
    for (n, vh), (y_ref, s_ref) in refs.items():  # every unit against the oracle
        assert_rms(yh[n, :, vh], y_ref, f"y ({n},{vh})")
        assert_rms(sth[n, vh], s_ref, f"final state ({n},{vh})")


def test_phases_equal_one_call(lib):
    """gdn_chunked_prepare / gdn_chunked_advance over consecutive ranges of 2 chunks,
    with slot routing and a skipped sequence: the bits of the one-kernel form, the
    skipped sequence counted once."""
    cfg, x, _ = case(2, 4, 3, 230, seed=57, pool=6)
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    pool0 = I.state_pool(cfg)
    slots = dev(np.array([5, -1, 2], dtype=np.int32))
    st_p, st_f = dev(pool0), dev(pool0)
    y_f = run(lib, cfg, x, st_f, "fused", slots=slots, pool=6)
    d = {key: dev(x[key]) for key in ("q", "k", "v", "g", "beta")}
    y_p = torch.zeros(N, T, H, S, device="cuda")
    ws = torch.full((2 * N * H * BLK // 4,), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_chunks = (T + 31) // 32
    for cb in range(0, n_chunks, 2):
        nc = min(2, n_chunks - cb)
        lib.gdn_chunked_prepare(d["q"], d["k"], d["v"], d["g"], d["beta"], ws, N, T,
                                cfg.n_k_heads, H, S, cb, nc)
        lib.gdn_chunked_advance(st_p, d["q"], d["k"], d["g"], ws, y_p, N, T, cfg.n_k_heads, H,
                                S, cfg.scale, cb, nc, slots=slots, pool=6, err_count=err)
    assert host(err)[0] == 1
    assert torch.equal(st_p, st_f)
    assert torch.equal(y_p, y_f)
