"""GPU parity of the chunked scan's snapshot form (gdn_recurrence_scan_chunked_snapshots).

The snapshots subsample what the per-position snapshot scan writes (the whole state
after a position's update) at every 32 * snap_every positions. Checks:
- y and the final state are the bits of gdn_recurrence_scan_chunked_ws (the
  snapshots only add stores), in one wave and in waves of 1 and 3 chunks;
- snapshot j is within the long-scan bound (max |gpu - ref| <= 2e-3 * RMS(ref)) of
  the oracle's state after position (j + 1) * 32 * snap_every - 1, for every
  (sequence, v-head) unit;
- a call that ends on a snapshot interval writes the final state there, bit for bit;
- a scan continued from snapshot j over the remaining positions gives the full call's
  later y and final state bit for bit (the snapshot is the state the scan carries);
- snapshots are indexed by call order; a skipped sequence's snapshots are untouched.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu

BLK = 36 * 1024  # workspace bytes per (chunk, sequence, v-head)
C = 32           # positions per chunk


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
                       pool=pool, cid=900 + seed)
    return cfg, I.recurrence_batch(cfg), I.state_pool(cfg)


def inputs(x, t0=0):
    """The device inputs of positions t0.. of every sequence (contiguous copies)."""
    return [dev(x[key][:, t0:]) for key in ("q", "k", "v", "g", "beta")]


def workspace(lib, N, T, H, ws_chunks):
    nbytes = (lib.gdn_recurrence_scan_chunked_ws_size(N, T, H, 128) if ws_chunks is None
              else ws_chunks * N * H * BLK)
    return torch.full((nbytes // 4,), float("nan"), device="cuda")  # contents must not matter


def run_snap(lib, cfg, d, st, every, ws_chunks=None, slots=None, pool=None, err=None, T=None):
    N, H, S = cfg.n_seqs, cfg.n_v_heads, cfg.state_size
    T = cfg.n_tokens if T is None else T
    n_snaps = lib.gdn_chunked_snapshot_count(T, every)
    y = torch.zeros(N, T, H, S, device="cuda")
    snaps = (torch.full((N, n_snaps, H, S, S), float("nan"), device="cuda") if n_snaps
             else None)
    lib.gdn_recurrence_scan_chunked_snapshots(
        st, *d, y, snaps, every, N, T, cfg.n_k_heads, H, S, cfg.scale,
        workspace(lib, N, T, H, ws_chunks), slots=slots, pool=pool, err_count=err)
    return y, snaps


def run_plain(lib, cfg, d, st, ws_chunks=None, slots=None, pool=None, T=None):
    N, H, S = cfg.n_seqs, cfg.n_v_heads, cfg.state_size
    T = cfg.n_tokens if T is None else T
    y = torch.zeros(N, T, H, S, device="cuda")
    lib.gdn_recurrence_scan_chunked_ws(st, *d, y, N, T, cfg.n_k_heads, H, S, cfg.scale,
                                       workspace(lib, N, T, H, ws_chunks), slots=slots,
                                       pool=pool)
    return y


def oracle_snapshots(cfg, x, st0, every):
    """The oracle's state after each snapshot position, [N][n_snaps][H][S][S]: the
    sequential recurrence run segment by segment on one state (the same steps as one
    run over the prefix)."""
    T = cfg.n_tokens
    n_snaps = T // (C * every)
    st = np.array(st0, dtype=np.float64)
    out = []
    t = 0
    for j in range(n_snaps):
        t1 = (j + 1) * C * every
        seg = {key: np.ascontiguousarray(x[key][:, t:t1]) for key in ("q", "k", "v", "g",
                                                                        "beta")}
        oracle.recurrence(st, seg["q"], seg["k"], seg["v"], seg["g"], seg["beta"], cfg.scale)
        out.append(st[: cfg.n_seqs].copy())
        t = t1
    return np.stack(out, axis=1) if out else np.zeros((cfg.n_seqs, 0))


# (Hk, H, N, T, snap_every): ragged tails, calls that end on an interval, intervals of
# 1 to 4 chunks, a call too short for any snapshot
CASES = [(2, 4, 2, 200, 1), (2, 4, 2, 256, 2), (1, 2, 1, 96, 3), (2, 8, 1, 100, 4),
         (1, 3, 2, 161, 1), (2, 4, 1, 31, 1)]


@pytest.mark.parametrize("Hk,H,N,T,every", CASES)
def test_snapshots_vs_oracle_and_plain(lib, Hk, H, N, T, every):
    cfg, x, st0 = case(Hk, H, N, T, seed=T + every)
    d = inputs(x)
    st_s, st_p = dev(st0), dev(st0)
    y_s, snaps = run_snap(lib, cfg, d, st_s, every)
    y_p = run_plain(lib, cfg, d, st_p)
    assert torch.equal(y_s, y_p)
    assert torch.equal(st_s, st_p)
    n_snaps = T // (C * every)
    assert lib.gdn_chunked_snapshot_count(T, every) == n_snaps
    if n_snaps == 0:
        assert snaps is None
        return
    ref = oracle_snapshots(cfg, x, st0, every)
    got = host(snaps)
    for n in range(N):
        for j in range(n_snaps):
            for vh in range(H):
                assert_rms(got[n, j, vh], ref[n, j, vh], f"snapshot ({n},{j},{vh})")
    if T % (C * every) == 0:  # the call ends on an interval: the last one is the final state
        assert torch.equal(snaps[:, -1], st_s[:N])


@pytest.mark.parametrize("chunks", [1, 3])
def test_snapshot_waves_equal_one_wave(lib, chunks):
    """Snapshots that fall on a wave's first chunk (read back from the state slot) and
    the final one of the last wave: the bits of the one-wave call."""
    cfg, x, st0 = case(2, 4, 2, 288, seed=5)
    d = inputs(x)
    st_1, st_w = dev(st0), dev(st0)
    y_1, s_1 = run_snap(lib, cfg, d, st_1, 3)
    y_w, s_w = run_snap(lib, cfg, d, st_w, 3, ws_chunks=chunks)
    assert s_1.shape[1] == 3
    assert torch.equal(y_w, y_1)
    assert torch.equal(st_w, st_1)
    assert torch.equal(s_w, s_1)


@pytest.mark.parametrize("j", [0, 2])
def test_continuation_from_a_snapshot(lib, j):
    """Restart from snapshot j over the remaining positions: the full call's later y
    and final state, bit for bit."""
    every = 2
    cfg, x, st0 = case(2, 4, 2, 230, seed=17)
    N, T, H = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads
    st = dev(st0)
    y, snaps = run_snap(lib, cfg, inputs(x), st, every)
    t0 = (j + 1) * C * every
    st_c = dev(st0)
    st_c[:N] = snaps[:, j]
    y_c = run_plain(lib, cfg, inputs(x, t0), st_c, T=T - t0)
    assert torch.equal(y_c, y[:, t0:])
    assert torch.equal(st_c, st)


def test_snapshots_follow_call_order_not_slots(lib):
    """With a slot map (one sequence skipped), sequence n's snapshots sit at n: those of
    the routed sequences equal the unrouted call's, the skipped one's stay untouched."""
    cfg, x, _ = case(2, 4, 3, 130, seed=29, pool=5)
    pool0 = I.state_pool(cfg)
    d = inputs(x)
    slots = dev(np.array([4, -1, 1], dtype=np.int32))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_r = dev(pool0)
    y_r, s_r = run_snap(lib, cfg, d, st_r, 1, slots=slots, pool=5, err=err)
    assert host(err)[0] == 1
    # the same sequences unrouted: slot n holds what slot slots[n] held
    st_u = dev(pool0[[4, 0, 1]])
    y_u, s_u = run_snap(lib, cfg, d, st_u, 1)
    for n in (0, 2):
        assert torch.equal(s_r[n], s_u[n])
        assert torch.equal(y_r[n], y_u[n])
    assert torch.isnan(s_r[1]).all()
    assert torch.equal(st_r[4], st_u[0]) and torch.equal(st_r[1], st_u[2])
    for s in (0, 2, 3):  # slots no sequence was routed to keep their bits
        np.testing.assert_array_equal(host(st_r)[s], pool0[s])


def offset16(shape):
    """A NaN-filled contiguous tensor whose data starts 16 bytes past a 32-byte boundary."""
    n = int(np.prod(shape))
    base = torch.full((n + 8,), float("nan"), device="cuda")
    view = base[4:4 + n].view(*shape)
    assert view.data_ptr() % 32 == 16
    return view


def test_sixteen_byte_aligned_buffers(lib):
    """State and snapshots at addresses that are 16- but not 32-byte aligned (the
    128-bit store path): the bits of the aligned call."""
    every = 1
    cfg, x, st0 = case(2, 4, 2, 128, seed=23)
    N, T, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads, cfg.state_size
    d = inputs(x)
    st_a = dev(st0)
    y_a, s_a = run_snap(lib, cfg, d, st_a, every)
    st_o = offset16(st0.shape)
    st_o.copy_(dev(st0))
    s_o = offset16((N, T // (C * every), H, S, S))
    y_o = torch.zeros(N, T, H, S, device="cuda")
    lib.gdn_recurrence_scan_chunked_snapshots(st_o, *d, y_o, s_o, every, N, T, cfg.n_k_heads,
                                              H, S, cfg.scale, workspace(lib, N, T, H, None))
    assert torch.equal(y_o, y_a)
    assert torch.equal(st_o, st_a)
    assert torch.equal(s_o, s_a)


def test_snapshot_validation(lib):
    cfg, x, st0 = case(2, 4, 1, 64, seed=3)
    d = inputs(x)
    st = dev(st0)
    y = torch.zeros(1, 64, 4, 128, device="cuda")
    ws = workspace(lib, 1, 64, 4, None)
    with pytest.raises(Exception, match="GDN_ERR_SHAPE"):
        lib.gdn_recurrence_scan_chunked_snapshots(st, *d, y, None, 0, 1, 64, 2, 4, 128,
                                                  cfg.scale, ws)
    with pytest.raises(Exception, match="GDN_ERR_NULL"):
        lib.gdn_recurrence_scan_chunked_snapshots(st, *d, y, None, 1, 1, 64, 2, 4, 128,
                                                  cfg.scale, ws)
    assert torch.equal(st, dev(st0))  # nothing ran


@pytest.mark.slow
def test_snapshots_prefill_4x4096(lib):
    """The prefill workload at full size with a snapshot every 16 chunks (512
    positions): y and state are the plain call's bits, the last snapshot is the final
    state, and a continuation from the middle snapshot reproduces the rest."""
    cfg = I.get_config(2)
    N, T, H = cfg.n_seqs, cfg.n_tokens, cfg.n_v_heads
    x = I.recurrence_batch(cfg)
    st0 = I.state_pool(cfg)
    every = 16
    st_s, st_p = dev(st0), dev(st0)
    y_s, snaps = run_snap(lib, cfg, inputs(x), st_s, every)
    y_p = run_plain(lib, cfg, inputs(x), st_p)
    assert torch.equal(y_s, y_p)
    assert torch.equal(st_s, st_p)
    del y_p, st_p
    assert snaps.shape[1] == T // (C * every)
    assert torch.equal(snaps[:, -1], st_s[:N])
    j = snaps.shape[1] // 2 - 1
    t0 = (j + 1) * C * every
    st_c = dev(st0)
    st_c[:N] = snaps[:, j]
    y_c = run_plain(lib, cfg, inputs(x, t0), st_c, T=T - t0)
    assert torch.equal(y_c, y_s[:, t0:])
    assert torch.equal(st_c, st_s)


# ------------------------------------------------------------------ ragged batches

class RaggedScan:
    """Sequences of the given lengths, each seeded on its own, packed position-major."""

    def __init__(self, lengths, Hk=2, H=4, seed=0, pool=None):
        self.lengths = list(lengths)
        self.n = len(lengths)
        self.cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=128, n_seqs=self.n,
                                n_tokens=max(lengths), pool=pool, cid=1300 + seed)
        self.per = [I.recurrence_batch(I.get_config(0, n_k_heads=Hk, n_v_heads=H,
                                                    state_size=128, n_seqs=1, n_tokens=L,
                                                    cid=1400 + 31 * seed + i))
                    for i, L in enumerate(lengths)]
        self.packed = {key: np.concatenate([p[key][0] for p in self.per])
                       for key in ("q", "k", "v", "g", "beta")}
        self.cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        self.total = int(self.cu[-1])
        self.st0 = I.state_pool(self.cfg)

    def run(self, lib, every, base, snap_pool, slots=None, pool=None, err=None, snaps=True):
        cfg, H, S = self.cfg, self.cfg.n_v_heads, 128
        st = dev(self.st0)
        y = torch.zeros(self.total, H, S, device="cuda")
        sn = (torch.full((snap_pool, H, S, S), float("nan"), device="cuda")
              if snaps else None)
        ws = torch.empty(lib.gdn_recurrence_scan_chunked_varlen_ws_size(
            self.n, self.total, H, S) // 4, device="cuda")
        d = [dev(self.packed[key]) for key in ("q", "k", "v", "g", "beta")]
        lib.gdn_recurrence_scan_chunked_snapshots_varlen(
            st, *d, y, sn, None if base is None else dev(np.asarray(base, np.int32)), snap_pool,
            every, dev(self.cu), self.n, self.total, max(self.lengths), cfg.n_k_heads, H, S,
            cfg.scale, ws, slots=slots, pool=pool, err_count=err)
        return y, st, sn

    def run_plain(self, lib, slots=None, pool=None):
        cfg, H, S = self.cfg, self.cfg.n_v_heads, 128
        st = dev(self.st0)
        y = torch.zeros(self.total, H, S, device="cuda")
        ws = torch.empty(lib.gdn_recurrence_scan_chunked_varlen_ws_size(
            self.n, self.total, H, S) // 4, device="cuda")
        d = [dev(self.packed[key]) for key in ("q", "k", "v", "g", "beta")]
        lib.gdn_recurrence_scan_chunked_varlen(st, *d, y, dev(self.cu), self.n, self.total,
                                               max(self.lengths), cfg.n_k_heads, H, S, cfg.scale,
                                               workspace=ws, slots=slots, pool=pool)
        return y, st

    def counts(self, every):
        return [L // (C * every) for L in self.lengths]


LENGTHS = [1, 31, 32, 33, 100, 257, 64, 130]


@pytest.mark.parametrize("every", [1, 2])
def test_ragged_snapshots_equal_single_sequence_calls(lib, every):
    """Each sequence's snapshots (at slots base[n] + j of a dense pool), y and final state:
    the bits of a uniform snapshot call of that sequence alone, and y and state the bits
    of the plain ragged call."""
    rg = RaggedScan(LENGTHS, seed=every)
    cnt = rg.counts(every)
    base = np.concatenate([[0], np.cumsum(cnt)[:-1]]).astype(np.int32)
    snap_pool = int(sum(cnt))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, st, sn = rg.run(lib, every, base, snap_pool, err=err)
    assert host(err)[0] == 0
    y_p, st_p = rg.run_plain(lib)
    assert torch.equal(y, y_p) and torch.equal(st, st_p)
    H, S = rg.cfg.n_v_heads, 128
    for n, L in enumerate(LENGTHS):
        one = I.get_config(0, n_k_heads=2, n_v_heads=H, state_size=128, n_seqs=1, n_tokens=L,
                           cid=1)
        st1 = dev(rg.st0[n:n + 1])
        y1, s1 = run_snap(lib, one, inputs(rg.per[n]), st1, every)
        assert torch.equal(y[rg.cu[n]:rg.cu[n + 1]], y1[0]), f"y of sequence {n}"
        assert torch.equal(st[n], st1[0]), f"state of sequence {n}"
        if cnt[n]:
            assert torch.equal(sn[base[n]:base[n] + cnt[n]], s1[0]), f"snapshots of sequence {n}"
    assert not torch.isnan(sn).any()  # the dense pool is filled exactly


def test_ragged_snapshots_vs_oracle(lib):
    """Two sequences' snapshots against the oracle's state at the same positions."""
    every = 1
    rg = RaggedScan(LENGTHS, seed=5)
    cnt = rg.counts(every)
    base = np.concatenate([[0], np.cumsum(cnt)[:-1]]).astype(np.int32)
    _, _, sn = rg.run(lib, every, base, int(sum(cnt)))
    got = host(sn)
    for n in (5, 7):  # 257 and 130 positions: 8 and 4 snapshots
        one = I.get_config(0, n_k_heads=2, n_v_heads=4, state_size=128, n_seqs=1,
                           n_tokens=LENGTHS[n], cid=1)
        ref = oracle_snapshots(one, rg.per[n], rg.st0[n:n + 1], every)
        for j in range(cnt[n]):
            for vh in range(4):
                assert_rms(got[base[n] + j, vh], ref[0, j, vh], f"snapshot ({n},{j},{vh})")


def test_ragged_snapshot_placement_and_slots(lib):
    """Snapshot ranges that leave the pool (a negative base, one past the end) are
    skipped and counted once each, a sequence with no snapshots is never counted, state
    slots route as usual, and y and state stay the plain call's."""
    lengths = [100, 40, 70, 20, 64]   # 3, 1, 2, 0, 2 snapshots at an interval of 1 chunk
    rg = RaggedScan(lengths, seed=9, pool=7)
    slots = dev(np.array([6, 0, 3, 5, 2], dtype=np.int32))
    base = [0, -1, 9, -5, 3]           # sequence 1 negative, 2 past the pool of 10 slots,
    err = torch.zeros(1, dtype=torch.int32, device="cuda")  # 3 has none (not counted)
    y, st, sn = rg.run(lib, 1, base, 10, slots=slots, pool=7, err=err)
    assert host(err)[0] == 2
    y_p, st_p = rg.run_plain(lib, slots=slots, pool=7)
    assert torch.equal(y, y_p) and torch.equal(st, st_p)
    got = host(sn)
    assert not np.isnan(got[0:3]).any() and not np.isnan(got[3:5]).any()
    assert np.isnan(got[5:]).all()     # nothing else written
    # sequence 4's second snapshot at slot 4 is its final state (64 = 2 chunks)
    np.testing.assert_array_equal(got[4], host(st)[2])


def test_ragged_snapshots_none_reachable(lib):
    """No sequence reaches 32 * snap_every positions: snaps and snap_base may be NULL,
    and the call is the plain ragged scan."""
    rg = RaggedScan([5, 40, 63], seed=4)
    y, st, _ = rg.run(lib, 2, None, 0, snaps=False)
    y_p, st_p = rg.run_plain(lib)
    assert torch.equal(y, y_p) and torch.equal(st, st_p)


def snap_draw(i):
    """Case i: a reproducible ragged batch, interval, slot routing and snapshot placement."""
    r = np.random.default_rng(9100 + i)
    Hk = int(r.choice([1, 2, 4]))
    ratio = int(r.choice([1, 2, 3, 4]))
    N = int(r.integers(1, 7))
    lengths = [int(x) for x in r.integers(1, 300, N)]
    every = int(r.integers(1, 5))
    pool = N + int(r.integers(0, 3))
    slots = r.permutation(pool)[:N].astype(np.int32)
    cnt = [L // (C * every) for L in lengths]
    # the sequences' snapshot ranges in shuffled order, with a gap of 0-2 slots before each
    base, nxt = [0] * N, 0
    for n in r.permutation(N):
        nxt += int(r.integers(0, 3))
        base[n] = nxt
        nxt += cnt[n]
    return dict(Hk=Hk, H=Hk * ratio, N=N, lengths=lengths, every=every, pool=pool,
                slots=slots, base=np.array(base, np.int32), snap_pool=nxt + 1, cnt=cnt)


@pytest.mark.parametrize("i", range(8))
def test_ragged_snapshots_random(lib, i):
    """Seeded ragged batches: every sequence's snapshots are the bits of a uniform call of
    that sequence alone (from its routed slot's state), the unwritten snapshot slots keep
    their contents, and y and the state pool are the plain ragged call's."""
    c = snap_draw(i)
    rg = RaggedScan(c["lengths"], Hk=c["Hk"], H=c["H"], seed=50 + i, pool=c["pool"])
    slots = dev(c["slots"])
    y, st, sn = rg.run(lib, c["every"], c["base"], c["snap_pool"], slots=slots, pool=c["pool"])
    y_p, st_p = rg.run_plain(lib, slots=slots, pool=c["pool"])
    assert torch.equal(y, y_p) and torch.equal(st, st_p)
    written = np.zeros(c["snap_pool"], bool)
    for n, L in enumerate(c["lengths"]):
        if not c["cnt"][n]:
            continue
        one = I.get_config(0, n_k_heads=c["Hk"], n_v_heads=c["H"], state_size=128, n_seqs=1,
                           n_tokens=L, cid=1)
        st1 = dev(rg.st0[c["slots"][n]:c["slots"][n] + 1])
        _, s1 = run_snap(lib, one, inputs(rg.per[n]), st1, c["every"])
        b0 = c["base"][n]
        assert torch.equal(sn[b0:b0 + c["cnt"][n]], s1[0]), f"case {i}: snapshots of sequence {n}"
        written[b0:b0 + c["cnt"][n]] = True
    got = host(sn)
    assert np.isnan(got[~written]).all(), f"case {i}: a slot outside every range was written"
