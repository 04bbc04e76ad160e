"""GPU parity of the ragged-batch (varlen) prefill: sequences of different lengths
packed token-major in one call, sequence n owning positions cu[n] .. cu[n+1] - 1.

Each sequence of a ragged call must give the bits of a call of its own (the same
kernels run the same operations on it), and match the oracle's block, stepped
token by token, under the stated bounds: the first token elementwise
(|d| <= 1e-4 + 1e-4 |ref|), the whole sequence and the final state within 2e-3 of
the reference RMS. Lengths mix the edge cases of the chunked form: a single
position, one short of a chunk, exactly one chunk, one past it, and long ones.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from gated_deltanet_linear_scan_gb300 import inputs as I

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LENGTHS = [1, 31, 32, 33, 700, 4096]


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def assert_step(gpu, ref, name):
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, name
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    err = np.abs(gpu - ref)
    worst = np.max(err - (1e-4 + 1e-4 * np.abs(ref)))
    assert worst <= 0, f"{name}: elementwise bound exceeded by {worst:.3e}"


def assert_rms(gpu, ref, name, rel=2e-3):
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    rms = np.sqrt(np.mean(ref * ref))
    err = np.max(np.abs(gpu - ref))
    assert err <= rel * rms, f"{name}: max err {err:.3e} > {rel} * RMS {rms:.3e}"


@pytest.fixture(scope="module", autouse=True)
def lib(cuda_lib):
    yield cuda_lib
    cuda_lib.gdn_device_error()


class Ragged:
    """A ragged batch: per-sequence inputs (seeded per sequence), their packed form, and
    the pool slots each sequence uses."""

    def __init__(self, cfg, lengths, slots=None, pool=None):
        self.cfg, self.lengths = cfg, list(lengths)
        self.n = len(lengths)
        self.cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        self.total = int(self.cu[-1])
        self.per = [I.prefill_seq(cfg, n, n_tokens=L) for n, L in enumerate(lengths)]
        self.packed = {key: np.concatenate([p[key] for p in self.per]) for key in self.per[0]}
        self.slots = None if slots is None else np.asarray(slots, np.int32)
        self.pool = pool if pool is not None else self.n
        self.st0 = I.state_pool(cfg, which=range(self.pool))
        self.cs0 = I.conv_state_pool(cfg, which=range(self.pool))
        self.static = I.block_static(cfg)
        self.d_static = {k: dev(v) for k, v in self.static.items()}

    def slot(self, n):
        return n if self.slots is None else int(self.slots[n])


def run_varlen(lib, rg, form, ws_bytes=None, err=None, out_fill=0.0, cu=None, max_tokens=None,
               snaps=False):
    """One ragged call; returns (out, state, conv[, snaps, conv_snaps]) device tensors."""
    cfg = rg.cfg
    Hk, H, S, K = cfg.n_k_heads, cfg.n_v_heads, cfg.state_size, cfg.conv_kernel
    state, conv = dev(rg.st0), dev(rg.cs0)
    out = torch.full((rg.total, H, S), out_fill, device="cuda")
    d = {key: dev(v) for key, v in rg.packed.items()}
    cu_d = dev(rg.cu if cu is None else np.asarray(cu, np.int32))
    maxt = max(rg.lengths) if max_tokens is None else max_tokens
    if ws_bytes is None:
        size = (lib.gdn_block_prefill_chunked_varlen_workspace_size if form == "chunked"
                else lib.gdn_block_prefill_varlen_workspace_size)
        ws_bytes = size(rg.n, rg.total, Hk, H, S)
    ws = torch.full(((ws_bytes + 3) // 4,), float("nan"), device="cuda")
    slots = None if rg.slots is None else dev(rg.slots)
    args = (d["qkv"], rg.d_static["conv_w"], conv, d["alpha"], d["b"], rg.d_static["dt"],
            rg.d_static["a"], d["z"], rg.d_static["norm_w"], state, out)
    tail = (cu_d, rg.n, rg.total, maxt, Hk, H, S, K, cfg.scale, cfg.eps, cfg.eps, ws)
    kw = dict(slots=slots, pool=rg.pool, err_count=err)
    if snaps:
        C = (2 * Hk + H) * S
        sn = torch.zeros(rg.total, H, S, S, device="cuda")
        csn = torch.zeros(rg.total, C, K - 1, device="cuda")
        lib.gdn_block_prefill_snapshots_varlen(*args, sn, csn, *tail, **kw)
        return out, state, conv, sn, csn
    fn = lib.gdn_block_prefill_chunked_varlen if form == "chunked" else lib.gdn_block_prefill_varlen
    fn(*args, *tail, **kw)
    return out, state, conv


def run_alone(lib, rg, n, form):
    """Sequence n in a uniform call of its own, on its own slot: (out [L][H][S], state, conv)."""
    cfg = rg.cfg
    Hk, H, S, K = cfg.n_k_heads, cfg.n_v_heads, cfg.state_size, cfg.conv_kernel
    L, sl = rg.lengths[n], rg.slot(n)
    state, conv = dev(rg.st0[sl:sl + 1]), dev(rg.cs0[sl:sl + 1])
    out = torch.zeros(1, L, H, S, device="cuda")
    p = {key: dev(v[None]) for key, v in rg.per[n].items()}
    size = (lib.gdn_block_prefill_chunked_workspace_size if form == "chunked"
            else lib.gdn_block_prefill_workspace_size)
    ws = torch.empty(size(1, L, Hk, H, S) // 4 + 64, device="cuda")
    fn = lib.gdn_block_prefill_chunked if form == "chunked" else lib.gdn_block_prefill
    fn(p["qkv"], rg.d_static["conv_w"], conv, p["alpha"], p["b"], rg.d_static["dt"],
       rg.d_static["a"], p["z"], rg.d_static["norm_w"], state, out, 1, L, Hk, H, S, K,
       cfg.scale, cfg.eps, cfg.eps, ws)
    return out[0], state[0], conv[0]


def oracle_sequence(rg, n):
    """The oracle's block stepped over sequence n: (out [L][H][S], state, conv_state)."""
    cfg, x, sl = rg.cfg, rg.per[n], rg.slot(n)
    st, cs = f64(rg.st0[sl:sl + 1]), f64(rg.cs0[sl:sl + 1])
    outs = []
    for t in range(rg.lengths[n]):
        r, _ = oracle.block_decode(x["qkv"][t:t + 1], rg.static["conv_w"], cs, x["alpha"][t:t + 1],
                                   x["b"][t:t + 1], rg.static["dt"], rg.static["a"],
                                   x["z"][t:t + 1], rg.static["norm_w"], st, cfg.n_k_heads,
                                   cfg.scale, cfg.eps, cfg.eps)
        outs.append(r[0])
    return np.stack(outs), st[0], cs[0]


def oracle_all(rg, seqs):
    oracle.sigmoid(np.zeros(1, np.float32))  # load the library before the threads start
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        return dict(zip(seqs, ex.map(lambda n: oracle_sequence(rg, n), seqs)))


def check_against_oracle(rg, refs, out, state, conv):
    o, st, cv = host(out), host(state), host(conv)
    for n, (r_out, r_st, r_cs) in refs.items():
        a, L, sl = rg.cu[n], rg.lengths[n], rg.slot(n)
        assert_step(o[a], r_out[0], f"seq {n} (length {L}): out, first position")
        assert_rms(o[a:a + L], r_out, f"seq {n} (length {L}): out")
        if L == 1:
            assert_step(st[sl], r_st, f"seq {n}: state after its one position")
            assert_step(cv[sl], r_cs, f"seq {n}: conv_state after its one position")
        else:
            assert_rms(st[sl], r_st, f"seq {n} (length {L}): state")
            assert_rms(cv[sl], r_cs, f"seq {n} (length {L}): conv_state")


@pytest.fixture(scope="module")
def mixed():
    """Lengths {1, 31, 32, 33, 700, 4096} on Hk=2, H=4, S=128, routed through a pool of 9
    slots, and the oracle's results for every sequence."""
    cfg = I.get_config(2, n_seqs=len(LENGTHS), n_k_heads=2, n_v_heads=4, cid=950)
    rg = Ragged(cfg, LENGTHS, slots=[7, 2, 5, 0, 8, 3], pool=9)
    return rg, oracle_all(rg, range(rg.n))


@pytest.mark.parametrize("form", ["sequential", "chunked"])
def test_block_prefill_varlen_mixed_lengths(lib, mixed, form):
    """Every sequence of one ragged call against the oracle, and bit for bit against a
    call of its own; slots no sequence uses keep their bits."""
    rg, refs = mixed
    out, state, conv = run_varlen(lib, rg, form)
    check_against_oracle(rg, refs, out, state, conv)
    for n in range(rg.n):
        a, L, sl = rg.cu[n], rg.lengths[n], rg.slot(n)
        o1, s1, c1 = run_alone(lib, rg, n, form)
        assert torch.equal(out[a:a + L], o1), f"seq {n}: out differs from its own call"
        assert torch.equal(state[sl], s1) and torch.equal(conv[sl], c1), f"seq {n}: states"
    for sl in (1, 4, 6):
        assert np.array_equal(host(state[sl]), rg.st0[sl])
        assert np.array_equal(host(conv[sl]), rg.cs0[sl])


def test_block_prefill_chunked_varlen_one_kernel_form(lib, mixed):
    """With only the intermediates' workspace the chunked ragged call takes the one-kernel
    form: the same bits as the two-phase form."""
    rg, _ = mixed
    cfg = rg.cfg
    small = lib.gdn_block_prefill_varlen_workspace_size(rg.n, rg.total, cfg.n_k_heads,
                                                        cfg.n_v_heads, cfg.state_size)
    o1, s1, c1 = run_varlen(lib, rg, "chunked", ws_bytes=small)
    o2, s2, c2 = run_varlen(lib, rg, "chunked")
    assert torch.equal(o1, o2) and torch.equal(s1, s2) and torch.equal(c1, c2)


def test_block_prefill_snapshots_varlen(lib, mixed):
    """The snapshot form gives gdn_block_prefill_varlen's bits, keeps the state and conv
    history after every position of every sequence (packed as the positions are), and
    gdn_snapshot_restore_varlen rolls each sequence back to its accepted count."""
    rg, _ = mixed
    cfg = rg.cfg
    short = Ragged(cfg, [1, 31, 33, 5, 0, 12], slots=[7, 2, 5, 0, 8, 3], pool=9)
    out_r, st_r, cs_r = run_varlen(lib, short, "sequential")
    out, st, cs, sn, csn = run_varlen(lib, short, "sequential", snaps=True)
    assert torch.equal(out, out_r) and torch.equal(st, st_r) and torch.equal(cs, cs_r)
    for n in range(short.n):
        a, L, sl = short.cu[n], short.lengths[n], short.slot(n)
        if L:
            assert torch.equal(sn[a + L - 1], st[sl]) and torch.equal(csn[a + L - 1], cs[sl])
        for t in sorted({0, L // 2, L - 2} & set(range(L))):  # a prefix in a call of its own
            pre = Ragged(cfg, [t + 1], slots=[sl], pool=9)
            pre.per = [{key: v[:t + 1] for key, v in short.per[n].items()}]
            pre.packed = pre.per[0]
            _, s_p, c_p = run_varlen(lib, pre, "sequential")
            assert torch.equal(sn[a + t], s_p[sl]), f"seq {n}: state snapshot {t}"
            assert torch.equal(csn[a + t], c_p[sl]), f"seq {n}: conv snapshot {t}"
    accepted = np.array([1, 17, 33, 5, 1, 3], np.int32)  # sequence 4 is empty: counted
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = (2 * cfg.n_k_heads + cfg.n_v_heads) * cfg.state_size
    lib.gdn_snapshot_restore_varlen(st, sn, dev(accepted), dev(short.cu), short.n, short.total,
                                    max(short.lengths), cfg.n_v_heads, cfg.state_size,
                                    conv_state=cs, conv_snaps=csn, conv_dim=C,
                                    conv_kernel=cfg.conv_kernel, slots=dev(short.slots), pool=9,
                                    err_count=err)
    assert int(err.item()) == 1
    for n in range(short.n):
        a, sl = short.cu[n], short.slot(n)
        if short.lengths[n]:
            assert torch.equal(st[sl], sn[a + accepted[n] - 1])
            assert torch.equal(cs[sl], csn[a + accepted[n] - 1])
    assert np.array_equal(host(st[8]), short.st0[8])  # the empty sequence's slot


@pytest.mark.parametrize("form", ["sequential", "chunked"])
def test_block_prefill_varlen_invalid_ranges_and_slots(lib, form):
    """A sequence longer than max_tokens, one past total_tokens and one on an out-of-range
    slot are skipped and counted; an empty one is a no-op; out rows of positions no valid
    sequence owns keep their contents; the valid sequences get their own calls' bits."""
    cfg = I.get_config(2, n_seqs=6, n_k_heads=2, n_v_heads=4, cid=951)
    lengths = [5, 20, 0, 9, 7, 4]
    rg = Ragged(cfg, lengths, slots=[0, 1, 2, 3, 11, 5], pool=6)  # slot 11: out of range
    cu = rg.cu.copy()
    cu[-1] = rg.total + 3  # the last sequence reaches past total_tokens
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, state, conv = run_varlen(lib, rg, form, err=err, out_fill=7.0, cu=cu, max_tokens=10)
    assert int(err.item()) == 3  # sequence 1 (20 > max_tokens), 4 (slot), 5 (past the end)
    o = host(out)
    for n in (1, 4, 5):
        a, L = cu[n], rg.lengths[n]
        assert np.all(o[a:min(a + L, rg.total)] == 7.0), f"seq {n}: out rows were written"
    for sl in (1, 2, 5):  # skipped, empty and past-the-end sequences' slots
        assert np.array_equal(host(state[sl]), rg.st0[sl])
        assert np.array_equal(host(conv[sl]), rg.cs0[sl])
    for n in (0, 3):
        a, L, sl = rg.cu[n], rg.lengths[n], rg.slot(n)
        o1, s1, c1 = run_alone(lib, rg, n, form)
        assert torch.equal(out[a:a + L], o1)
        assert torch.equal(state[sl], s1) and torch.equal(conv[sl], c1)


def test_recurrence_scans_varlen_against_own_calls(lib):
    """The scan-level ragged calls: the sequential scan (any state size) and the chunked
    one (S = 128, with and without its workspace) give each sequence the bits of a call
    of its own."""
    for S, Hk, H in ((64, 1, 2), (128, 2, 4)):
        cfg = I.get_config(2, n_seqs=5, n_k_heads=Hk, n_v_heads=H, state_size=S, cid=952 + S)
        lengths = [3, 64, 1, 45, 130]
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        per = [I.recurrence_seq(cfg, n, n_tokens=L) for n, L in enumerate(lengths)]
        x = {key: dev(np.concatenate([p[key] for p in per])) for key in per[0]}
        st0 = I.state_pool(cfg)
        total = int(cu[-1])
        forms = ["sequential"] + (["chunked", "chunked_ws"] if S == 128 else [])
        for form in forms:
            st = dev(st0)
            y = torch.zeros(total, H, S, device="cuda")
            if form == "sequential":
                lib.gdn_recurrence_scan_varlen(st, x["q"], x["k"], x["v"], x["g"], x["beta"], y,
                                               dev(cu), 5, total, 130, Hk, H, S, cfg.scale)
            else:
                ws = None
                if form == "chunked_ws":
                    ws = torch.empty(lib.gdn_recurrence_scan_chunked_varlen_ws_size(5, total, H, S)
                                     // 4, device="cuda")
                lib.gdn_recurrence_scan_chunked_varlen(st, x["q"], x["k"], x["v"], x["g"],
                                                       x["beta"], y, dev(cu), 5, total, 130, Hk,
                                                       H, S, cfg.scale, workspace=ws)
            for n, L in enumerate(lengths):
                s1 = dev(st0[n:n + 1])
                y1 = torch.zeros(1, L, H, S, device="cuda")
                p = {key: dev(v[None]) for key, v in per[n].items()}
                fn = lib.gdn_recurrence_scan if form == "sequential" else lib.gdn_recurrence_scan_chunked
                fn(s1, p["q"], p["k"], p["v"], p["g"], p["beta"], y1, 1, L, Hk, H, S, cfg.scale)
                assert torch.equal(y[cu[n]:cu[n + 1]], y1[0]), f"{form} S={S} seq {n}: y"
                assert torch.equal(st[n], s1[0]), f"{form} S={S} seq {n}: state"
            if form == "sequential":  # and the oracle on the longest one
                n = 4
                ref_s = f64(st0[n:n + 1])
                y_ref, _ = oracle.recurrence(ref_s, scale=cfg.scale,
                                             **{key: v[None] for key, v in per[n].items()})
                assert_rms(host(y[cu[n]:cu[n + 1]]), y_ref[0], f"S={S}: y vs oracle")
                assert_rms(host(st[n]), ref_s[0], f"S={S}: state vs oracle")


@pytest.mark.parametrize("form", ["sequential", "chunked"])
def test_block_prefill_varlen_many_sequences(lib, form):
    """300 short sequences (more than the batches scheduled longest-first): every sequence
    gets the bits of a call of its own (checked on a sample), and sampled ones match the
    oracle."""
    cfg = I.get_config(2, n_seqs=300, n_k_heads=1, n_v_heads=2, cid=953)
    lengths = [int(x) for x in np.random.default_rng(954).integers(0, 40, 300)]
    rg = Ragged(cfg, lengths)
    out, state, conv = run_varlen(lib, rg, form)
    sample = [0, 1, 77, 150, 299] + [n for n in range(300) if lengths[n] in (0, 1, 32, 33)][:6]
    for n in sample:
        a, L = rg.cu[n], rg.lengths[n]
        if L == 0:
            assert np.array_equal(host(state[n]), rg.st0[n])
            continue
        o1, s1, c1 = run_alone(lib, rg, n, form)
        assert torch.equal(out[a:a + L], o1), f"seq {n}: out differs from its own call"
        assert torch.equal(state[n], s1) and torch.equal(conv[n], c1), f"seq {n}: states"
    refs = oracle_all(rg, [n for n in (1, 150, 299) if lengths[n] > 0])
    check_against_oracle(rg, refs, out, state, conv)


def test_block_prefill_varlen_unowned_positions(lib):
    """Offsets need not start at 0 nor end at total_tokens: rows of out at positions no
    sequence owns keep their contents, and the sequences get their own calls' bits."""
    cfg = I.get_config(2, n_seqs=2, n_k_heads=2, n_v_heads=4, cid=955)
    rg = Ragged(cfg, [7, 40])
    cu = np.array([3, 10, 50], np.int32)
    packed = {key: np.concatenate([np.zeros((3,) + v.shape[1:], v.dtype), v,
                                   np.zeros((5,) + v.shape[1:], v.dtype)])
              for key, v in rg.packed.items()}
    rg.packed, rg.total = packed, 55
    for form in ("sequential", "chunked"):
        out, state, conv = run_varlen(lib, rg, form, out_fill=3.0, cu=cu, max_tokens=40)
        o = host(out)
        assert np.all(o[:3] == 3.0) and np.all(o[50:] == 3.0), f"{form}: unowned rows written"
        for n in range(2):
            o1, s1, c1 = run_alone(lib, rg, n, form)
            assert torch.equal(out[cu[n]:cu[n + 1]], o1), f"{form} seq {n}: out"
            assert torch.equal(state[n], s1) and torch.equal(conv[n], c1), f"{form} seq {n}"
