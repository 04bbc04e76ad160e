"""Host-side checks of the C ABI (no GPU needed).

libgdn.so must load, export every function include/gdn.h declares, and reject
bad arguments on the host with the documented status before anything is
enqueued. Only argument combinations that fail validation (or are documented
no-ops) are passed here, so no CUDA call is made.
"""
import ctypes
import os
import re

import pytest

import gated_deltanet_linear_scan_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

OK, NULL, SHAPE, UNSUP, ALIGN = 0, 1, 2, 3, 4
P = 0x10000      # a 16-byte aligned fake device address (never dereferenced here)
MIS = 0x10004    # a misaligned one


@pytest.fixture(scope="module")
def lib():
    gdn.build_if_needed()
    return gdn.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("gdn_decay_gate", "gdn_beta_sigmoid", "gdn_conv1d_silu", "gdn_conv1d_silu_seq",
                 "gdn_qkv_split_norm", "gdn_recurrence_decode", "gdn_recurrence_scan",
                 "gdn_gated_norm", "gdn_block_decode", "gdn_status_str", "gdn_version",
                 "gdn_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libgdn.so does not export {name}"
    # and the binding wraps each of them under the same name
    for name in declared_functions():
        assert hasattr(gdn, name), f"binding lacks {name}"


def declared_arity():
    """Parameter count of every function include/gdn.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_binding_arity_matches_the_header():
    """The ctypes table gives each call as many arguments as its C declaration has."""
    arity = declared_arity()
    assert len(arity) == len(declared_functions())
    for name, (args, _) in gdn._SIGS.items():
        assert name in arity, f"{name} is bound but not declared"
        assert len(args) == arity[name], f"{name}: {len(args)} argtypes, {arity[name]} parameters"


def test_status_strings_and_version(lib):
    for code, name in gdn.STATUS.items():
        assert lib.gdn_status_str(code).decode() == name
    assert lib.gdn_status_str(99).decode() == "GDN_ERR_UNKNOWN"
    assert lib.gdn_version() >> 16 == 1


def rec(lib, name, state=P, q=P, k=P, v=P, g=P, beta=P, y=P, n_seqs=1, n_tokens=1, hk=2, hv=4,
        s=32, scale=0.1, slots=None, pool=None, err=None):
    pool = max(1, n_seqs) if pool is None else pool
    if name == "gdn_recurrence_decode":
        return lib.gdn_recurrence_decode(state, q, k, v, g, beta, y, n_seqs, hk, hv, s, scale,
                                         slots, pool, err, None)
    return lib.gdn_recurrence_scan(state, q, k, v, g, beta, y, n_seqs, n_tokens, hk, hv, s, scale,
                                   slots, pool, err, None)


@pytest.mark.parametrize("name", ["gdn_recurrence_decode", "gdn_recurrence_scan"])
def test_recurrence_validation(lib, name):
    assert rec(lib, name, state=None) == NULL
    assert rec(lib, name, y=None) == NULL
    assert rec(lib, name, n_seqs=-1) == SHAPE
    assert rec(lib, name, hk=3, hv=4) == SHAPE          # H % Hk != 0
    assert rec(lib, name, hk=0) == SHAPE
    assert rec(lib, name, s=48) == SHAPE                # not a multiple of 32... 48 % 32 != 0
    assert rec(lib, name, s=512) == SHAPE               # beyond 8 cells per lane
    assert rec(lib, name, s=96) == UNSUP                # valid for the method, no kernel built
    assert rec(lib, name, n_seqs=3, pool=2) == SHAPE    # no slots and pool < n_seqs
    assert rec(lib, name, pool=0) == SHAPE
    assert rec(lib, name, state=MIS) == ALIGN
    assert rec(lib, name, q=MIS) == ALIGN
    assert rec(lib, name, n_seqs=0) == OK               # documented no-op
    if name == "gdn_recurrence_scan":
        assert rec(lib, name, n_tokens=-1) == SHAPE
        assert rec(lib, name, n_tokens=0) == OK


def test_conv_validation(lib):
    f = lib.gdn_conv1d_silu
    assert f(None, P, P, P, 1, 256, 4, None, 1, None, None) == NULL
    assert f(P, P, P, P, 1, 256, 1, None, 1, None, None) == SHAPE
    assert f(P, P, P, P, 1, 256, 9, None, 1, None, None) == SHAPE
    assert f(P, P, P, P, 1, 0, 4, None, 1, None, None) == SHAPE
    assert f(P, P, P, P, 2, 256, 4, None, 1, None, None) == SHAPE
    assert f(P, P, P, P, 0, 256, 4, None, 1, None, None) == OK
    fs = lib.gdn_conv1d_silu_seq
    assert fs(P, P, P, P, 1, -2, 256, 4, None, 1, None, None) == SHAPE
    assert fs(P, P, P, P, 1, 0, 256, 4, None, 1, None, None) == OK



def test_snapshot_restore_validation(lib):
    f = lib.gdn_snapshot_restore
    # state, snaps, conv_state, conv_snaps, accepted, N, T, H, S, conv_dim, K, slots, pool, err
    assert f(None, P, None, None, P, 1, 4, 4, 128, 0, 0, None, 1, None, None) == NULL
    assert f(P, P, None, None, None, 1, 4, 4, 128, 0, 0, None, 1, None, None) == NULL
    assert f(P, P, P, None, P, 1, 4, 4, 128, 256, 4, None, 1, None, None) == NULL  # one conv buffer
    assert f(P, P, None, None, P, 1, 0, 4, 128, 0, 0, None, 1, None, None) == SHAPE
    assert f(P, P, None, None, P, 1, 4, 0, 128, 0, 0, None, 1, None, None) == SHAPE
    assert f(P, P, None, None, P, 1, 4, 4, 100, 0, 0, None, 1, None, None) == SHAPE
    assert f(P, P, None, None, P, 1, 4, 4, 96, 0, 0, None, 1, None, None) == UNSUP
    assert f(P, P, P, P, P, 1, 4, 4, 128, 256, 1, None, 1, None, None) == SHAPE
    assert f(P, P, None, None, P, 2, 4, 4, 128, 0, 0, None, 1, None, None) == SHAPE  # pool < N
    assert f(MIS, P, None, None, P, 1, 4, 4, 128, 0, 0, None, 1, None, None) == ALIGN
    assert f(P, MIS, None, None, P, 1, 4, 4, 128, 0, 0, None, 1, None, None) == ALIGN
    assert f(P, P, P, P, P, 0, 4, 4, 128, 256, 4, None, 1, None, None) == OK  # nothing to do

def test_elementwise_validation(lib):
    assert lib.gdn_decay_gate(P, P, None, P, 4, 2, None) == NULL
    assert lib.gdn_decay_gate(P, P, P, P, 0, 2, None) == SHAPE
    assert lib.gdn_decay_gate(P, P, P, P, 4, 0, None) == OK
    assert lib.gdn_beta_sigmoid(P, None, 4, None) == NULL
    assert lib.gdn_beta_sigmoid(P, P, -1, None) == SHAPE
    assert lib.gdn_beta_sigmoid(P, P, 0, None) == OK
    assert lib.gdn_gated_norm(P, P, P, None, 4, 128, 1e-6, None) == NULL
    assert lib.gdn_gated_norm(P, P, P, P, 4, 100, 1e-6, None) == SHAPE
    assert lib.gdn_gated_norm(P, P, P, P, 4, 96, 1e-6, None) == UNSUP
    assert lib.gdn_gated_norm(MIS, P, P, P, 4, 128, 1e-6, None) == ALIGN
    assert lib.gdn_gated_norm(P, P, P, P, 0, 128, 1e-6, None) == OK
    assert lib.gdn_qkv_split_norm(P, P, P, None, 1, 2, 4, 32, 1e-6, None) == NULL
    assert lib.gdn_qkv_split_norm(P, P, P, P, 1, 3, 4, 32, 1e-6, None) == SHAPE
    assert lib.gdn_qkv_split_norm(P, P, MIS, P, 1, 2, 4, 32, 1e-6, None) == ALIGN
    assert lib.gdn_qkv_split_norm(P, P, P, P, 0, 2, 4, 32, 1e-6, None) == OK


def block(lib, qkv=P, state=P, out=P, conv_state=P, n_seqs=1, hk=2, hv=4, s=32, K=4, slots=None,
          pool=None):
    pool = max(1, n_seqs) if pool is None else pool
    return lib.gdn_block_decode(qkv, P, conv_state, P, P, P, P, P, P, state, out, n_seqs, hk, hv, s, K,
                                0.1, 1e-6, 1e-6, slots, pool, None, None)


def test_variant_validation(lib):
    f = lib.gdn_recurrence_decode_2pass
    assert f(P, P, P, P, P, P, None, 1, 2, 4, 32, 0.1, None, 1, None, None) == NULL
    assert f(P, P, P, P, P, P, P, 1, 2, 4, 96, 0.1, None, 1, None, None) == UNSUP
    assert f(P, P, P, P, P, P, P, 0, 2, 4, 32, 0.1, None, 1, None, None) == OK
    fs = lib.gdn_recurrence_scan_snapshots
    assert fs(P, P, P, P, P, P, P, None, 1, 4, 2, 4, 32, 0.1, None, 1, None, None) == NULL
    assert fs(P, P, P, P, P, P, P, MIS, 1, 4, 2, 4, 32, 0.1, None, 1, None, None) == ALIGN
    assert fs(P, P, P, P, P, P, P, P, 1, 0, 2, 4, 32, 0.1, None, 1, None, None) == OK
    fc = lib.gdn_conv1d_silu_seq_snapshots
    assert fc(P, P, P, P, None, 1, 4, 256, 4, None, 1, None, None) == NULL
    assert fc(P, P, P, P, P, 1, 4, 256, 1, None, 1, None, None) == SHAPE
    assert fc(P, P, P, P, P, 1, 0, 256, 4, None, 1, None, None) == OK


def test_prefill_validation(lib):
    ws = lib.gdn_block_prefill_workspace_size
    ws.restype = ctypes.c_size_t
    need = ws(2, 16, 2, 4, 32)
    # q + k + v + g + beta, each rounded up to 64 floats (the conv pass feeds the
    # split-norm on chip, so no [n][t][C] intermediate)
    parts = [2 * 16 * 2 * 32, 2 * 16 * 2 * 32, 2 * 16 * 4 * 32, 2 * 16 * 4, 2 * 16 * 4]
    assert need == 4 * sum((p + 63) // 64 * 64 for p in parts)
    assert ws(-1, 16, 2, 4, 32) == 0
    f = lib.gdn_block_prefill
    f.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int] * 6 + [ctypes.c_float] * 3 + [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_void_p]

    def call(workspace=P, nbytes=need, n_tokens=16, K=4, qkv=P):
        return f(qkv, P, P, P, P, P, P, P, P, P, P, 2, n_tokens, 2, 4, 32, K, 0.1, 1e-6, 1e-6,
                 None, 2, None, workspace, nbytes, None)
    assert call(qkv=None) == NULL
    assert call(workspace=None) == NULL
    assert call(nbytes=need - 4) == SHAPE
    assert call(workspace=MIS) == ALIGN
    assert call(K=9) == SHAPE
    assert call(n_tokens=0, workspace=None) == OK
    fs = lib.gdn_block_prefill_snapshots  # + snaps, conv_snaps after out

    def call_s(snaps=P, conv_snaps=P, n_tokens=16, workspace=P):
        return fs(P, P, P, P, P, P, P, P, P, P, P, snaps, conv_snaps, 2, n_tokens, 2, 4, 32, 4,
                  0.1, 1e-6, 1e-6, None, 2, None, workspace, ws(2, n_tokens, 2, 4, 32), None)
    assert call_s(snaps=None) == NULL
    assert call_s(conv_snaps=None) == NULL
    assert call_s(snaps=MIS) == ALIGN
    assert call_s(n_tokens=70000) == UNSUP  # positions beyond a grid dimension
    assert call_s(n_tokens=0, workspace=None) == OK


def test_chunked_scan_validation(lib):
    f = lib.gdn_recurrence_scan_chunked
    f.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p,
                                                                ctypes.c_int, ctypes.c_void_p,
                                                                ctypes.c_void_p]

    def call(state=P, q=P, s=128, hk=2, hv=4, n_tokens=40, pool=2, y=P):
        return f(state, q, P, P, P, P, y, 2, n_tokens, hk, hv, s, 0.1, None, pool, None, None)
    assert call(state=None) == NULL
    assert call(y=None) == NULL
    assert call(q=MIS) == ALIGN
    assert call(state=MIS) == ALIGN
    assert call(s=64) == UNSUP            # valid for the method; the tensor-core form is S = 128
    assert call(s=96) == UNSUP
    assert call(s=100) == SHAPE
    assert call(hk=3) == SHAPE
    assert call(pool=1) == SHAPE          # more sequences than slots, no slot map
    assert call(n_tokens=0) == OK


def test_chunked_ws_validation(lib):
    f = lib.gdn_recurrence_scan_chunked_ws
    f.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [
        ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]
    size = lib.gdn_recurrence_scan_chunked_ws_size
    size.argtypes = [ctypes.c_int] * 4
    size.restype = ctypes.c_size_t
    blk = 36 * 1024  # W, Ut and M of one chunk of one (sequence, v-head), fp32
    assert size(2, 40, 4, 128) == 2 * 2 * 4 * blk
    assert size(3, 32, 8, 128) == 1 * 3 * 8 * blk
    assert size(1, 4096, 32, 128) == 128 * 32 * blk
    assert size(2, 40, 4, 64) == 0 and size(0, 40, 4, 128) == 0 and size(2, 0, 4, 128) == 0

    def call(state=P, q=P, s=128, hk=2, hv=4, n_tokens=40, pool=2, y=P, workspace=P,
             nbytes=None):
        nbytes = size(2, n_tokens, hv, 128) if nbytes is None else nbytes
        return f(state, q, P, P, P, P, y, 2, n_tokens, hk, hv, s, 0.1, None, pool, None,
                 workspace, nbytes, None)
    assert call(state=None) == NULL
    assert call(y=None) == NULL
    assert call(workspace=None) == NULL
    assert call(q=MIS) == ALIGN
    assert call(workspace=MIS) == ALIGN
    assert call(s=64) == UNSUP
    assert call(s=100) == SHAPE
    assert call(hk=3) == SHAPE
    assert call(pool=1) == SHAPE
    assert call(nbytes=2 * 4 * blk - 16) == SHAPE  # less than one chunk of every unit
    assert call(n_tokens=0, workspace=None) == OK


def test_chunked_snapshot_validation(lib):
    count = lib.gdn_chunked_snapshot_count
    count.argtypes = [ctypes.c_int] * 2
    count.restype = ctypes.c_int
    assert count(64, 1) == 2 and count(63, 1) == 1 and count(31, 1) == 0
    assert count(4096, 16) == 8 and count(4095, 16) == 7 and count(0, 3) == 0
    assert count(2**31 - 1, 2**30) == 0  # no overflow in 32 * snap_every
    assert count(10, 0) == -1 and count(-1, 1) == -1
    f = lib.gdn_recurrence_scan_chunked_snapshots
    f.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] * 6 + [
        ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_size_t, ctypes.c_void_p]
    blk = 36 * 1024

    def call(snaps=P, every=1, n_tokens=64, q=P, workspace=P, nbytes=None, s=128, pool=2,
             state=P):
        nbytes = 2 * 2 * 4 * blk if nbytes is None else nbytes
        return f(state, q, P, P, P, P, P, snaps, every, 2, n_tokens, 2, 4, s, 0.1, None, pool,
                 None, workspace, nbytes, None)
    assert call(every=0) == SHAPE
    assert call(every=-3) == SHAPE
    assert call(snaps=None) == NULL              # two snapshots to write
    assert call(snaps=MIS) == ALIGN
    assert call(state=None) == NULL
    assert call(workspace=None) == NULL
    assert call(s=64) == UNSUP
    assert call(pool=1) == SHAPE
    # no snapshot falls in 40 positions at an interval of 2 chunks: snaps may be NULL
    # or unaligned, the call gets as far as the workspace check
    assert call(snaps=None, every=2, n_tokens=40, q=MIS) == ALIGN
    assert call(snaps=MIS, every=2, n_tokens=40, nbytes=16) == SHAPE
    assert call(n_tokens=0, snaps=None, workspace=None) == OK
    assert call(n_tokens=0, every=0) == SHAPE  # the interval is checked even when empty


def test_ragged_chunked_snapshot_validation(lib):
    f = lib.gdn_recurrence_scan_chunked_snapshots_varlen
    size = lib.gdn_recurrence_scan_chunked_varlen_ws_size
    size.argtypes = [ctypes.c_int] * 4
    size.restype = ctypes.c_size_t

    def call(snaps=P, base=P, snap_pool=4, every=1, max_tokens=64, total=100, cu=P, state=P,
             q=P, workspace=P, nbytes=None, n_seqs=2):
        nbytes = size(2, total, 4, 128) if nbytes is None else nbytes
        return f(state, q, P, P, P, P, P, snaps, base, snap_pool, every, cu, n_seqs, total,
                 max_tokens, 2, 4, 128, 0.1, None, 2, None, workspace, nbytes, None)
    assert call(state=None) == NULL
    assert call(cu=None) == NULL
    assert call(every=0) == SHAPE
    assert call(snap_pool=-1) == SHAPE
    assert call(snaps=None) == NULL           # a 64-position sequence reaches a snapshot
    assert call(base=None) == NULL
    assert call(snaps=MIS) == ALIGN
    assert call(q=MIS) == ALIGN
    assert call(workspace=None) == NULL
    assert call(workspace=MIS) == ALIGN
    assert call(nbytes=16) == SHAPE           # less than the ragged workspace
    # at most 63 positions and an interval of 2 chunks: no snapshot can fall, so snaps
    # and snap_base may be NULL (the call gets as far as the workspace check)
    assert call(snaps=None, base=None, every=2, max_tokens=63, nbytes=16) == SHAPE
    assert call(n_seqs=0, total=0, max_tokens=0, snaps=None, base=None, workspace=None) == OK


def test_chunked_phase_validation(lib):
    prep = lib.gdn_chunked_prepare
    prep.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_size_t] + [ctypes.c_int] * 7 + [
        ctypes.c_void_p]
    adv = lib.gdn_chunked_advance
    adv.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_size_t, ctypes.c_void_p] + [
        ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    blk = 36 * 1024 * 2 * 4  # one chunk of 2 sequences x 4 v-heads

    def p(cb=0, nc=2, nbytes=2 * blk, ws=P, q=P, s=128, n_tokens=40):
        return prep(q, P, P, P, P, ws, nbytes, 2, n_tokens, 2, 4, s, cb, nc, None)

    def a(cb=0, nc=2, nbytes=2 * blk, ws=P, state=P, pool=2, n_tokens=40):
        return adv(state, P, P, P, ws, nbytes, P, 2, n_tokens, 2, 4, 128, 0.1, cb, nc, None,
                   pool, None, None)
    for f in (p, a):
        assert f(ws=None) == NULL
        assert f(ws=MIS) == ALIGN
        assert f(nbytes=2 * blk - 4) == SHAPE   # the range does not fit
        assert f(cb=1, nc=2) == SHAPE           # 40 positions are 2 chunks
        assert f(cb=-1, nc=1) == SHAPE
        assert f(cb=2, nc=0, ws=None) == OK     # an empty range at the end
        assert f(n_tokens=0, nc=0, ws=None) == OK
    assert p(q=None) == NULL
    assert p(q=MIS) == ALIGN
    assert p(s=64) == UNSUP
    assert a(state=None) == NULL
    assert a(pool=1) == SHAPE


def test_prefill_chunked_workspace_size(lib):
    base = lib.gdn_block_prefill_workspace_size
    base.restype = ctypes.c_size_t
    full = lib.gdn_block_prefill_chunked_workspace_size
    full.restype = ctypes.c_size_t
    scan = lib.gdn_recurrence_scan_chunked_ws_size
    scan.restype = ctypes.c_size_t
    for args in ((2, 40, 2, 4), (4, 4096, 16, 32), (1, 7, 1, 3)):
        b = base(*args, 128)
        assert full(*args, 128) == (b + 15) // 16 * 16 + scan(args[0], args[1], args[3], 128)
        assert full(*args, 64) == base(*args, 64)  # no tensor-core form: nothing extra


def test_prefill_chunked_validation(lib):
    f = lib.gdn_block_prefill_chunked
    f.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int] * 6 + [ctypes.c_float] * 3 + [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_void_p]
    ws = lib.gdn_block_prefill_workspace_size
    ws.restype = ctypes.c_size_t

    def call(s=128, workspace=P, n_tokens=16):
        need = ws(2, n_tokens, 2, 4, s)
        return f(P, P, P, P, P, P, P, P, P, P, P, 2, n_tokens, 2, 4, s, 4, 0.1, 1e-6, 1e-6,
                 None, 2, None, workspace, need, None)
    assert call(s=64) == UNSUP   # the tensor-core scan is built for S = 128
    assert call(workspace=None) == NULL
    assert call(workspace=MIS) == ALIGN
    assert call(n_tokens=0, workspace=None) == OK


def test_block_validation(lib):
    assert block(lib, qkv=None) == NULL
    assert block(lib, out=None) == NULL
    assert block(lib, K=1) == SHAPE
    assert block(lib, K=3) == UNSUP        # valid conv kernel, the fused block is built for 4
    assert block(lib, hk=1, hv=16) == UNSUP  # GQA ratio beyond a portable cluster
    assert block(lib, hk=3, hv=4) == SHAPE
    assert block(lib, s=96) == UNSUP
    assert block(lib, state=MIS) == ALIGN
    assert block(lib, conv_state=MIS) == ALIGN
    assert block(lib, n_seqs=4, pool=2) == SHAPE
    assert block(lib, n_seqs=0) == OK


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(4)
    with pytest.raises(ValueError):
        gdn.gdn_beta_sigmoid(x, x, 4, stream=0)


def declared_signatures():
    """{name: [parameter type strings]} of every function include/gdn.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"#define[^\n]*", "", text)
    sigs = {}
    for m in re.finditer(r"\b(gdn_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).replace("\n", " ").split(",")]
        sigs[m.group(1)] = [] if params == ["void"] else params
    return sigs


def _ctype_of(param):
    """The ctypes type a header parameter declaration maps to."""
    decl = " ".join(param.split())
    if "*" in decl or decl.startswith("gdn_stream_t"):
        return ctypes.c_void_p
    if decl.startswith("size_t"):
        return ctypes.c_size_t
    if decl.startswith("float"):
        return ctypes.c_float
    if decl.startswith("unsigned"):
        return ctypes.c_uint
    if decl.startswith(("int", "gdn_status")):
        return ctypes.c_int
    raise AssertionError(f"unmapped parameter type: {param}")


def test_binding_signatures_match_the_header(lib):
    """Every ctypes signature of the binding has the header's parameter count and types:
    a miscounted argument list would pass garbage through the C ABI."""
    sigs = declared_signatures()
    assert set(sigs) == set(declared_functions())
    for name, params in sigs.items():
        assert name in gdn._SIGS, f"binding has no signature for {name}"
        argtypes = gdn._SIGS[name][0]
        assert len(argtypes) == len(params), f"{name}: {len(argtypes)} != {len(params)} params"
        for i, (got, param) in enumerate(zip(argtypes, params)):
            assert got is _ctype_of(param), f"{name} argument {i} ({param}): {got}"


def test_varlen_validation(lib):
    """Ragged-batch calls: NULL cu_seqlens, negative sizes, and the documented no-ops are
    decided on the host, before anything is enqueued."""
    f = lib.gdn_recurrence_scan_varlen
    # state q k v g beta y cu | n_seqs total max Hk H S | scale slots pool err stream
    assert f(P, P, P, P, P, P, P, None, 2, 10, 8, 2, 4, 32, 0.1, None, 2, None, None) == NULL
    assert f(P, P, P, P, P, P, P, P, -1, 10, 8, 2, 4, 32, 0.1, None, 2, None, None) == SHAPE
    assert f(P, P, P, P, P, P, P, P, 2, -1, 8, 2, 4, 32, 0.1, None, 2, None, None) == SHAPE
    assert f(P, P, P, P, P, P, P, P, 2, 10, -1, 2, 4, 32, 0.1, None, 2, None, None) == SHAPE
    assert f(P, P, P, P, P, P, P, P, 2, 10, 8, 3, 4, 32, 0.1, None, 2, None, None) == SHAPE
    assert f(MIS, P, P, P, P, P, P, P, 2, 10, 8, 2, 4, 32, 0.1, None, 2, None, None) == ALIGN
    assert f(P, P, P, P, P, P, P, P, 0, 0, 0, 2, 4, 32, 0.1, None, 1, None, None) == OK
    assert f(P, P, P, P, P, P, P, P, 2, 0, 8, 2, 4, 32, 0.1, None, 2, None, None) == OK
    c = lib.gdn_recurrence_scan_chunked_varlen
    assert c(P, P, P, P, P, P, P, P, 2, 10, 8, 2, 4, 64, 0.1, None, 2, None, None, 0,
             None) == UNSUP
    assert c(P, P, P, P, P, P, P, P, 2, 10, 8, 2, 4, 128, 0.1, None, 2, None, MIS, 1 << 20,
             None) == ALIGN
    assert lib.gdn_recurrence_scan_chunked_varlen_ws_size(3, 100, 4, 128) == (100 // 32 + 3) * 4 * 36864
    assert lib.gdn_recurrence_scan_chunked_varlen_ws_size(3, 100, 4, 64) == 0
    b = lib.gdn_block_prefill_varlen
    args = [P] * 11
    tail = [2, 4, 32, 4, 0.1, 1e-6, 1e-6, None, 2, None]
    assert b(*args, None, 2, 10, 8, *tail, P, 1 << 30, None) == NULL
    assert b(*args, P, 2, 10, 8, *tail, P, 16, None) == SHAPE  # workspace too small
    assert b(*args, P, 2, 0, 8, *tail, None, 0, None) == OK    # nothing to do
    need = lib.gdn_block_prefill_varlen_workspace_size(2, 10, 2, 4, 32)
    assert need == lib.gdn_block_prefill_workspace_size(1, 10, 2, 4, 32) > 0
    assert (lib.gdn_block_prefill_chunked_varlen_workspace_size(2, 100, 2, 4, 128)
            >= lib.gdn_block_prefill_varlen_workspace_size(2, 100, 2, 4, 128)
            + lib.gdn_recurrence_scan_chunked_varlen_ws_size(2, 100, 4, 128))
    r = lib.gdn_snapshot_restore_varlen
    # state snaps conv_state conv_snaps accepted cu | n total max H S C K | slots pool err stream
    assert r(P, P, None, None, P, None, 2, 10, 8, 4, 32, 0, 0, None, 2, None, None) == NULL
    assert r(P, P, None, None, P, P, 2, -1, 8, 4, 32, 0, 0, None, 2, None, None) == SHAPE
    assert r(P, P, P, None, P, P, 2, 10, 8, 4, 32, 8, 4, None, 2, None, None) == NULL


def test_selftest_validation(lib):
    f = lib.gdn_selftest_bounded_wait
    assert f(1, 1000, None, None) == NULL
    assert f(16, 1000, P, None) == SHAPE
    assert f(1, 0, P, None) == SHAPE
    assert f(1, 2000001, P, None) == SHAPE
