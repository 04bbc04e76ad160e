"""The allocation-free prefill entry point against the workspace one.

Some callers cannot allocate device memory: a plugin that only receives the
input and output buffers of the engine hosting it, or a serving loop that must
not allocate mid-step. gdn_block_prefill_noalloc serves them from a fixed scratch
array inside the library. It runs the same kernels as gdn_block_prefill, so its
results must be the same bits. This file is collected last, so a run that stops
at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import gated_deltanet_linear_scan_gb300 as gdn
from gated_deltanet_linear_scan_gb300 import inputs as I

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _ptr(t):
    return None if t is None else P(t.data_ptr())


def noalloc(lib, x, st, conv, state, out, N, T, Hk, H, S, cfg, slots=None, pool=None,
            err=None):
    """One call of gdn_block_prefill_noalloc through the C ABI; returns its status."""
    stream = torch.cuda.current_stream().cuda_stream
    return lib.gdn_block_prefill_noalloc(
        _ptr(x["qkv"]), _ptr(st["conv_w"]), _ptr(conv), _ptr(x["alpha"]), _ptr(x["b"]),
        _ptr(st["dt"]), _ptr(st["a"]), _ptr(x["z"]), _ptr(st["norm_w"]), _ptr(state), _ptr(out),
        N, T, Hk, H, S, 4, cfg.scale, cfg.eps, cfg.eps, _ptr(slots), N if pool is None else pool,
        _ptr(err), P(stream))


def workspace_call(x, st, conv, state, out, N, T, Hk, H, S, cfg, slots=None, pool=None,
                   err=None):
    need = gdn.gdn_block_prefill_workspace_size(N, T, Hk, H, S)
    ws = torch.full((need // 4,), float("nan"), device="cuda")
    gdn.gdn_block_prefill(x["qkv"], st["conv_w"], conv, x["alpha"], x["b"], st["dt"], st["a"],
                          x["z"], st["norm_w"], state, out, N, T, Hk, H, S, 4, cfg.scale, cfg.eps,
                          cfg.eps, ws, slots=slots, pool=pool, err_count=err)


def inputs(cfg, N, T, first):
    per = [I.prefill_seq(cfg, first + n, n_tokens=T) for n in range(N)]
    return {key: dev(np.stack([p_[key] for p_ in per])) for key in per[0]}


def test_noalloc_prefill_matches_workspace_prefill_on_two_calls(cuda_lib):
    lib = cuda_lib.library()
    cfg = I.get_config(3, n_seqs=2, n_tokens=24, cid=900)
    N, T, Hk, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    assert 0 < gdn.gdn_block_prefill_workspace_size(N, T, Hk, H, S) <= \
        gdn.PREFILL_NOALLOC_SCRATCH_BYTES
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    state0, conv0 = dev(I.state_pool(cfg)), dev(I.conv_state_pool(cfg))
    ref_state, ref_conv = state0.clone(), conv0.clone()
    na_state, na_conv = state0.clone(), conv0.clone()
    for call in range(2):  # the second call continues from the states the first left
        x = inputs(cfg, N, T, 10 * call)
        ref_out = torch.empty(N, T, H, S, device="cuda")
        na_out = torch.full((N, T, H, S), float("nan"), device="cuda")
        workspace_call(x, st, ref_conv, ref_state, ref_out, N, T, Hk, H, S, cfg)
        rc = noalloc(lib, x, st, na_conv, na_state, na_out, N, T, Hk, H, S, cfg)
        assert rc == 0, gdn.gdn_status_str(rc)
        torch.cuda.synchronize()
        assert torch.equal(na_out, ref_out), f"call {call}: out differs"
        assert torch.equal(na_state, ref_state), f"call {call}: state differs"
        assert torch.equal(na_conv, ref_conv), f"call {call}: conv_state differs"
    gdn.gdn_device_error()


def test_noalloc_prefill_smaller_call_with_skipped_slot_after_larger_one(cuda_lib):
    """The scratch keeps the previous call's contents; a later, smaller call with an
    out-of-range slot must still leave that sequence's out rows and every slot it does
    not own untouched, and give the workspace call's bits for the others."""
    lib = cuda_lib.library()
    cfg = I.get_config(3, n_seqs=3, n_tokens=40, pool=5, cid=901)
    Hk, H, S = cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    state0, conv0 = dev(I.state_pool(cfg)), dev(I.conv_state_pool(cfg))
    # a larger call first fills the scratch
    big = inputs(cfg, 3, 40, 0)
    s_big, c_big = state0.clone(), conv0.clone()
    out_big = torch.empty(3, 40, H, S, device="cuda")
    rc = noalloc(lib, big, st, c_big, s_big, out_big, 3, 40, Hk, H, S, cfg,
                 slots=dev(np.array([0, 1, 2], np.int32)), pool=5)
    assert rc == 0, gdn.gdn_status_str(rc)
    # then a smaller one with sequence 1 on an out-of-range slot
    T = 7
    small = inputs(cfg, 3, T, 20)
    slots = dev(np.array([4, 9, 1], np.int32))
    err_na = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_ws = torch.zeros(1, dtype=torch.int32, device="cuda")
    na_state, na_conv = state0.clone(), conv0.clone()
    ws_state, ws_conv = state0.clone(), conv0.clone()
    na_out = torch.full((3, T, H, S), 5.0, device="cuda")
    ws_out = torch.full((3, T, H, S), 5.0, device="cuda")
    rc = noalloc(lib, small, st, na_conv, na_state, na_out, 3, T, Hk, H, S, cfg, slots=slots,
                 pool=5, err=err_na)
    assert rc == 0, gdn.gdn_status_str(rc)
    workspace_call(small, st, ws_conv, ws_state, ws_out, 3, T, Hk, H, S, cfg, slots=slots,
                   pool=5, err=err_ws)
    torch.cuda.synchronize()
    assert int(err_na.item()) == 1 and int(err_ws.item()) == 1
    assert torch.all(na_out[1] == 5.0), "the skipped sequence's out rows were written"
    for sl in (0, 2, 3):  # slots no valid sequence of the small call owns
        assert torch.equal(na_state[sl], state0[sl]) and torch.equal(na_conv[sl], conv0[sl])
    assert torch.equal(na_out, ws_out)
    assert torch.equal(na_state, ws_state) and torch.equal(na_conv, ws_conv)
    gdn.gdn_device_error()


def test_noalloc_prefill_at_its_size_limit(cuda_lib):
    """The longest single sequence whose workspace fits the scratch runs and gives the
    workspace call's bits; one position more is GDN_ERR_UNSUPPORTED, with nothing
    enqueued."""
    lib = cuda_lib.library()
    cfg = I.get_config(3, n_seqs=1, cid=902)
    Hk, H, S = cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    limit = gdn.PREFILL_NOALLOC_SCRATCH_BYTES
    T = 1
    while gdn.gdn_block_prefill_workspace_size(1, T + 1, Hk, H, S) <= limit:
        T += 1
    assert gdn.gdn_block_prefill_workspace_size(1, T, Hk, H, S) <= limit
    assert gdn.gdn_block_prefill_workspace_size(1, T + 1, Hk, H, S) > limit
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    state0, conv0 = dev(I.state_pool(cfg)), dev(I.conv_state_pool(cfg))
    x = inputs(cfg, 1, T, 0)
    na_state, na_conv = state0.clone(), conv0.clone()
    ws_state, ws_conv = state0.clone(), conv0.clone()
    na_out = torch.empty(1, T, H, S, device="cuda")
    ws_out = torch.empty(1, T, H, S, device="cuda")
    rc = noalloc(lib, x, st, na_conv, na_state, na_out, 1, T, Hk, H, S, cfg)
    assert rc == 0, gdn.gdn_status_str(rc)
    workspace_call(x, st, ws_conv, ws_state, ws_out, 1, T, Hk, H, S, cfg)
    torch.cuda.synchronize()
    assert torch.equal(na_out, ws_out)
    assert torch.equal(na_state, ws_state) and torch.equal(na_conv, ws_conv)
    # one position more: rejected on the host before anything is enqueued, so the
    # state is left as it was
    before = na_state.clone()
    x1 = inputs(cfg, 1, T + 1, 0)
    out1 = torch.empty(1, T + 1, H, S, device="cuda")
    rc = noalloc(lib, x1, st, na_conv, na_state, out1, 1, T + 1, Hk, H, S, cfg)
    assert gdn.gdn_status_str(rc) == "GDN_ERR_UNSUPPORTED"
    torch.cuda.synchronize()
    assert torch.equal(na_state, before)
    gdn.gdn_device_error()


def test_noalloc_prefill_rejects_sizes_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.library()
    cfg = I.get_config(2)
    assert (gdn.gdn_block_prefill_workspace_size(4, 4096, 16, 32, 128)
            > gdn.PREFILL_NOALLOC_SCRATCH_BYTES)
    dummy = torch.zeros(16, device="cuda")
    p = P(dummy.data_ptr())
    rc = lib.gdn_block_prefill_noalloc(p, p, p, p, p, p, p, p, p, p, p, 4, 4096, 16, 32, 128, 4,
                                       cfg.scale, cfg.eps, cfg.eps, None, 4, None, None)
    assert gdn.gdn_status_str(rc) == "GDN_ERR_UNSUPPORTED"
