"""The allocation-free prefill entry point against the workspace one.

Some callers cannot allocate device memory: a plugin that only receives the
input and output buffers of the engine hosting it, or a serving loop that must
not allocate mid-step. gdn_block_prefill_noalloc serves them from a fixed scratch
array inside the library. This file is collected last, so a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import gated_deltanet_linear_scan_gb300 as gdn
from gated_deltanet_linear_scan_gb300 import inputs as I

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def test_noalloc_prefill_matches_workspace_prefill_on_two_calls(cuda_lib):
    lib = cuda_lib.library()
    cfg = I.get_config(3, n_seqs=2, n_tokens=24, cid=900)
    N, T, Hk, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    need = cuda_lib.gdn_block_prefill_workspace_size(N, T, Hk, H, S)
    assert 0 < need <= cuda_lib.PREFILL_NOALLOC_SCRATCH_BYTES
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    state0, conv0 = dev(I.state_pool(cfg)), dev(I.conv_state_pool(cfg))
    ref_state, ref_conv = state0.clone(), conv0.clone()
    na_state, na_conv = state0.clone(), conv0.clone()
    ws = torch.empty(need // 4, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    P = ctypes.c_void_p
    for call in range(2):  # the second call continues from the states the first left
        per = [I.prefill_seq(cfg, n + 10 * call, n_tokens=T) for n in range(N)]
        x = {key: dev(np.stack([p[key] for p in per])) for key in per[0]}
        ref_out = torch.empty(N, T, H, S, device="cuda")
        na_out = torch.full((N, T, H, S), float("nan"), device="cuda")
        cuda_lib.gdn_block_prefill(x["qkv"], st["conv_w"], ref_conv, x["alpha"], x["b"], st["dt"],
                                   st["a"], x["z"], st["norm_w"], ref_state, ref_out, N, T, Hk, H,
                                   S, 4, cfg.scale, cfg.eps, cfg.eps, ws)
        # through the C ABI directly
        rc = lib.gdn_block_prefill_noalloc(
            P(x["qkv"].data_ptr()), P(st["conv_w"].data_ptr()), P(na_conv.data_ptr()),
            P(x["alpha"].data_ptr()), P(x["b"].data_ptr()), P(st["dt"].data_ptr()),
            P(st["a"].data_ptr()), P(x["z"].data_ptr()), P(st["norm_w"].data_ptr()),
            P(na_state.data_ptr()), P(na_out.data_ptr()), N, T, Hk, H, S, 4, cfg.scale, cfg.eps,
            cfg.eps, None, N, None, P(stream))
        assert rc == 0, gdn.gdn_status_str(rc)
        torch.cuda.synchronize()
        for name, got, want in (("out", na_out, ref_out), ("state", na_state, ref_state),
                                ("conv_state", na_conv, ref_conv)):
            g, w = got.cpu().double().numpy(), want.cpu().double().numpy()
            assert np.all(np.isfinite(g)), f"call {call}: {name} not finite"
            err = np.abs(g - w)
            assert np.all(err <= 1e-4 + 1e-4 * np.abs(w)), f"call {call}: {name} differs"
    cuda_lib.gdn_device_error()


def test_noalloc_prefill_rejects_sizes_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.library()
    cfg = I.get_config(2)
    assert (cuda_lib.gdn_block_prefill_workspace_size(4, 4096, 16, 32, 128)
            > cuda_lib.PREFILL_NOALLOC_SCRATCH_BYTES)
    P = ctypes.c_void_p
    dummy = torch.zeros(16, device="cuda")
    p = P(dummy.data_ptr())
    rc = lib.gdn_block_prefill_noalloc(p, p, p, p, p, p, p, p, p, p, p, 4, 4096, 16, 32, 128, 4,
                                       cfg.scale, cfg.eps, cfg.eps, None, 4, None, None)
    assert gdn.gdn_status_str(rc) == "GDN_ERR_UNSUPPORTED"
