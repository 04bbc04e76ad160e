"""The decode calls visit their work in alternating directions from one launch to the
next (so that a step starts on the state its predecessor left in L2). The results must
not depend on the direction: two consecutive calls from the same state, one in each
direction, give the same bits, for the fused block (its persistent form at 64 sequences,
with and without a slot map) and for the recurrence alone."""
import numpy as np
import pytest

from gated_deltanet_linear_scan_gb300 import inputs as I

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.fixture(scope="module", autouse=True)
def lib(cuda_lib):
    yield cuda_lib
    cuda_lib.gdn_device_error()


@pytest.mark.parametrize("which", [3, 4])
def test_block_decode_both_directions_same_bits(lib, which):
    cfg = I.get_config(which)
    N, H, Hk, S = cfg.n_seqs, cfg.n_v_heads, cfg.n_k_heads, cfg.state_size
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    a = {k: dev(v) for k, v in I.block_step(cfg, 0).items()}
    slots = I.slots(cfg)
    d_slots = None if slots is None else dev(slots)
    state0, conv0 = dev(I.state_pool(cfg)), dev(I.conv_state_pool(cfg))
    results = []
    for _ in range(3):  # directions d, not d, d
        state, conv = state0.clone(), conv0.clone()
        out = torch.full((N, H, S), float("nan"), device="cuda")
        lib.gdn_block_decode(a["qkv"], st["conv_w"], conv, a["alpha"], a["b"], st["dt"],
                             st["a"], a["z"], st["norm_w"], state, out, N, Hk, H, S,
                             cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps, slots=d_slots,
                             pool=cfg.pool_size)
        results.append((out, state, conv))
    for out, state, conv in results[1:]:
        assert torch.equal(out, results[0][0])
        assert torch.equal(state, results[0][1])
        assert torch.equal(conv, results[0][2])


def test_recurrence_decode_both_directions_same_bits(lib):
    cfg = I.get_config(3)
    N, H, Hk, S = cfg.n_seqs, cfg.n_v_heads, cfg.n_k_heads, cfg.state_size
    x = I.recurrence_batch(cfg, n_tokens=1)
    d = {k: dev(np.ascontiguousarray(v[:, 0])) for k, v in x.items()}
    state0 = dev(I.state_pool(cfg))
    results = []
    for _ in range(3):
        state = state0.clone()
        y = torch.full((N, H, S), float("nan"), device="cuda")
        lib.gdn_recurrence_decode(state, d["q"], d["k"], d["v"], d["g"], d["beta"], y, N, Hk, H,
                                  S, cfg.scale)
        results.append((y, state))
    for y, state in results[1:]:
        assert torch.equal(y, results[0][0])
        assert torch.equal(state, results[0][1])
