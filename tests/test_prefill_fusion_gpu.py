"""The prefill block's fused kernels against the library's stand-alone kernels on the same
inputs. The block runs the conv scan with the q/k split + L2-norm in one pass, and the
decay gate with beta in another. The chain runs the conv scan, the split-norm, the decay
gate, beta, the sequential scan and the gated norm as separate calls. Each fused kernel
performs the stand-alone kernels' operations in the same order, so out, state and
conv_state must agree bit for bit. The cases cover:
- every state size, i.e. every lane width of the fused pass (1, 2, 4 and 8 channels);
- conv widths 2 to 8;
- lengths that end inside a position block, or that are shorter than the conv history;
- head counts whose slices do not fill the last group of a CTA;
- a slot map into a larger pool."""
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


CASES = [  # (Hk, H, S, K, N, T, pool)
    (2, 4, 32, 2, 2, 37, None),
    (2, 4, 64, 3, 2, 45, None),
    (4, 8, 128, 4, 3, 70, None),
    (2, 4, 256, 5, 2, 40, None),
    (2, 6, 128, 8, 2, 5, None),
    (1, 1, 128, 4, 1, 1, None),
    (16, 32, 128, 4, 2, 100, 5),
    (3, 6, 64, 6, 3, 33, 7),
]


@pytest.mark.parametrize("Hk,H,S,K,N,T,pool", CASES)
def test_block_prefill_equals_standalone_chain(lib, Hk, H, S, K, N, T, pool):
    cfg = I.get_config(0, n_k_heads=Hk, n_v_heads=H, state_size=S, conv_kernel=K, n_seqs=N,
                       n_tokens=T, pool=pool, cid=900 + 7 * S + K + T)
    C = cfg.conv_dim
    seqs = [I.prefill_seq(cfg, n) for n in range(N)]
    x = {key: dev(np.stack([s[key] for s in seqs])) for key in ("qkv", "alpha", "b", "z")}
    st = {key: dev(v) for key, v in I.block_static(cfg).items()}
    sl = I.slots(cfg)
    d_slots = None if sl is None else dev(sl)
    P = cfg.pool_size
    state0, conv0 = dev(I.state_pool(cfg)), dev(I.conv_state_pool(cfg))

    # the block
    state_b, conv_b = state0.clone(), conv0.clone()
    out_b = torch.full((N, T, H, S), float("nan"), device="cuda")
    ws = torch.empty(lib.gdn_block_prefill_workspace_size(N, T, Hk, H, S) // 4 + 1,
                     device="cuda")
    lib.gdn_block_prefill(x["qkv"], st["conv_w"], conv_b, x["alpha"], x["b"], st["dt"], st["a"],
                          x["z"], st["norm_w"], state_b, out_b, N, T, Hk, H, S, K, cfg.scale,
                          cfg.eps, cfg.eps, ws, slots=d_slots, pool=P)

    # the chain of stand-alone kernels
    state_c, conv_c = state0.clone(), conv0.clone()
    conv_out = torch.empty(N, T, C, device="cuda")
    lib.gdn_conv1d_silu_seq(x["qkv"], st["conv_w"], conv_c, conv_out, N, T, C, K,
                            slots=d_slots, pool=P)
    q = torch.empty(N, T, Hk, S, device="cuda")
    k = torch.empty_like(q)
    v = torch.empty(N, T, H, S, device="cuda")
    lib.gdn_qkv_split_norm(conv_out, q, k, v, N * T, Hk, H, S, cfg.eps)
    g = torch.empty(N, T, H, device="cuda")
    lib.gdn_decay_gate(x["alpha"], st["dt"], st["a"], g, H, N * T)
    beta = torch.empty(N, T, H, device="cuda")
    lib.gdn_beta_sigmoid(x["b"], beta, N * T * H)
    y = torch.empty(N, T, H, S, device="cuda")
    lib.gdn_recurrence_scan(state_c, q, k, v, g, beta, y, N, T, Hk, H, S, cfg.scale,
                            slots=d_slots, pool=P)
    out_c = torch.empty_like(y)
    lib.gdn_gated_norm(y, st["norm_w"], x["z"], out_c, N * T * H, S, cfg.eps)
    torch.cuda.synchronize()

    assert torch.equal(conv_b, conv_c), "conv_state"
    assert torch.equal(state_b, state_c), "state"
    assert torch.equal(out_b, out_c), "out"
