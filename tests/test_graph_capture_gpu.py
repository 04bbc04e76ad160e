"""The library under CUDA-graph capture, as a serving loop would run it: a chain of fused
decode steps, and the chunked scans (one-kernel and two-phase, with their per-launch
attribute calls), captured once and replayed, give the bits of the same calls made
eagerly on the same stream order."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.fixture(scope="module", autouse=True)
def lib(cuda_lib):
    yield cuda_lib
    cuda_lib.gdn_device_error()


@pytest.mark.parametrize("n_seqs", [1, 40])  # the cluster form and the persistent form
def test_decode_chain_in_a_graph(lib, n_seqs):
    cfg = I.get_config(3, n_seqs=n_seqs, cid=810 + n_seqs)
    N, Hk, H, S = cfg.n_seqs, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    steps = [{k: dev(v) for k, v in I.block_step(cfg, t).items()} for t in range(6)]
    state0, conv0 = I.state_pool(cfg), I.conv_state_pool(cfg)

    def run(state, conv, outs):
        for t, a in enumerate(steps):
            lib.gdn_block_decode(a["qkv"], st["conv_w"], conv, a["alpha"], a["b"], st["dt"],
                                 st["a"], a["z"], st["norm_w"], state, outs[t], N, Hk, H, S,
                                 cfg.conv_kernel, cfg.scale, cfg.eps, cfg.eps)

    state_e, conv_e = dev(state0), dev(conv0)
    outs_e = [torch.empty(N, H, S, device="cuda") for _ in steps]
    run(state_e, conv_e, outs_e)

    state_g, conv_g = dev(state0), dev(conv0)
    outs_g = [torch.empty(N, H, S, device="cuda") for _ in steps]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(state_g, conv_g, outs_g)
    # capture records the work without running it: restore the inputs, then replay
    state_g.copy_(dev(state0))
    conv_g.copy_(dev(conv0))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(state_g, state_e)
    assert torch.equal(conv_g, conv_e)
    for a, b in zip(outs_g, outs_e):
        assert torch.equal(a, b)


@pytest.mark.parametrize("form", ["one_kernel", "two_phase"])
def test_chunked_scan_in_a_graph(lib, form):
    cfg = I.get_config(0, n_k_heads=2, n_v_heads=4, state_size=128, n_seqs=2, n_tokens=75,
                       cid=830)
    N, T, Hk, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    x = {k: dev(v) for k, v in I.recurrence_batch(cfg).items()}
    st0 = I.state_pool(cfg)
    ws = torch.empty(lib.gdn_recurrence_scan_chunked_ws_size(N, T, H, S) // 4, device="cuda")

    def run(state, y):
        args = (state, x["q"], x["k"], x["v"], x["g"], x["beta"], y, N, T, Hk, H, S, cfg.scale)
        if form == "one_kernel":
            lib.gdn_recurrence_scan_chunked(*args)
        else:
            lib.gdn_recurrence_scan_chunked_ws(*args, ws)

    state_e, y_e = dev(st0), torch.zeros(N, T, H, S, device="cuda")
    run(state_e, y_e)
    state_g, y_g = dev(st0), torch.zeros(N, T, H, S, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(state_g, y_g)
    state_g.copy_(dev(st0))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(state_g, state_e)
    assert torch.equal(y_g, y_e)


@pytest.mark.parametrize("chunked", [False, True])
def test_ragged_prefill_in_a_graph(lib, chunked):
    """A ragged prefill call (cu_seqlens on the device, read only by the kernels) captured
    once and replayed gives the eager call's bits."""
    cfg = I.get_config(2, n_seqs=4, n_k_heads=2, n_v_heads=4, cid=820 + chunked)
    Hk, H, S, K = cfg.n_k_heads, cfg.n_v_heads, cfg.state_size, cfg.conv_kernel
    lengths = [40, 1, 65, 9]
    cu = dev(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32))
    total = sum(lengths)
    per = [I.prefill_seq(cfg, n, n_tokens=L) for n, L in enumerate(lengths)]
    x = {key: dev(np.concatenate([p[key] for p in per])) for key in per[0]}
    st = {k: dev(v) for k, v in I.block_static(cfg).items()}
    state0, conv0 = I.state_pool(cfg), I.conv_state_pool(cfg)
    size = (lib.gdn_block_prefill_chunked_varlen_workspace_size if chunked
            else lib.gdn_block_prefill_varlen_workspace_size)
    ws = torch.empty(size(4, total, Hk, H, S) // 4 + 64, device="cuda")
    fn = lib.gdn_block_prefill_chunked_varlen if chunked else lib.gdn_block_prefill_varlen

    def run(state, conv, out):
        fn(x["qkv"], st["conv_w"], conv, x["alpha"], x["b"], st["dt"], st["a"], x["z"],
           st["norm_w"], state, out, cu, 4, total, max(lengths), Hk, H, S, K, cfg.scale, cfg.eps,
           cfg.eps, ws)

    state_e, conv_e = dev(state0), dev(conv0)
    out_e = torch.empty(total, H, S, device="cuda")
    run(state_e, conv_e, out_e)
    state_g, conv_g = dev(state0), dev(conv0)
    out_g = torch.empty(total, H, S, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(state_g, conv_g, out_g)
    state_g.copy_(dev(state0))
    conv_g.copy_(dev(conv0))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert torch.equal(state_g, state_e) and torch.equal(conv_g, conv_e)
