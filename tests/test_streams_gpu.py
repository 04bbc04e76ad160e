"""Independent calls on two streams at once: a fused decode chain on one pool and a
ragged chunked prefill on another, enqueued on two streams so that their kernels can run
side by side, give the bits of the same calls run one after the other. The library keeps
no per-call state in device globals that such calls could share (the allocation-free
prefill, whose scratch is shared by design, is not used here)."""
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


def test_two_streams_equal_sequential(lib):
    # decode: 40 sequences (the persistent form), 4 chained steps
    dcfg = I.get_config(3, n_seqs=40, cid=840)
    N, Hk, H, S = dcfg.n_seqs, dcfg.n_k_heads, dcfg.n_v_heads, dcfg.state_size
    dst = {k: dev(v) for k, v in I.block_static(dcfg).items()}
    dsteps = [{k: dev(v) for k, v in I.block_step(dcfg, t).items()} for t in range(4)]
    dstate0, dconv0 = dev(I.state_pool(dcfg)), dev(I.conv_state_pool(dcfg))
    # ragged chunked prefill: 5 sequences on a pool of its own
    pcfg = I.get_config(2, n_seqs=5, n_k_heads=2, n_v_heads=4, cid=841)
    lengths = [100, 3, 64, 1, 257]
    cu = dev(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32))
    total = sum(lengths)
    per = [I.prefill_seq(pcfg, n, n_tokens=L) for n, L in enumerate(lengths)]
    px = {key: dev(np.concatenate([p[key] for p in per])) for key in per[0]}
    pst = {k: dev(v) for k, v in I.block_static(pcfg).items()}
    pstate0, pconv0 = dev(I.state_pool(pcfg)), dev(I.conv_state_pool(pcfg))
    pk, ph, ps = pcfg.n_k_heads, pcfg.n_v_heads, pcfg.state_size
    wbytes = lib.gdn_block_prefill_chunked_varlen_workspace_size(5, total, pk, ph, ps)

    def decode_chain(state, conv, outs, stream):
        for t, a in enumerate(dsteps):
            lib.gdn_block_decode(a["qkv"], dst["conv_w"], conv, a["alpha"], a["b"], dst["dt"],
                                 dst["a"], a["z"], dst["norm_w"], state, outs[t], N, Hk, H, S,
                                 4, dcfg.scale, dcfg.eps, dcfg.eps, stream=stream)

    def prefill(state, conv, out, ws, stream):
        lib.gdn_block_prefill_chunked_varlen(
            px["qkv"], pst["conv_w"], conv, px["alpha"], px["b"], pst["dt"], pst["a"], px["z"],
            pst["norm_w"], state, out, cu, 5, total, max(lengths), pk, ph, ps, 4, pcfg.scale,
            pcfg.eps, pcfg.eps, ws, stream=stream)

    def run(concurrent):
        ds, dc = dstate0.clone(), dconv0.clone()
        douts = [torch.empty(N, H, S, device="cuda") for _ in dsteps]
        pstate, pconv = pstate0.clone(), pconv0.clone()
        pout = torch.empty(total, ph, ps, device="cuda")
        ws = torch.empty(wbytes // 4 + 64, device="cuda")
        torch.cuda.synchronize()
        if concurrent:
            s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
            decode_chain(ds, dc, douts, s1.cuda_stream)
            prefill(pstate, pconv, pout, ws, s2.cuda_stream)
        else:
            s = torch.cuda.current_stream().cuda_stream
            decode_chain(ds, dc, douts, s)
            prefill(pstate, pconv, pout, ws, s)
        torch.cuda.synchronize()
        return [ds, dc, pstate, pconv, pout] + douts

    seq, conc = run(False), run(True)
    for i, (a, b) in enumerate(zip(seq, conc)):
        assert torch.equal(a, b), f"tensor {i} differs between two streams and one"
