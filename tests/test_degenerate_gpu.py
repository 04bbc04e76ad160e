"""Degenerate inputs on the GPU, where the method's result is known exactly.

beta = 0 and g = 0 make every delta-rule step the identity on the state (the decay
factor is exp(0) = 1 and the rank-1 write is multiplied by 0), so the decode step, the
sequential scan and both chunked scans must leave the state bit for bit as it was, and
read out y = scale * S^T q. With q = 0 the readout is exactly 0. With k = 0 the state
only decays: S_T = exp(g_0 + ... + g_{T-1}) S_0.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gated_deltanet_linear_scan_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


@pytest.fixture(scope="module", autouse=True)
def lib(cuda_lib):
    yield cuda_lib
    cuda_lib.gdn_device_error()


FORMS = ["decode", "scan", "chunked", "chunked_ws"]


def run_form(lib, form, cfg, x, st):
    N, T, Hk, H, S = cfg.n_seqs, cfg.n_tokens, cfg.n_k_heads, cfg.n_v_heads, cfg.state_size
    d = {key: dev(v) for key, v in x.items()}
    y = torch.full((N, T, H, S), float("nan"), device="cuda")
    if form == "decode":
        for t in range(T):
            yt = torch.empty(N, H, S, device="cuda")
            lib.gdn_recurrence_decode(st, d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                      d["v"][:, t].contiguous(), d["g"][:, t].contiguous(),
                                      d["beta"][:, t].contiguous(), yt, N, Hk, H, S, cfg.scale)
            y[:, t] = yt
        return y
    args = (st, d["q"], d["k"], d["v"], d["g"], d["beta"], y, N, T, Hk, H, S, cfg.scale)
    if form == "scan":
        lib.gdn_recurrence_scan(*args)
    elif form == "chunked":
        lib.gdn_recurrence_scan_chunked(*args)
    else:
        ws = torch.empty(lib.gdn_recurrence_scan_chunked_ws_size(N, T, H, S) // 4, device="cuda")
        lib.gdn_recurrence_scan_chunked_ws(*args, ws)
    return y


def case(T, seed):
    cfg = I.get_config(0, n_k_heads=2, n_v_heads=4, state_size=128, n_seqs=2, n_tokens=T,
                       cid=880 + seed)
    return cfg, I.recurrence_batch(cfg), I.state_pool(cfg)


@pytest.mark.parametrize("form", FORMS)
def test_identity_steps_leave_the_state_bitwise(lib, form):
    cfg, x, st0 = case(40, 1)
    x["beta"] = np.zeros_like(x["beta"])
    x["g"] = np.zeros_like(x["g"])
    st = dev(st0)
    y = run_form(lib, form, cfg, x, st)
    np.testing.assert_array_equal(host(st), st0)
    # y_t = scale * S^T q_t with S the initial state (transposed layout: row j = S[:, j])
    kh = np.arange(cfg.n_v_heads) % cfg.n_k_heads
    want = cfg.scale * np.einsum("nhji,nthi->nthj", st0.astype(np.float64),
                                 x["q"][:, :, kh].astype(np.float64))
    got = host(y).astype(np.float64)
    assert np.abs(got - want).max() <= 1e-5 * (1 + np.abs(want).max())


@pytest.mark.parametrize("form", FORMS)
def test_zero_query_reads_zero(lib, form):
    cfg, x, st0 = case(33, 2)
    x["q"] = np.zeros_like(x["q"])
    y = run_form(lib, form, cfg, x, dev(st0))
    assert np.all(host(y) == 0.0)


@pytest.mark.parametrize("form", FORMS)
def test_zero_key_only_decays(lib, form):
    cfg, x, st0 = case(37, 3)
    x["k"] = np.zeros_like(x["k"])
    st = dev(st0)
    run_form(lib, form, cfg, x, st)
    total = x["g"].astype(np.float64).sum(axis=1)  # [N][H]
    want = np.exp(total)[:, :, None, None] * st0.astype(np.float64)
    got = host(st).astype(np.float64)
    assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max() * math.sqrt(37)
