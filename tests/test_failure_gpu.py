"""Failure detection on the GPU without a fault: the bounded-wait path.

Every kernel that waits on its own asynchronous copies bounds the wait; a wait that
gives up skips the work it guarded and raises a device flag that gdn_device_error()
reads and clears. gdn_selftest_bounded_wait makes such a wait run out on purpose (an
mbarrier armed for bytes no copy brings, bounded at a millisecond here) in each of the
library's flags in turn. The test checks that the give-up is reported once, that the
guarded write did not happen, that an unarmed probe completes, and that the context
stays usable for real work afterwards. Nothing faults, traps or hangs.
"""
import numpy as np
import pytest

import oracle
from gated_deltanet_linear_scan_gb300 import inputs as I

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

GDN_OK, GDN_ERR_DEVICE = 0, 6


def status(lib):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.library().gdn_device_error(stream)


@pytest.mark.parametrize("probe", range(4))
def test_bounded_wait_runs_out_and_is_reported(cuda_lib, probe):
    assert status(cuda_lib) == GDN_OK  # nothing pending from earlier work
    out = torch.full((4,), 5.0, device="cuda")
    cuda_lib.gdn_selftest_bounded_wait(1 << probe, 1000, out)  # 1 ms bound
    assert status(cuda_lib) == GDN_ERR_DEVICE
    assert status(cuda_lib) == GDN_OK  # read and cleared
    got = out.cpu().numpy()
    assert got[probe] == 5.0, "the armed probe's guarded write happened"
    others = [i for i in range(4) if i != probe]
    assert np.all(got[others] == 1.0), "an unarmed probe did not complete"


def test_no_probe_armed_reports_nothing(cuda_lib):
    out = torch.zeros(4, device="cuda")
    cuda_lib.gdn_selftest_bounded_wait(0, 1000, out)
    assert status(cuda_lib) == GDN_OK
    assert torch.all(out == 1.0)


def test_all_probes_armed_then_real_work(cuda_lib):
    """After every flag was raised and cleared, a decode step still matches the oracle."""
    out = torch.full((4,), 5.0, device="cuda")
    cuda_lib.gdn_selftest_bounded_wait(15, 1000, out)
    assert status(cuda_lib) == GDN_ERR_DEVICE
    assert status(cuda_lib) == GDN_OK
    assert torch.all(out == 5.0)
    cfg = I.get_config(0, n_seqs=2, cid=990)
    x = I.recurrence_batch(cfg, n_tokens=1)
    st0 = I.state_pool(cfg)
    st = torch.from_numpy(st0).cuda()
    y = torch.zeros(2, cfg.n_v_heads, cfg.state_size, device="cuda")
    d = {k: torch.from_numpy(np.ascontiguousarray(v[:, 0])).cuda() for k, v in x.items()}
    cuda_lib.gdn_recurrence_decode(st, d["q"], d["k"], d["v"], d["g"], d["beta"], y, 2,
                                   cfg.n_k_heads, cfg.n_v_heads, cfg.state_size, cfg.scale)
    ref_st = np.ascontiguousarray(st0, dtype=np.float64)
    y_ref, _ = oracle.recurrence(ref_st, x["q"], x["k"], x["v"], x["g"], x["beta"], cfg.scale)
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - y_ref[:, 0])
    assert np.all(err <= 1e-4 + 1e-4 * np.abs(y_ref[:, 0]))
    assert status(cuda_lib) == GDN_OK
