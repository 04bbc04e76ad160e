"""GPU unit test of the tcgen05 building blocks (gdn_tc.cuh) on a single tile.

D[128 x N] = A[128 x 32] B[N x 32]^T on the tensor cores: one tf32 pass must
equal the product of tf32-rounded inputs (up to accumulation order), and the
three-pass hi/lo split must match the fp64 product to fp32 accuracy; A comes
from shared memory (N = 64) or from tensor memory (N = 32, 128). The bf16 form
(kind::f16): one pass equals the product of bf16-rounded inputs (nearest, ties to
even), and the three-pass bf16 hi/lo split stays within its 3 * 2^-16 relative
bound of the fp64 product, A from shared or tensor memory, N = 32 .. 160 (the
shapes the chunked scans issue).
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gated_deltanet_linear_scan_gb300", "csrc")


@pytest.fixture(scope="module")
def tclib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("tc") / "libtc_gemm_test.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-shared", "-Xcompiler", "-fPIC", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "cuda", "tc_gemm_test.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.tc_gemm_test.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_void_p]
    lib.tc_gemm_test.restype = ctypes.c_int
    lib.tc_gemm_ts_test.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 2
    lib.tc_gemm_ts_test.restype = ctypes.c_int
    lib.tc_gemm_bf16_test.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    lib.tc_gemm_bf16_test.restype = ctypes.c_int
    return lib


def tf32_round(x):
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x1000) & 0xFFFFE000  # nearest, ties away from zero (magnitude bits)
    return b.astype(np.uint32).view(np.float32)


def run(tclib, A, B, split):
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dD = torch.full((128, 64), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = tclib.tc_gemm_test(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), split, st.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0, "the MMA completion wait gave up"
    return dD.cpu().numpy()


def test_single_pass_tf32(tclib):
    r = np.random.default_rng(1)
    A = r.normal(0, 1, (128, 32)).astype(np.float32)
    B = r.normal(0, 1, (64, 32)).astype(np.float32)
    D = run(tclib, A, B, 0)
    want = tf32_round(A).astype(np.float64) @ tf32_round(B).astype(np.float64).T
    np.testing.assert_allclose(D, want, rtol=0, atol=1e-4)


def test_three_pass_split_tf32(tclib):
    r = np.random.default_rng(2)
    A = r.normal(0, 1, (128, 32)).astype(np.float32)
    B = r.normal(0, 1, (64, 32)).astype(np.float32)
    D = run(tclib, A, B, 1)
    want = A.astype(np.float64) @ B.astype(np.float64).T
    np.testing.assert_allclose(D, want, rtol=0, atol=2e-5)
    single = run(tclib, A, B, 0)
    assert np.abs(single - want).max() > 10 * np.abs(D - want).max()


def run_ts(tclib, A, B, split):
    n = B.shape[0]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dD = torch.full((128, n), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = tclib.tc_gemm_ts_test(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), n, split,
                               st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0, "the MMA completion wait gave up"
    return dD.cpu().numpy()


@pytest.mark.parametrize("n", [32, 128])
def test_a_from_tensor_memory(tclib, n):
    r = np.random.default_rng(3 + n)
    A = r.normal(0, 1, (128, 32)).astype(np.float32)
    B = r.normal(0, 1, (n, 32)).astype(np.float32)
    want = A.astype(np.float64) @ B.astype(np.float64).T
    D1 = run_ts(tclib, A, B, 0)
    np.testing.assert_allclose(D1, tf32_round(A).astype(np.float64)
                               @ tf32_round(B).astype(np.float64).T, rtol=0, atol=1e-4)
    D3 = run_ts(tclib, A, B, 1)
    np.testing.assert_allclose(D3, want, rtol=0, atol=2e-5)


def bf16_round(x):
    """Nearest bf16 value, ties to even, as float32."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def run_bf16(tclib, A, B, a_tmem, split):
    n = B.shape[0]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dD = torch.full((128, n), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = tclib.tc_gemm_bf16_test(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), n, a_tmem, split,
                                 st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert st.item() == 0, "the MMA completion wait gave up"
    return dD.cpu().numpy().astype(np.float64)


def test_bf16_round_helper():
    """The host rounding used below: ties go to the even neighbour, others to the nearest."""
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -9, -(1 + 2.0 ** -8 + 2.0 ** -20)],
                 np.float32)
    np.testing.assert_array_equal(bf16_round(x), np.array([1, 1 + 2.0 ** -6, 1, -(1 + 2.0 ** -7)],
                                                          np.float32))


@pytest.mark.parametrize("n", [32, 64, 128, 160])
@pytest.mark.parametrize("a_tmem", [0, 1])
def test_bf16_products(tclib, n, a_tmem):
    r = np.random.default_rng(40 + n + a_tmem)
    A = r.normal(0, 1, (128, 32)).astype(np.float32)
    B = r.normal(0, 1, (n, 32)).astype(np.float32)
    exact = A.astype(np.float64) @ B.astype(np.float64).T
    mag = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
    D1 = run_bf16(tclib, A, B, a_tmem, 0)
    want1 = bf16_round(A).astype(np.float64) @ bf16_round(B).astype(np.float64).T
    np.testing.assert_allclose(D1, want1, rtol=0, atol=1e-4)
    D3 = run_bf16(tclib, A, B, a_tmem, 1)
    err3 = np.abs(D3 - exact)
    assert np.all(err3 <= 4 * 2.0 ** -16 * mag + 1e-6), f"max excess {(err3 - 4 * 2.0 ** -16 * mag).max()}"
    assert np.abs(D1 - exact).max() > 10 * err3.max()
