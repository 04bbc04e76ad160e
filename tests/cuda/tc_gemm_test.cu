// Unit test of the tcgen05 building blocks in gdn_tc.cuh: one CTA computes
// D[128 x N] = A[128 x 32] * B[N x 32]^T on the tensor cores with tf32 inputs
// (one pass) or the hi/lo split (three passes), accumulator in tensor memory,
// with A in shared memory (N = 64) or in tensor memory (N = 32 or 128); and the
// same with bf16 operands (kind::f16), A in shared or tensor memory, N = 32 .. 160.
// Built by tests/test_tc_primitives.py into its own shared library.
#include <cstdint>

#include "gdn_tc.cuh"

namespace {

constexpr int M = 128, N = 64, K = 32;
constexpr uint32_t LBO = 128;             // next 4 elements of K
constexpr uint32_t SBO = (K / 4) * 128;   // next 8 rows

__global__ void __launch_bounds__(128) tc_gemm_kernel(const float *__restrict__ A,
                                                      const float *__restrict__ B,
                                                      float *__restrict__ D, int split,
                                                      int *status) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *a_hi = smem, *a_lo = smem + M * K * 4;
    unsigned char *b_hi = a_lo + M * K * 4, *b_lo = b_hi + N * K * 4;
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_taddr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int i = tid; i < M * K; i += 128) {
        const int r = i / K, k = i % K;
        float hi, lo;
        gdn::tc::split_tf32(A[i], hi, lo);
        const uint32_t off = gdn::tc::kmajor_offset(r, k, LBO, SBO);
        *reinterpret_cast<float *>(a_hi + off) = hi;
        *reinterpret_cast<float *>(a_lo + off) = lo;
    }
    for (int i = tid; i < N * K; i += 128) {
        const int r = i / K, k = i % K;
        float hi, lo;
        gdn::tc::split_tf32(B[i], hi, lo);
        const uint32_t off = gdn::tc::kmajor_offset(r, k, LBO, SBO);
        *reinterpret_cast<float *>(b_hi + off) = hi;
        *reinterpret_cast<float *>(b_lo + off) = lo;
    }
    gdn::fence_proxy_async_smem();  // generic-proxy writes -> tensor core reads
    if (tid == 0) {
        gdn::mbar_init(&bar, 1);
        gdn::fence_mbar_init();
    }
    if (warp == 0) {
        gdn::tc::tmem_alloc(&s_taddr, 64);
        gdn::tc::tmem_relinquish();
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    gdn::tc::fence_after_sync();
    const uint32_t taddr = s_taddr;

    if (tid == 0) {
        const uint32_t idesc = gdn::tc::idesc_tf32(M, N);
        const unsigned char *as[3] = {a_hi, a_hi, a_lo};
        const unsigned char *bs[3] = {b_hi, b_lo, b_hi};
        const int passes = split ? 3 : 1;
        for (int p = 0; p < passes; ++p)
            for (int ks = 0; ks < K / 8; ++ks) {
                const uint64_t ad = gdn::tc::smem_desc(as[p] + ks * 2 * LBO, LBO, SBO);
                const uint64_t bd = gdn::tc::smem_desc(bs[p] + ks * 2 * LBO, LBO, SBO);
                gdn::tc::mma_tf32(taddr, ad, bd, idesc, p > 0 || ks > 0);
            }
        gdn::tc::mma_commit(&bar);
    }
    const bool done = gdn::mbar_wait(&bar, 0);
    if (!done && lane == 0) atomicOr(status, 1);
    gdn::tc::fence_after_sync();
    if (done) {
        const uint32_t tw = taddr + (static_cast<uint32_t>(32 * warp) << 16);
        for (int cb = 0; cb < N / 16; ++cb) {
            float v[16];
            gdn::tc::tmem_ld16(tw + cb * 16, v);
            for (int i = 0; i < 16; ++i) D[(32 * warp + lane) * N + cb * 16 + i] = v[i];
        }
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) gdn::tc::tmem_dealloc(taddr, 64);
}

// A in tensor memory: thread t (lanes of warp t/32) writes row t of A, hi part to
// columns [0, 32), lo part to [32, 64); D occupies columns [64, 64 + NN).
template <int NN>
__global__ void __launch_bounds__(128) tc_gemm_ts_kernel(const float *__restrict__ A,
                                                         const float *__restrict__ B,
                                                         float *__restrict__ D, int split,
                                                         int *status) {
    constexpr uint32_t kCols = NN + 64 <= 128 ? 128 : 256;
    constexpr uint32_t kSbo = (K / 4) * 128;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *b_hi = smem, *b_lo = smem + NN * K * 4;
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_taddr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int i = tid; i < NN * K; i += 128) {
        const int r = i / K, k = i % K;
        float hi, lo;
        gdn::tc::split_tf32(B[i], hi, lo);
        const uint32_t off = gdn::tc::kmajor_offset(r, k, LBO, kSbo);
        *reinterpret_cast<float *>(b_hi + off) = hi;
        *reinterpret_cast<float *>(b_lo + off) = lo;
    }
    gdn::fence_proxy_async_smem();
    if (tid == 0) {
        gdn::mbar_init(&bar, 1);
        gdn::fence_mbar_init();
    }
    if (warp == 0) {
        gdn::tc::tmem_alloc(&s_taddr, kCols);
        gdn::tc::tmem_relinquish();
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    gdn::tc::fence_after_sync();
    const uint32_t taddr = s_taddr;
    const uint32_t tw = taddr + (static_cast<uint32_t>(32 * warp) << 16);
    {
        uint32_t hi[32], lo[32];
        for (int k = 0; k < K; ++k) {
            float h, l;
            gdn::tc::split_tf32(A[tid * K + k], h, l);
            hi[k] = __float_as_uint(h);
            lo[k] = __float_as_uint(l);
        }
        gdn::tc::tmem_st32(tw, hi);
        gdn::tc::tmem_st32(tw + 32, lo);
        gdn::tc::tmem_st_wait();
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    gdn::tc::fence_after_sync();

    if (tid == 0) {
        const uint32_t idesc = gdn::tc::idesc_tf32(M, NN);
        const uint32_t acol[3] = {0, 0, 32};
        const unsigned char *bs[3] = {b_hi, b_lo, b_hi};
        const int passes = split ? 3 : 1;
        for (int p = 0; p < passes; ++p)
            for (int ks = 0; ks < K / 8; ++ks) {
                const uint64_t bd = gdn::tc::smem_desc(bs[p] + ks * 2 * LBO, LBO, kSbo);
                gdn::tc::mma_tf32_ts(taddr + 64, taddr + acol[p] + ks * 8, bd, idesc,
                                     p > 0 || ks > 0);
            }
        gdn::tc::mma_commit(&bar);
    }
    const bool done = gdn::mbar_wait(&bar, 0);
    if (!done && lane == 0) atomicOr(status, 1);
    gdn::tc::fence_after_sync();
    if (done) {
        for (int cb = 0; cb < NN / 32; ++cb) {
            uint32_t v[32];
            gdn::tc::tmem_ld32_nowait(tw + 64 + cb * 32, v);
            gdn::tc::tmem_ld_wait();
            for (int i = 0; i < 32; ++i) D[(32 * warp + lane) * NN + cb * 32 + i] = __uint_as_float(v[i]);
        }
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) gdn::tc::tmem_dealloc(taddr, kCols);
}

// bf16 operands: A and B split into bf16 hi / lo parts (split_bf16x2); one pass
// (hi * hi) or three (hi * hi + hi * lo + lo * hi). B in shared memory (K-major,
// 16-bit core matrices); A in shared memory (a_tmem = 0) or in tensor memory (hi at
// columns [0, 16), lo at [16, 32), two elements to a column); D at column 32.
template <int NN>
__global__ void __launch_bounds__(128) tc_gemm_bf16_kernel(const float *__restrict__ A,
                                                           const float *__restrict__ B,
                                                           float *__restrict__ D, int a_tmem,
                                                           int split, int *status) {
    constexpr uint32_t kSbo = (K / 8) * 128;  // next 8 rows of a K = 32 bf16 operand
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *a_hi = smem, *a_lo = smem + M * K * 2;
    unsigned char *b_hi = a_lo + M * K * 2, *b_lo = b_hi + NN * K * 2;
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_taddr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // pairs (k, k + 1) of a row, k even: both halves of one packed word
    for (int i = tid; i < M * K / 2; i += 128) {
        const int r = i / (K / 2), k = 2 * (i % (K / 2));
        uint32_t hi, lo;
        gdn::tc::split_bf16x2(A[r * K + k], A[r * K + k + 1], hi, lo);
        const uint32_t off = gdn::tc::kmajor_offset16(r, k, LBO, kSbo);
        *reinterpret_cast<uint32_t *>(a_hi + off) = hi;
        *reinterpret_cast<uint32_t *>(a_lo + off) = lo;
    }
    for (int i = tid; i < NN * K / 2; i += 128) {
        const int r = i / (K / 2), k = 2 * (i % (K / 2));
        uint32_t hi, lo;
        gdn::tc::split_bf16x2(B[r * K + k], B[r * K + k + 1], hi, lo);
        const uint32_t off = gdn::tc::kmajor_offset16(r, k, LBO, kSbo);
        *reinterpret_cast<uint32_t *>(b_hi + off) = hi;
        *reinterpret_cast<uint32_t *>(b_lo + off) = lo;
    }
    gdn::fence_proxy_async_smem();
    if (tid == 0) {
        gdn::mbar_init(&bar, 1);
        gdn::fence_mbar_init();
    }
    if (warp == 0) {
        gdn::tc::tmem_alloc(&s_taddr, 256);
        gdn::tc::tmem_relinquish();
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    gdn::tc::fence_after_sync();
    const uint32_t taddr = s_taddr;
    const uint32_t tw = taddr + (static_cast<uint32_t>(32 * warp) << 16);
    if (a_tmem) {  // row tid of A: hi to columns 0..15, lo to 16..31
        uint32_t hi[16], lo[16];
        for (int c = 0; c < K / 2; ++c)
            gdn::tc::split_bf16x2(A[tid * K + 2 * c], A[tid * K + 2 * c + 1], hi[c], lo[c]);
        gdn::tc::tmem_st16(tw, hi);
        gdn::tc::tmem_st16(tw + 16, lo);
        gdn::tc::tmem_st_wait();
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    gdn::tc::fence_after_sync();

    if (tid == 0) {
        const uint32_t idesc = gdn::tc::idesc_bf16(M, NN);
        const unsigned char *as[3] = {a_hi, a_hi, a_lo};
        const uint32_t acol[3] = {0, 0, 16};
        const unsigned char *bs[3] = {b_hi, b_lo, b_hi};
        const int passes = split ? 3 : 1;
        for (int p = 0; p < passes; ++p)
            for (int ks = 0; ks < K / 16; ++ks) {
                const uint64_t bd = gdn::tc::smem_desc(bs[p] + ks * 2 * LBO, LBO, kSbo);
                if (a_tmem) {
                    gdn::tc::mma_bf16_ts(taddr + 32, taddr + acol[p] + ks * 8, bd, idesc,
                                         p > 0 || ks > 0);
                } else {
                    const uint64_t ad = gdn::tc::smem_desc(as[p] + ks * 2 * LBO, LBO, kSbo);
                    gdn::tc::mma_bf16(taddr + 32, ad, bd, idesc, p > 0 || ks > 0);
                }
            }
        gdn::tc::mma_commit(&bar);
    }
    const bool done = gdn::mbar_wait(&bar, 0);
    if (!done && lane == 0) atomicOr(status, 1);
    gdn::tc::fence_after_sync();
    if (done) {
        for (int cb = 0; cb < NN / 16; ++cb) {
            float v[16];
            gdn::tc::tmem_ld16(tw + 32 + cb * 16, v);
            for (int i = 0; i < 16; ++i) D[(32 * warp + lane) * NN + cb * 16 + i] = v[i];
        }
    }
    gdn::tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) gdn::tc::tmem_dealloc(taddr, 256);
}

template <int NN>
int launch_bf16(const float *A, const float *B, float *D, int a_tmem, int split, int *status,
                cudaStream_t st) {
    const int smem = (M + NN) * K * 2 * 2;
    cudaFuncSetAttribute(tc_gemm_bf16_kernel<NN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    tc_gemm_bf16_kernel<NN><<<1, 128, smem, st>>>(A, B, D, a_tmem, split, status);
    return static_cast<int>(cudaGetLastError());
}

}  // namespace

extern "C" int tc_gemm_bf16_test(const float *A, const float *B, float *D, int n, int a_tmem,
                                 int split, int *status, void *stream) {
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (n) {
        case 32: return launch_bf16<32>(A, B, D, a_tmem, split, status, st);
        case 64: return launch_bf16<64>(A, B, D, a_tmem, split, status, st);
        case 128: return launch_bf16<128>(A, B, D, a_tmem, split, status, st);
        case 160: return launch_bf16<160>(A, B, D, a_tmem, split, status, st);
        default: return -1;
    }
}

extern "C" int tc_gemm_test(const float *A, const float *B, float *D, int split, int *status,
                            void *stream) {
    const int smem = (M + N) * K * 4 * 2;
    cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    tc_gemm_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(A, B, D, split, status);
    return static_cast<int>(cudaGetLastError());
}

extern "C" int tc_gemm_ts_test(const float *A, const float *B, float *D, int n, int split,
                               int *status, void *stream) {
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int smem = n * K * 4 * 2;
    if (n == 32) {
        cudaFuncSetAttribute(tc_gemm_ts_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        tc_gemm_ts_kernel<32><<<1, 128, smem, st>>>(A, B, D, split, status);
    } else if (n == 128) {
        cudaFuncSetAttribute(tc_gemm_ts_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        tc_gemm_ts_kernel<128><<<1, 128, smem, st>>>(A, B, D, split, status);
    } else {
        return -1;
    }
    return static_cast<int>(cudaGetLastError());
}
