// Unit test of the tcgen05 building blocks in gdn_tc.cuh: one CTA computes
// D[128 x 64] = A[128 x 32] * B[64 x 32]^T on the tensor cores with tf32 inputs
// (one pass) or the hi/lo split (three passes), accumulator in tensor memory.
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

}  // namespace

extern "C" int tc_gemm_test(const float *A, const float *B, float *D, int split, int *status,
                            void *stream) {
    const int smem = (M + N) * K * 4 * 2;
    cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    tc_gemm_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(A, B, D, split, status);
    return static_cast<int>(cudaGetLastError());
}
