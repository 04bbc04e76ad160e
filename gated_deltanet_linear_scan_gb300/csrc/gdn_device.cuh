// gdn_device.cuh -- device helpers shared by the sm_103a kernels: inline PTX for
// mbarriers, bulk (TMA) copies and thread-block clusters, bounded waits, and the
// warp reductions of the delta-rule row step.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gdn {

constexpr unsigned FULL_MASK = 0xffffffffu;
// Upper bound of any wait on an asynchronous copy, in globaltimer nanoseconds.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// Watchdog bits raised in a kernel's device flag when a bounded wait gives up.
constexpr unsigned WD_STATE_COPY = 1u;   // state tile bulk copy
constexpr unsigned WD_STAGE_COPY = 2u;   // per-token operand stage
constexpr unsigned WD_STAGE_FREE = 4u;   // consumer release of a stage

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// A waiting thread is suspended in hardware (not spinning on the issue slots of the
// warps that do work) until the phase completes or this many nanoseconds pass.
constexpr uint32_t kTryWaitSuspendNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kTryWaitSuspendNs)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, for at most limit_ns. Returns false
// if it gave up.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// The bounded wait of every kernel here: at most WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, WAIT_LIMIT_NS);
}

// Self-test of the bounded-wait path (one thread): arms an mbarrier for `bytes` that no
// copy will bring when `arm` is set (a plain arrival completes the phase otherwise),
// waits at most limit_ns, and on giving up raises `bit` in `flag` and leaves `out`
// alone, as a kernel's guarded work is skipped; a completed wait writes 1 to out[0].
// Nothing follows the wait that could block, so the thread always returns.
__device__ __forceinline__ void bounded_wait_probe(bool arm, uint64_t limit_ns, unsigned *flag,
                                                   unsigned bit, float *out) {
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (arm) mbar_arrive_expect_tx(&bar, 16);
    else mbar_arrive(&bar);
    if (mbar_wait_for(&bar, 0, limit_ns)) {
        out[0] = 1.0f;
    } else {
        atomicOr(flag, bit);
    }
}

// The same bounded wait for a thread that shares its SM sub-partition with warps
// doing arithmetic: between polls it sleeps (backing off from 32 ns to max_sleep_ns),
// so it takes next to no issue slots; the cost is up to max_sleep_ns of extra latency.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity,
                                                unsigned max_sleep_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    unsigned ns = 32;
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
        __nanosleep(ns);
        ns = ns < max_sleep_ns ? 2 * ns : max_sleep_ns;
    }
    return true;
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar` in bytes.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared by one thread (the non-bulk form: a warp
// moves 512 contiguous bytes with one instruction, where a bulk copy per lane costs
// the issuing thread tens of cycles per copy). Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

// Arrive on `bar` once every cp_async16 this thread issued before has landed. The
// arrival is not counted in advance (.noinc): `bar`'s expected count includes it.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier `id` over `count` threads (a multiple of 32), leaving the other warps
// of the CTA free to run.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- thread-block clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Reads a float from the shared memory of CTA `rank` of this cluster, at the
// offset `local` has in this CTA's shared memory.
__device__ __forceinline__ float ld_shared_cluster(const float *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ------------------------------------------------------------------ math

// SiLU in the divisor form, x / (1 + exp(-x)), with CUDA's fast exponential and fast
// division intrinsics: a few ulp at the magnitudes a conv output takes, against the
// 1e-4 relative bound of one step; where exp(-x) overflows (x below about -88) the
// quotient is a signed zero, the exact value being below 1e-36 in magnitude. Every
// kernel calls this one function, so the fused and stand-alone paths keep the same
// bits. (The IEEE division and expf cost three times the instructions and made the
// prefill block's conv pass issue-bound.)
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ float softplus_guarded(float v) {
    return v > 20.0f ? v : log1pf(expf(v));
}

// ------------------------------------------------------------------ reductions

// Sum over the 32 lanes; every lane returns the identical value (each butterfly
// step adds the same two operands on both partner lanes, and fp addition is
// commutative bit for bit).
__device__ __forceinline__ float warp_allsum(float p) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) p = __fadd_rn(p, __shfl_xor_sync(FULL_MASK, p, m));
    return p;
}

// Lane partial of a length-(32*E) dot: lane L holds elements [E*L, E*L + E).
// Explicit _rn intrinsics keep the compiler from re-contracting the chain, so
// every kernel that calls this gets the same bits.
template <int E>
__device__ __forceinline__ float lane_dot(const float (&a)[E], const float (&b)[E]) {
    float p = __fmul_rn(a[0], b[0]);
#pragma unroll
    for (int e = 1; e < E; ++e) p = __fmaf_rn(a[e], b[e], p);
    return p;
}

// Packed butterfly over R = 2^m independent lane partials (rows). At butterfly
// levels 16, 8, ... the partner lanes split the work: the lane whose level bit
// is clear keeps the even row and sends the odd one, so one shuffle serves two
// rows. Each row's sum is formed with exactly the operand pairs of warp_allsum,
// hence bit-identical to it. After the call, row r's sum sits in every lane whose
// bits (4, 3, ..., 5-m) spell r (bit 4 = r's bit 0); row_home_lane(r) names one.
template <int R>
__device__ __forceinline__ float warp_sum_packed(float (&p)[R], int lane) {
    static_assert(R == 1 || R == 2 || R == 4 || R == 8, "R must be 1, 2, 4 or 8");
    constexpr int LEVELS = (R == 1) ? 0 : (R == 2) ? 1 : (R == 4) ? 2 : 3;
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = p[r];
    int n = R;
#pragma unroll
    for (int lv = 0; lv < LEVELS; ++lv) {
        const int m = 16 >> lv;
        const bool hi = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
            if (2 * i + 1 < n) {
                const float keep = hi ? v[2 * i + 1] : v[2 * i];
                const float send = hi ? v[2 * i] : v[2 * i + 1];
                v[i] = __fadd_rn(keep, __shfl_xor_sync(FULL_MASK, send, m));
            }
        }
        n >>= 1;
    }
    float acc = v[0];
#pragma unroll
    for (int m = 16 >> LEVELS; m >= 1; m >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(FULL_MASK, acc, m));
    return acc;
}

template <int R>
__device__ __forceinline__ int row_home_lane(int r) {
    int lane = 0;
    if (R >= 2) lane |= (r & 1) << 4;
    if (R >= 4) lane |= ((r >> 1) & 1) << 3;
    if (R >= 8) lane |= ((r >> 2) & 1) << 2;
    return lane;
}

// Full sums of R rows in every lane (packed butterfly, then R broadcasts).
template <int R>
__device__ __forceinline__ void warp_allsum_rows(float (&p)[R], int lane) {
    const float s = warp_sum_packed<R>(p, lane);
    if constexpr (R == 1) {
        p[0] = s;  // a plain butterfly already leaves the sum in every lane
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r) p[r] = __shfl_sync(FULL_MASK, s, row_home_lane<R>(r));
    }
}

// ------------------------------------------------------------------ the row step

// One token of the delta-rule update for R state rows held by a warp (lane L
// holds cells [E*L, E*L+E) of each row), in the order of fm_kernel_ssm.m,
// "Delta-rule recurrence -- register-resident":
//   row *= decay; pred = row.k; delta = (v - pred) * beta; row += k * delta;
//   y = scale * (row . q)   (after the write)
// Returns, in every lane, the packed readout sum; row r's y is scale * that sum
// in lane row_home_lane<R>(r). v[r] is the v element of row r.
template <int E, int R>
__device__ __forceinline__ float row_step(float (&row)[R][E], const float (&k)[E],
                                          const float (&q)[E], const float (&v)[R], float decay,
                                          float beta, int lane) {
    float part[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int e = 0; e < E; ++e) row[r][e] = __fmul_rn(row[r][e], decay);
        part[r] = lane_dot<E>(row[r], k);
    }
    warp_allsum_rows<R>(part, lane);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float delta = __fmul_rn(__fsub_rn(v[r], part[r]), beta);
#pragma unroll
        for (int e = 0; e < E; ++e) row[r][e] = __fmaf_rn(k[e], delta, row[r][e]);
        part[r] = lane_dot<E>(row[r], q);
    }
    return warp_sum_packed<R>(part, lane);
}

// The same token with the readout factorised (ssm_gated_delta.cu, "T4: 3-pass ->
// 2-pass state-access factorization"): with r the decayed row,
//   y = scale * (r_new . q) = scale * (r . q + delta * (k . q)),
// so both dots reduce off the same decayed row and the second no longer waits for
// the update. `kq` is k . q of the token (the same for every row). The state update
// is the row step's, bit for bit; y differs from it by rounding only. Returns
// scale * y in lane row_home_lane<R>(r) for row r.
template <int E, int R>
__device__ __forceinline__ float row_step_factored(float (&row)[R][E], const float (&k)[E],
                                                   const float (&q)[E], const float (&v)[R],
                                                   float decay, float beta, float kq, float scale,
                                                   int lane) {
    float pk[R], pq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int e = 0; e < E; ++e) row[r][e] = __fmul_rn(row[r][e], decay);
        pk[r] = lane_dot<E>(row[r], k);
        pq[r] = lane_dot<E>(row[r], q);
    }
    warp_allsum_rows<R>(pk, lane);
    const float oq = warp_sum_packed<R>(pq, lane);
    float my_delta = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float delta = __fmul_rn(__fsub_rn(v[r], pk[r]), beta);
#pragma unroll
        for (int e = 0; e < E; ++e) row[r][e] = __fmaf_rn(k[e], delta, row[r][e]);
        if (row_home_lane<R>(r) == (lane & (R == 1 ? 0 : R == 2 ? 16 : R == 4 ? 24 : 28)))
            my_delta = delta;
    }
    return __fmul_rn(scale, __fmaf_rn(my_delta, kq, oq));
}

// ------------------------------------------------------------------ vector memory

template <int E>
__device__ __forceinline__ void load_vec(float (&dst)[E], const float *src) {
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src + e);
            dst[e] = t.x; dst[e + 1] = t.y; dst[e + 2] = t.z; dst[e + 3] = t.w;
        }
    } else if constexpr (E == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(src);
        dst[0] = t.x; dst[1] = t.y;
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = src[e];
    }
}

template <int E>
__device__ __forceinline__ void store_vec(float *dst, const float (&src)[E]) {
    if constexpr (E % 4 == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(src[e], src[e + 1], src[e + 2], src[e + 3]);
    } else if constexpr (E == 2) {
        *reinterpret_cast<float2 *>(dst) = make_float2(src[0], src[1]);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = src[e];
    }
}

}  // namespace gdn
