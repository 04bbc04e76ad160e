// gdn_chunked.cu -- the multi-token scan of the delta-rule recurrence in chunks of
// 32 positions, with the state-dependent contractions on the 5th-generation tensor
// cores (tcgen05, TF32 inputs, fp32 accumulation in tensor memory).
//
// fm_kernel_ssm.m (its softplus note and the sequential-scan section) speaks of a
// chunked prefill path that takes cumulative sums of g along each chunk, with the
// sequential scan kept as its permanent reference; the pages do not spell the
// chunked algebra out. The form used here is derived from the recurrence itself
// (the WY/UT representation of a product of generalised Householder steps). Per
// (sequence, v-head) and chunk of positions t = 0..31 with log-decays g_t, write
// gam_t = g_0 + .. + g_t,
// Gam_t = exp(gam_t), S the state at the chunk start as a [dk][dv] matrix, and
//   A[t][s] = beta_t exp(gam_t - gam_s) (k_t . k_s)        (s < t, else 0)
//   (I + A) W  = diag(beta Gam) K,   (I + A) Ut = diag(beta) V   (forward substitution)
//   U  = Ut - W S                                            (the per-position delta)
//   y_t = scale (Gam_t q_t^T S + sum_{s<=t} exp(gam_t - gam_s) (q_t . k_s) u_s)
//   S' = Gam_31 S + sum_s exp(gam_31 - gam_s) k_s u_s^T.
// This is the recurrence of the sequential scan regrouped exactly (no truncation
// or approximation); only the rounding differs.
//
// Two kernels:
//  1. chunk_prep_kernel (one CTA per (sequence, v-head, chunk), all in parallel,
//     fp32 on the CUDA cores): gam, the Gram products, the forward substitution,
//     and a record holding the tensor-core operands of the chunk, laid out as the
//     shared-memory image the second kernel copies in with one bulk copy:
//        W          [32 c][128 dk]         single tf32 pass operand
//        wK^T  hi/lo [128 dk][32 c]        exp(gam_31 - gam_c) k_c, split for 3 passes
//        QM    hi/lo [32 t][128 + 32]      (Gam_t q_t | exp(gam_t - gam_s)(q_t . k_s), s<=t)
//        Ut          [32 c][128 dv]        fp32, read by the CUDA cores
//        Gam_31
//  2. chunk_scan_kernel (one CTA per (sequence, v-head), sequential over chunks):
//     the state lives in tensor memory as S^T (lane = dv, column = dk) for the
//     whole scan; per chunk, four warps split it into tf32 hi/lo parts (also in
//     tensor memory, the A operand of the MMAs), one thread issues
//        D_u = S^T W^T                 (U^T = Ut^T - D_u, one tf32 pass)
//        D_y = S^T (Gam Q)^T + U^T M^T (three passes)
//        S^T <- Gam_31 S^T + U^T (wK)  (three passes, accumulated in place)
//     and the four warps turn D_u into U and D_y into y.
//
// Precision: a single TF32 pass (10-bit mantissa) in any product that feeds the
// state or y misses a 2e-3-of-RMS error bound after 4096 positions; the split
// x = hi + lo with hi*hi + hi*lo + lo*hi ("3xTF32") restores fp32-level products.
// Only W S tolerates one pass: its error enters U, which the delta rule corrects
// at the next write.
#include <mutex>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kC = 32;    // positions per chunk
constexpr int kS = 128;   // state size (dk = dv) of the tensor-core form
constexpr uint32_t kLbo = 128;  // K-major core matrices: next 4 elements of K

// Record / shared-memory stage layout (bytes).
constexpr uint32_t kSboW = (kS / 4) * 128;        // W: 32 rows x K = 128
constexpr uint32_t kSboK = (kC / 4) * 128;        // wK^T: 128 rows x K = 32
constexpr uint32_t kQmK = kS + kC;                // QM: K = 160
constexpr uint32_t kSboQ = (kQmK / 4) * 128;      // QM: 32 rows x K = 160
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffKhi = kOffW + kC * kS * 4;
constexpr uint32_t kOffKlo = kOffKhi + kS * kC * 4;
constexpr uint32_t kOffQhi = kOffKlo + kS * kC * 4;
constexpr uint32_t kOffQlo = kOffQhi + kC * kQmK * 4;
constexpr uint32_t kOffUt = kOffQlo + kC * kQmK * 4;
constexpr uint32_t kOffScal = kOffUt + kC * kS * 4;
constexpr uint32_t kRecord = kOffScal + 128;       // 106,624 bytes, a multiple of 128
static_assert(kRecord % 128 == 0, "records stay 128-byte aligned");


__device__ unsigned g_watchdog_chunked;

// ============================================================================ chunk prep
constexpr int kPrepThreads = 256;
constexpr int kRowPad = kS + 4;  // 132 floats: row r starts on bank 4r, float4 aligned

struct PrepSmem {
    float k[kC][kRowPad];   // k_t (k-head kh), zero past the end of the sequence
    float q[kC][kRowPad];
    float w[kC][kRowPad];   // W, from the forward substitution
    float v[kC][kS];        // v_t, overwritten in place by Ut
    float a[kC][kC + 1];    // A (strictly lower)
    float m[kC][kC];        // exp(gam_t - gam_s)(q_t . k_s), s <= t
    float gam[kC], Gam[kC], wdec[kC], beta[kC];
};

// One CTA per (chunk, v-head, sequence). Chunk positions past n_tokens are padded
// with k = q = v = 0, g = 0, beta = 0: an identity step that writes nothing.
__global__ void __launch_bounds__(kPrepThreads) chunk_prep_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    const float *__restrict__ g, const float *__restrict__ beta, unsigned char *__restrict__ ws,
    int n_tokens, int n_k_heads, int n_v_heads, const int32_t *__restrict__ slots, int pool) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(smem_raw);
    const int ci = blockIdx.x, vh = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = slots ? slots[n] : n;
    if (slot < 0 || slot >= pool) return;  // counted by the scan kernel
    const int H = n_v_heads, Hk = n_k_heads, kh = vh % Hk;
    const int n_chunks = gridDim.x;
    const int t0 = ci * kC, valid = min(kC, n_tokens - t0);

    // ---- inputs: 32 rows of k, q (k-head space) and v, as float4
    for (int idx = tid; idx < kC * kS / 4; idx += kPrepThreads) {
        const int t = idx / (kS / 4), c4 = (idx % (kS / 4)) * 4;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), qq = kk, vv = kk;
        if (t < valid) {
            const size_t row = static_cast<size_t>(n) * n_tokens + t0 + t;
            kk = *reinterpret_cast<const float4 *>(k + (row * Hk + kh) * kS + c4);
            qq = *reinterpret_cast<const float4 *>(q + (row * Hk + kh) * kS + c4);
            vv = *reinterpret_cast<const float4 *>(v + (row * H + vh) * kS + c4);
        }
        *reinterpret_cast<float4 *>(&sm.k[t][c4]) = kk;
        *reinterpret_cast<float4 *>(&sm.q[t][c4]) = qq;
        *reinterpret_cast<float4 *>(&sm.v[t][c4]) = vv;
    }
    // ---- cumulative log-decay within the chunk (warp 0, lane = position)
    if (warp == 0) {
        float gt = 0.f, bt = 0.f;
        if (lane < valid) {
            const size_t gi = (static_cast<size_t>(n) * n_tokens + t0 + lane) * H + vh;
            gt = g[gi];
            bt = beta[gi];
        }
        float c = gt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(FULL_MASK, c, off);
            if (lane >= off) c += o;
        }
        const float last = __shfl_sync(FULL_MASK, c, 31);
        sm.gam[lane] = c;
        sm.Gam[lane] = expf(c);
        sm.wdec[lane] = expf(last - c);
        sm.beta[lane] = bt;
    }
    __syncthreads();

    // ---- Gram products: thread -> row t = tid / 8, columns s = tid % 8 + 8 j
    {
        const int t = tid >> 3, s0 = tid & 7;
        float kk[4] = {0.f, 0.f, 0.f, 0.f}, qk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int i = 0; i < kS; i += 4) {
            const float4 kt = *reinterpret_cast<const float4 *>(&sm.k[t][i]);
            const float4 qt = *reinterpret_cast<const float4 *>(&sm.q[t][i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 ks = *reinterpret_cast<const float4 *>(&sm.k[s0 + 8 * j][i]);
                kk[j] = fmaf(kt.x, ks.x, kk[j]);
                kk[j] = fmaf(kt.y, ks.y, kk[j]);
                kk[j] = fmaf(kt.z, ks.z, kk[j]);
                kk[j] = fmaf(kt.w, ks.w, kk[j]);
                qk[j] = fmaf(qt.x, ks.x, qk[j]);
                qk[j] = fmaf(qt.y, ks.y, qk[j]);
                qk[j] = fmaf(qt.z, ks.z, qk[j]);
                qk[j] = fmaf(qt.w, ks.w, qk[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int s = s0 + 8 * j;
            const float e = s <= t ? expf(sm.gam[t] - sm.gam[s]) : 0.f;
            sm.a[t][s] = s < t ? sm.beta[t] * (e * kk[j]) : 0.f;
            sm.m[t][s] = e * qk[j];
        }
    }
    __syncthreads();

    // ---- forward substitution, one column per thread: W (threads 0..127) and Ut
    // (threads 128..255). Row t = base_t - sum_{s<t} A[t][s] row_s.
    {
        const int col = tid & (kS - 1);
        const bool is_w = tid < kS;
        float x[kC];
#pragma unroll
        for (int t = 0; t < kC; ++t) {
            float acc = is_w ? sm.beta[t] * sm.Gam[t] * sm.k[t][col] : sm.beta[t] * sm.v[t][col];
#pragma unroll
            for (int s = 0; s < t; ++s) acc = fmaf(-sm.a[t][s], x[s], acc);
            x[t] = acc;
        }
#pragma unroll
        for (int t = 0; t < kC; ++t) {
            if (is_w) sm.w[t][col] = x[t];
            else sm.v[t][col] = x[t];
        }
    }
    __syncthreads();

    // ---- the record, written as 16-byte pieces in image order (coalesced)
    unsigned char *rec = ws + ((static_cast<size_t>(n) * H + vh) * n_chunks + ci) * kRecord;
    auto split4 = [](float4 x, float4 &hi, float4 &lo) {
        tc::split_tf32(x.x, hi.x, lo.x);
        tc::split_tf32(x.y, hi.y, lo.y);
        tc::split_tf32(x.z, hi.z, lo.z);
        tc::split_tf32(x.w, hi.w, lo.w);
    };
    // W: rows c, K = dk (one tf32 pass; the tensor core reads the fp32 bits as tf32)
    for (int idx = tid; idx < kC * kS / 4; idx += kPrepThreads) {
        const uint32_t o = idx * 16u;
        const int c = (o / kSboW) * 8 + (o % 128) / 16, k0 = ((o % kSboW) / 128) * 4;
        *reinterpret_cast<float4 *>(rec + kOffW + o) = *reinterpret_cast<const float4 *>(&sm.w[c][k0]);
    }
    // wK^T: rows dk, K = c
    for (int idx = tid; idx < kS * kC / 4; idx += kPrepThreads) {
        const uint32_t o = idx * 16u;
        const int d = (o / kSboK) * 8 + (o % 128) / 16, c0 = ((o % kSboK) / 128) * 4;
        const float4 x = make_float4(sm.wdec[c0] * sm.k[c0][d], sm.wdec[c0 + 1] * sm.k[c0 + 1][d],
                                     sm.wdec[c0 + 2] * sm.k[c0 + 2][d],
                                     sm.wdec[c0 + 3] * sm.k[c0 + 3][d]);
        float4 hi, lo;
        split4(x, hi, lo);
        *reinterpret_cast<float4 *>(rec + kOffKhi + o) = hi;
        *reinterpret_cast<float4 *>(rec + kOffKlo + o) = lo;
    }
    // QM: rows t, K = (dk | s)
    for (int idx = tid; idx < kC * kQmK / 4; idx += kPrepThreads) {
        const uint32_t o = idx * 16u;
        const int t = (o / kSboQ) * 8 + (o % 128) / 16, k0 = ((o % kSboQ) / 128) * 4;
        float4 x;
        if (k0 < kS) {
            x = *reinterpret_cast<const float4 *>(&sm.q[t][k0]);
            const float G = sm.Gam[t];
            x.x *= G; x.y *= G; x.z *= G; x.w *= G;
        } else {
            x = *reinterpret_cast<const float4 *>(&sm.m[t][k0 - kS]);
        }
        float4 hi, lo;
        split4(x, hi, lo);
        *reinterpret_cast<float4 *>(rec + kOffQhi + o) = hi;
        *reinterpret_cast<float4 *>(rec + kOffQlo + o) = lo;
    }
    // Ut: plain [c][dv]
    for (int idx = tid; idx < kC * kS / 4; idx += kPrepThreads) {
        const int c = idx / (kS / 4), d4 = (idx % (kS / 4)) * 4;
        *reinterpret_cast<float4 *>(rec + kOffUt + idx * 16) = *reinterpret_cast<const float4 *>(&sm.v[c][d4]);
    }
    if (tid == 0) *reinterpret_cast<float *>(rec + kOffScal) = sm.Gam[kC - 1];
}


// ============================================================================ chunk scan
constexpr int kScanTcThreads = 192;  // warp 0 producer, warp 1 MMA issuer, warps 2..5 state
constexpr unsigned WD_MMA = 8u;      // a hand-off between the MMA issuer and the state warps
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns (lane = dv): the state S^T, its tf32 hi/lo split (A operand
// of the S products), U^T hi/lo (A operand of the U products), D_u and D_y.
constexpr uint32_t kColSacc = 0, kColShi = 128, kColSlo = 256, kColUhi = 384, kColUlo = 416,
                   kColDu = 448, kColDy = 480;
static_assert(kColDy + kC == kTmemCols, "tensor-memory plan fills the allocation");

struct ScanBars {
    uint64_t full[2], empty[2];  // stage landed / stage free
    uint64_t s_ready, a_done, u_ready, b_done, y_done, fin;
    uint32_t taddr;
    int abort;
};
constexpr size_t kScanSmem = 2 * static_cast<size_t>(kRecord) + sizeof(ScanBars);

__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// One CTA per (sequence, v-head); grid = n_seqs * n_v_heads. One CTA per SM (its
// shared memory and all 512 tensor-memory columns).
__global__ void __launch_bounds__(kScanTcThreads, 1) chunk_scan_kernel(
    float *__restrict__ state, const unsigned char *__restrict__ ws, float *__restrict__ y,
    int n_tokens, int n_v_heads, float scale, const int32_t *__restrict__ slots, int pool,
    int32_t *err_count) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanBars &bars = *reinterpret_cast<ScanBars *>(smem_raw + 2 * kRecord);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = n_v_heads;
    const int vh = blockIdx.x % H, n = blockIdx.x / H;
    const int slot = slots ? slots[n] : n;
    if (slot < 0 || slot >= pool) {  // uniform over the CTA, before any barrier
        if (vh == 0 && tid == 0 && err_count) atomicAdd(err_count, 1);
        return;
    }
    const int n_chunks = (n_tokens + kC - 1) / kC;
    const unsigned char *rec0 = ws + (static_cast<size_t>(n) * H + vh) * n_chunks * kRecord;
    auto stage = [&](int st) { return smem_raw + st * kRecord; };

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.full[i], 1);
            mbar_init(&bars.empty[i], 1 + 4);  // the MMA commit + one arrival per state warp
        }
        mbar_init(&bars.s_ready, 4);
        mbar_init(&bars.a_done, 1);
        mbar_init(&bars.u_ready, 4);
        mbar_init(&bars.b_done, 1);
        mbar_init(&bars.y_done, 1);
        mbar_init(&bars.fin, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&bars.taddr, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.taddr;
    volatile int *abort_flag = &bars.abort;

    // A wait that gives up raises the watchdog flag and sets `abort`; every role then
    // leaves its loop and all threads meet at the final barrier.
    auto wait1 = [&](uint64_t *bar, int parity, unsigned bit) {
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity & 1)) return true;
        atomicOr(&g_watchdog_chunked, bit);
        *abort_flag = 1;
        return false;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;  // copies issued; chunk ci went to stage ci & 1
            for (int ci = 0; ci < n_chunks; ++ci) {
                const int st = ci & 1, use = ci >> 1;
                if (use > 0 && !wait1(&bars.empty[st], use - 1, WD_STAGE_FREE)) break;
                mbar_arrive_expect_tx(&bars.full[st], kRecord);
                bulk_g2s(stage(st), rec0 + static_cast<size_t>(ci) * kRecord, kRecord,
                         &bars.full[st]);
                issued = ci + 1;
            }
            // never leave with a copy still landing in shared memory: wait for the last
            // copy into each stage
            for (int ci = max(0, issued - 2); ci < issued; ++ci)
                mbar_wait(&bars.full[ci & 1], (ci >> 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id32 = tc::idesc_tf32(128, kC), id128 = tc::idesc_tf32(128, kS);
            const uint32_t a_s[3] = {kColShi, kColShi, kColSlo}, a_u[3] = {kColUhi, kColUhi, kColUlo};
            const uint32_t b_q[3] = {kOffQhi, kOffQlo, kOffQhi}, b_k[3] = {kOffKhi, kOffKlo, kOffKhi};
            for (int ci = 0; ci < n_chunks; ++ci) {
                const int st = ci & 1, use = ci >> 1;
                if (!wait1(&bars.full[st], use, WD_STAGE_COPY)) break;
                if (!wait1(&bars.s_ready, ci, WD_MMA)) break;
                tc::fence_after_sync();
                const unsigned char *sb = stage(st);
                // D_u = S^T W^T: U^T before the subtraction (one pass)
                for (int ks = 0; ks < kS / 8; ++ks)
                    tc::mma_tf32_ts(tmem + kColDu, tmem + kColShi + 8 * ks,
                                    tc::smem_desc(sb + kOffW + ks * 2 * kLbo, kLbo, kSboW), id32,
                                    ks > 0);
                tc::mma_commit(&bars.a_done);
                // D_y = S^T (Gam Q)^T (three passes; the U part follows below)
                for (int p = 0; p < 3; ++p)
                    for (int ks = 0; ks < kS / 8; ++ks)
                        tc::mma_tf32_ts(tmem + kColDy, tmem + a_s[p] + 8 * ks,
                                        tc::smem_desc(sb + b_q[p] + ks * 2 * kLbo, kLbo, kSboQ),
                                        id32, p > 0 || ks > 0);
                if (!wait1(&bars.u_ready, ci, WD_MMA)) break;
                tc::fence_after_sync();
                // S^T += U^T (w K): the state update, accumulated in place
                for (int p = 0; p < 3; ++p)
                    for (int ks = 0; ks < kC / 8; ++ks)
                        tc::mma_tf32_ts(tmem + kColSacc, tmem + a_u[p] + 8 * ks,
                                        tc::smem_desc(sb + b_k[p] + ks * 2 * kLbo, kLbo, kSboK),
                                        id128, true);
                tc::mma_commit(&bars.b_done);
                // D_y += U^T M^T
                for (int p = 0; p < 3; ++p)
                    for (int ks = 0; ks < kC / 8; ++ks)
                        tc::mma_tf32_ts(
                            tmem + kColDy, tmem + a_u[p] + 8 * ks,
                            tc::smem_desc(sb + b_q[p] + (kS / 8 + ks) * 2 * kLbo, kLbo, kSboQ),
                            id32, true);
                tc::mma_commit(&bars.y_done);
                tc::mma_commit(&bars.empty[st]);
            }
            tc::mma_commit(&bars.fin);  // tensor memory stays allocated until all MMAs end
            mbar_wait(&bars.fin, 0);
        }
    } else {
        // ------------------------------------------------------------ state warps
        const int quarter = warp & 3;  // the tensor-memory lanes this warp may access
        const int dv = quarter * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float *srow = state + ((static_cast<size_t>(slot) * H + vh) * kS + dv) * kS;
        auto waitw = [&](uint64_t *bar, int parity, unsigned bit) {
            return __all_sync(FULL_MASK, wait1(bar, parity, bit)) != 0;
        };
#pragma unroll 1
        for (int blk = 0; blk < kS / 32; ++blk) {
            uint32_t r[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(srow + 32 * blk + e);
                r[e] = f2u(x.x); r[e + 1] = f2u(x.y); r[e + 2] = f2u(x.z); r[e + 3] = f2u(x.w);
            }
            tc::tmem_st32(trow + kColSacc + 32 * blk, r);
        }
        tc::tmem_st_wait();
        bool ok = true;
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int st = ci & 1, use = ci >> 1;
            const unsigned char *sb = stage(st);
            if (ci > 0) {
                if (!(ok = waitw(&bars.b_done, ci - 1, WD_MMA))) break;
                tc::fence_after_sync();
            }
            if (!(ok = waitw(&bars.full[st], use, WD_STAGE_COPY))) break;
            const float gn = *reinterpret_cast<const float *>(sb + kOffScal);
            // S -> (hi, lo) for the tensor cores; the accumulator becomes Gam_31 S
#pragma unroll 1
            for (int blk = 0; blk < kS / 32; ++blk) {
                uint32_t r[32], hi[32], lo[32];
                tc::tmem_ld32_nowait(trow + kColSacc + 32 * blk, r);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float x = __uint_as_float(r[e]);
                    float h, l;
                    tc::split_tf32(x, h, l);
                    hi[e] = f2u(h);
                    lo[e] = f2u(l);
                    r[e] = f2u(gn * x);
                }
                tc::tmem_st32(trow + kColShi + 32 * blk, hi);
                tc::tmem_st32(trow + kColSlo + 32 * blk, lo);
                tc::tmem_st32(trow + kColSacc + 32 * blk, r);
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.s_ready);

            // U^T = Ut^T - D_u
            if (!(ok = waitw(&bars.a_done, ci, WD_MMA))) break;
            tc::fence_after_sync();
            {
                uint32_t du[32], hi[32], lo[32];
                tc::tmem_ld32_nowait(trow + kColDu, du);
                tc::tmem_ld_wait();
                const float *ut = reinterpret_cast<const float *>(sb + kOffUt);
#pragma unroll
                for (int c = 0; c < kC; ++c) {
                    const float u = ut[c * kS + dv] - __uint_as_float(du[c]);
                    float h, l;
                    tc::split_tf32(u, h, l);
                    hi[c] = f2u(h);
                    lo[c] = f2u(l);
                }
                tc::tmem_st32(trow + kColUhi, hi);
                tc::tmem_st32(trow + kColUlo, lo);
                tc::tmem_st_wait();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars.u_ready);
                mbar_arrive(&bars.empty[st]);  // done reading Ut and Gam_31 of this stage
            }

            // y_t = scale D_y[dv][t]
            if (!(ok = waitw(&bars.y_done, ci, WD_MMA))) break;
            tc::fence_after_sync();
            {
                uint32_t dy[32];
                tc::tmem_ld32_nowait(trow + kColDy, dy);
                tc::tmem_ld_wait();
                const int t0 = ci * kC, valid = min(kC, n_tokens - t0);
                float *yp = y + ((static_cast<size_t>(n) * n_tokens + t0) * H + vh) * kS + dv;
#pragma unroll
                for (int t = 0; t < kC; ++t)
                    if (t < valid) yp[static_cast<size_t>(t) * H * kS] = scale * __uint_as_float(dy[t]);
            }
        }
        if (ok && (ok = waitw(&bars.b_done, n_chunks - 1, WD_MMA))) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int blk = 0; blk < kS / 32; ++blk) {
                uint32_t r[32];
                tc::tmem_ld32_nowait(trow + kColSacc + 32 * blk, r);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(srow + 32 * blk + e) =
                        make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                    __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

unsigned read_and_clear_watchdog_chunked(cudaStream_t s) {
    unsigned flags = 0;
    const unsigned zero = 0;
    cudaMemcpyFromSymbolAsync(&flags, g_watchdog_chunked, sizeof(flags), 0, cudaMemcpyDeviceToHost, s);
    cudaMemcpyToSymbolAsync(g_watchdog_chunked, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return flags;
}

}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_recurrence_scan_chunked_workspace_size(int n_seqs, int n_tokens, int n_v_heads,
                                                  int state_size) {
    if (n_seqs < 0 || n_tokens < 0 || n_v_heads < 1 || state_size != kS) return 0;
    const size_t n_chunks = (static_cast<size_t>(n_tokens) + kC - 1) / kC;
    return static_cast<size_t>(n_seqs) * n_v_heads * n_chunks * kRecord;
}

gdn_status gdn_recurrence_scan_chunked(float *state, const float *q, const float *k,
                                       const float *v, const float *g, const float *beta,
                                       float *y, int n_seqs, int n_tokens, int n_k_heads,
                                       int n_v_heads, int state_size, float scale,
                                       const int32_t *slots, int pool, int32_t *err_count,
                                       void *workspace, size_t workspace_bytes,
                                       gdn_stream_t stream) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    if (n_seqs < 0 || n_tokens < 0) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    if (state_size != kS) return GDN_ERR_UNSUPPORTED;
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y))
        return GDN_ERR_ALIGN;
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    if (n_seqs > 65535 || n_v_heads > 65535 ||
        static_cast<long long>(n_seqs) * n_v_heads > 0x7fffffffLL)
        return GDN_ERR_UNSUPPORTED;
    const size_t need = gdn_recurrence_scan_chunked_workspace_size(n_seqs, n_tokens, n_v_heads,
                                                                   state_size);
    if (!workspace) return GDN_ERR_NULL;
    if (workspace_bytes < need) return GDN_ERR_SHAPE;
    if (!aligned16(workspace)) return GDN_ERR_ALIGN;
    const cudaStream_t s = as_cuda(stream);
    const int n_chunks = (n_tokens + kC - 1) / kC;
    static bool attrs = [] {
        cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(PrepSmem)));
        cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kScanSmem));
        return true;
    }();
    (void)attrs;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    chunk_prep_kernel<<<dim3(n_chunks, n_v_heads, n_seqs), kPrepThreads, sizeof(PrepSmem), s>>>(
        q, k, v, g, beta, ws, n_tokens, n_k_heads, n_v_heads, slots, pool);
    GDN_TRY(launch_status());
    chunk_scan_kernel<<<n_seqs * n_v_heads, kScanTcThreads, kScanSmem, s>>>(
        state, ws, y, n_tokens, n_v_heads, scale, slots, pool, err_count);
    return launch_status();
}

}  // extern "C"
