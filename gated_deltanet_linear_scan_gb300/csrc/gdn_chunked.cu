// gdn_chunked.cu -- the multi-token scan of the delta-rule recurrence in chunks of
// 32 positions, with the state-dependent contractions on the 5th-generation tensor
// cores (tcgen05, bf16 hi / lo operand parts, fp32 accumulation in tensor memory).
//
// fm_kernel_ssm.m (its softplus note and the sequential-scan section) speaks of a
// chunked prefill path that takes cumulative sums of g along each chunk, with the
// sequential scan kept as its permanent reference; the pages do not spell the
// chunked algebra out. The form used here is derived from the recurrence itself
// (the WY/UT representation of a product of generalised Householder steps). Per
// (sequence, v-head) and chunk of positions t = 0..31 with log-decays g_t, write
// gam_t = g_0 + .. + g_t, Gam_t = exp(gam_t), S the state at the chunk start as a
// [dk][dv] matrix, and
//   A[t][s] = beta_t exp(gam_t - gam_s) (k_t . k_s)        (s < t, else 0)
//   (I + A) W  = diag(beta Gam) K,   (I + A) Ut = diag(beta) V   (forward substitution)
//   U  = Ut - W S                                            (the per-position delta)
//   y_t = scale (Gam_t q_t^T S + sum_{s<=t} exp(gam_t - gam_s) (q_t . k_s) u_s)
//   S' = Gam_31 S + sum_s exp(gam_31 - gam_s) k_s u_s^T.
// This is the recurrence of the sequential scan regrouped exactly (no truncation
// or approximation); only the rounding differs.
//
// One kernel, one CTA per (sequence, v-head), sequential over chunks, one CTA per
// SM. The state lives in tensor memory as S^T (lane = dv, column = dk) for the
// whole scan. Warp roles, linked only by mbarriers:
//   producer (1 warp)  bulk-copies the k, q, v rows of each chunk into a 2-deep ring;
//   state (8 warps)    split S into bf16 hi/lo parts in tensor memory (the A
//                      operand), form U^T = Ut^T - D_u and its split, write y, and in
//                      between, on the CUDA cores in fp32, the next chunk's Gram stage
//                      (gam and the Gram products A and M);
//   prep (8 warps)     per chunk, in fp32: the forward substitution and the
//                      tensor-core operands in shared memory (each written as soon as
//                      the previous chunk's MMAs have finished reading it);
//   MMA (1 thread)     the S products D_u = S^T W^T and D_y = S^T (Gam Q)^T in two
//                      passes (gdn_chunk_common.cuh), then S^T = Gam_31 S^T + U^T (w K)
//                      and D_y += U^T M^T.
//
// Precision: one pass of bf16 (8 significant bits) or of tf32 (11) in the products
// that feed the state or y misses a 2e-3-of-RMS error bound over long scans. Every
// product here takes the split x = hi + lo into two bf16 parts (hi = bf16(x),
// lo = bf16(x - hi)) and sums hi*hi + hi*lo + lo*hi ("3xBF16"): products within about
// 3 * 2^-16 relative, which keeps a 4096-position scan near 1e-4 of the output's RMS.
// A bf16 MMA (K = 16) takes the tensor pipe about as long as a tf32 one (K = 8), so
// the three bf16 passes cost half of what three tf32 passes would.
#include "gdn_chunk_common.cuh"
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace chunk;

__device__ unsigned g_watchdog_chunked;
constexpr unsigned WD_MMA = 8u;  // a hand-off between the roles of the chunked scan

// ---- shared memory (bytes)
// tensor-core operand images at kOffWQ .. kImgBytes (gdn_chunk_common.cuh), then
constexpr uint32_t kOffUt = kImgBytes;                  // Ut, plain [c][dv] fp32
constexpr uint32_t kOffWs = kOffUt + kC * kS * 4;       // W [32][132] fp32, from the substitution
// raw rows of k and q: 2 buffers x 2 arrays x 32 rows (v is read from global memory)
constexpr uint32_t kRawBuf = 2 * kRawArr;
constexpr uint32_t kOffRaw = kOffWs + kRawArr;
constexpr int kAtRow = kC + 4;                         // A^T rows: 36 floats, float4 aligned
constexpr uint32_t kAtBytes = kC * kAtRow * 4, kMBytes = kC * kC * 4;
constexpr uint32_t kOffA = kOffRaw + 2 * kRawBuf;      // 2 x A^T [32][36] (At[s][t] = A[t][s])
constexpr uint32_t kOffM = kOffA + 2 * kAtBytes;       // 2 x M [32][32] (until emitted)
constexpr uint32_t kOffScale = kOffM + 2 * kMBytes;  // beta Gam[32], beta[32] of a chunk
constexpr uint32_t kOffBars = kOffScale + 2 * kC * 4;

struct Bars {
    uint64_t raw_full[2], raw_empty[2], gram_ready[2];
    uint64_t img_ready, s_ready, u_ready;
    uint64_t a_done, b_done, fin;
    uint32_t taddr;
    int abort;
};
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "fits the opt-in shared memory of one CTA");
static_assert(kOffWs % 16 == 0 && kOffRaw % 16 == 0, "bulk-copy and float4 alignment");
static_assert(kOffBars % 8 == 0, "mbarrier alignment");

// ---- warps
constexpr int kProducerWarp = 0, kMmaWarp = 1;
constexpr int kStateWarp0 = 2, kStateWarps = 8;
constexpr int kPrepWarp0 = kStateWarp0 + kStateWarps, kPrepWarps = 8;
constexpr int kThreads = 32 * (kPrepWarp0 + kPrepWarps);  // 576
constexpr int kPrepThreads = 32 * kPrepWarps;
constexpr int kStateThreads = 32 * kStateWarps;
// Named barriers: one per multi-warp role. In each role one leader thread polls the
// mbarriers and the other warps sleep in the named barrier, which leaves the issue
// slots to the warps doing arithmetic.
constexpr int kPrepBarrier = 1, kStateBarrier = 2;
// 16-byte image units (8 bf16) of an operand image part
constexpr int kUnits128x32 = kC * kS / 8, kUnitsM = kC * kC / 8;

// The Gram stage of a chunk, by the 256 threads of one role (warp gw = 0..7), on the
// thread mapping of gram_products:
//   At[s][t] = beta_t exp(gam_t - gam_s) (k_t . k_s)   (s < t, else 0)
//   M[t][s]  = exp(gam_t - gam_s) (q_t . k_s)          (s <= t, else 0)
// gam and bet hold the chunk's gam_lane and beta_lane.
__device__ __forceinline__ void chunk_gram(const float *rk, const float *rq, float *At, float *Msc,
                                           float gam, float bet, int gw, int lane) {
    int t, s0;
    float kk[4], qk[4];
    gram_products(rk, rq, gw, lane, t, s0, kk, qk);
    const float gam_t = __shfl_sync(FULL_MASK, gam, t);
    const float bet_t = __shfl_sync(FULL_MASK, bet, t);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int s = s0 + 8 * j;
        const float gam_s = __shfl_sync(FULL_MASK, gam, s);
        const float e = s <= t ? expf(gam_t - gam_s) : 0.f;
        At[s * kAtRow + t] = s < t ? bet_t * (e * kk[j]) : 0.f;
        Msc[t * kC + s] = e * qk[j];
    }
}

// One CTA per (sequence, v-head); grid = n_seqs * n_v_heads.
__global__ void __launch_bounds__(kThreads, 1) chunked_scan_kernel(
    float *__restrict__ state, const float *__restrict__ q, const float *__restrict__ k,
    const float *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
    float *__restrict__ y, const SeqMap seqs, int n_k_heads, int n_v_heads, float scale,
    const int32_t *__restrict__ slots, int pool, int32_t *err_count) {
    extern __shared__ __align__(16) unsigned char smem[];
    Bars &bars = *reinterpret_cast<Bars *>(smem + kOffBars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = n_v_heads, Hk = n_k_heads;
    const int vh = blockIdx.x % H, n = blockIdx.x / H, kh = vh % Hk;
    const int slot = slots ? slots[n] : n;
    size_t row0;   // (n, t = 0) in the token-major arrays
    int n_tokens;  // positions of sequence n
    if (slot < 0 || slot >= pool || !seqs.range(n, row0, n_tokens)) {
        // uniform over the CTA, before any barrier
        if (vh == 0 && tid == 0 && err_count) atomicAdd(err_count, 1);
        return;
    }
    if (n_tokens == 0) return;  // nothing to scan: the state keeps its bits
    const int n_chunks = (n_tokens + kC - 1) / kC;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.raw_full[i], 32);  // one arrival per producer lane
            mbar_init(&bars.raw_empty[i], 1);
            mbar_init(&bars.gram_ready[i], 1);
        }
        mbar_init(&bars.img_ready, 1);  // arrived by the leader of each role after its
        mbar_init(&bars.s_ready, 1);    // named barrier
        mbar_init(&bars.u_ready, 1);
        mbar_init(&bars.a_done, 1);
        mbar_init(&bars.b_done, 1);
        mbar_init(&bars.fin, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
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
    // Polls sleep between tries (at most 128 ns): the pollers share SM sub-partitions
    // with the prep warps, whose issue slots bound the whole scan.
    auto wait1 = [&](uint64_t *bar, int parity, unsigned bit) {
        if (*abort_flag) return false;
        if (mbar_wait_sleep(bar, parity & 1, 128)) return true;
        atomicOr(&g_watchdog_chunked, bit);
        *abort_flag = 1;
        return false;
    };
    // One lane polls, the rest of the warp waits at the shuffle: warp-uniform result.
    auto waitw = [&](uint64_t *bar, int parity, unsigned bit) {
        int ok = 0;
        if (lane == 0) ok = wait1(bar, parity, bit);
        return __shfl_sync(FULL_MASK, ok, 0) != 0;
    };
    // The same for a multi-warp role: its leader thread polls, the role's other
    // threads sleep in the role's named barrier, and all get the same answer.
    auto group_wait = [&](bool leader, int barrier_id, int threads, uint64_t *bar, int parity,
                          unsigned bit) {
        bool failed = false;
        if (leader) failed = !wait1(bar, parity, bit);
        return !named_barrier_or(barrier_id, threads, failed || *abort_flag);
    };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int b = ci & 1, use = ci >> 1;
            if (use > 0 && !waitw(&bars.raw_empty[b], use - 1, WD_STAGE_FREE)) break;
            const int t0 = ci * kC, valid = min(kC, n_tokens - t0);
            unsigned char *raw = smem + kOffRaw + b * kRawBuf;
            // row r of k and of q: lane l moves bytes 16 l .. 16 l + 15 (one 512-byte row a
            // warp instruction); each lane then arrives on raw_full once its copies land
            for (int r = 0; r < valid; ++r) {
                const size_t row = ((row0 + t0 + r) * Hk + kh) * kS + 4 * lane;
                cp_async16(raw + r * kRawRow + 16 * lane, k + row);
                cp_async16(raw + kRawArr + r * kRawRow + 16 * lane, q + row);
            }
            cp_async_arrive_noinc(&bars.raw_full[b]);
            issued = ci + 1;
        }
        // never leave with a copy still landing: wait for the last fill of each buffer
        for (int ci = max(0, issued - 2); ci < issued; ++ci)
            mbar_wait_sleep(&bars.raw_full[ci & 1], (ci >> 1) & 1, 128);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id64 = tc::idesc_bf16(128, 2 * kC), id128 = tc::idesc_bf16(128, kS),
                           id160 = tc::idesc_bf16(128, kS + kC);
            auto desc = [&](uint32_t off, uint32_t sbo) { return tc::smem_desc(smem + off, kLbo, sbo); };
            // K step ks starts 2 core matrices (256 bytes) further: + 16 in the
            // descriptor's address field (no carry: shared memory stays below 256 KiB)
            const uint64_t d_wq = desc(kOffWQ, kSbo128);
            constexpr uint64_t kStep = (2 * kLbo) >> 4;
            const uint64_t d_hi = desc(kOffKhi, kSbo32), d_lo = desc(kOffKlo, kSbo32);
            for (int ci = 0; ci < n_chunks; ++ci) {
                if (!wait1(&bars.img_ready, ci, WD_MMA)) break;
                if (!wait1(&bars.s_ready, ci, WD_MMA)) break;
                tc::fence_after_sync();
                // the S products, K = 16 a step (8 packed columns of S): hi(S) against all
                // 128 image rows (N = 128), then lo(S) against hi(Gam q) and hi(W) (N = 64)
                // into the first two blocks of D
                for (int ks = 0; ks < kS / 16; ++ks)
                    tc::mma_bf16_ts(tmem + kColD, tmem + kColShi + 8 * ks, d_wq + kStep * ks,
                                    id128, ks > 0);
                for (int ks = 0; ks < kS / 16; ++ks)
                    tc::mma_bf16_ts(tmem + kColD, tmem + kColSlo + 8 * ks, d_wq + kStep * ks,
                                    id64, true);
                tc::mma_commit(&bars.a_done);
                if (!wait1(&bars.u_ready, ci, WD_MMA)) break;
                tc::fence_after_sync();
                // [S^T | D_y] += U^T [w K | M]^T: hi hi + hi lo + lo hi
                for (int p = 0; p < 3; ++p) {
                    const uint32_t a = p == 2 ? kColUlo : kColUhi;
                    const uint64_t bd = p == 1 ? d_lo : d_hi;
                    for (int ks = 0; ks < kC / 16; ++ks)
                        tc::mma_bf16_ts(tmem + kColSacc, tmem + a + 8 * ks, bd + kStep * ks, id160,
                                        true);
                }
                tc::mma_commit(&bars.b_done);
            }
            tc::mma_commit(&bars.fin);  // tensor memory stays allocated until all MMAs end
            mbar_wait_sleep(&bars.fin, 0, 128);
        }
    } else if (warp < kPrepWarp0) {
        // ------------------------------------------------------------ state warps
        // Warp w may access tensor-memory lanes 32 (w % 4) ..; two warps share each
        // quarter of the lanes and split the columns: S columns c0 .. c0 + 63, U and
        // D_y columns (positions) u0 .. u0 + 15.
        const int quarter = warp & 3, half = (warp - kStateWarp0) >> 2;
        const int dv = quarter * 32 + lane;
        const int c0 = half * 64, u0 = half * 16;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float *srow = state + ((static_cast<size_t>(slot) * H + vh) * kS + dv) * kS;
        const float *ut = reinterpret_cast<const float *>(smem + kOffUt);
        const bool leader = warp == kStateWarp0 && lane == 0;
        auto st_wait = [&](uint64_t *bar, int parity, unsigned bit = WD_MMA) {
            return group_wait(leader, kStateBarrier, kStateThreads, bar, parity, bit);
        };
        // Signal the MMA issuer once every state warp's tensor-memory stores are done.
        auto st_signal = [&](uint64_t *bar) {
            tc::fence_before_sync();
            named_barrier_sync(kStateBarrier, kStateThreads);
            if (leader) mbar_arrive(bar);
        };

        // y of chunk cj from D_y; false if the wait gave up
        // y of chunk cj: read from D_y once its b_done has been waited for (before the
        // next chunk's MMAs overwrite it), then written out (after those MMAs are under
        // way)
        auto read_y = [&](float (&yv)[16]) {
            uint32_t dy[16], dy2[16];
            tc::tmem_ld16_nowait(trow + kColDyA + u0, dy);
            tc::tmem_ld16_nowait(trow + kColDyB + u0, dy2);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) yv[e] = scale * (u2f(dy[e]) + u2f(dy2[e]));
        };
        auto write_y = [&](int cj, const float (&yv)[16]) {
            const int t0 = cj * kC, valid = min(kC, n_tokens - t0);
            float *yp = y + ((row0 + t0) * H + vh) * kS + dv;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (u0 + e < valid) yp[static_cast<size_t>(u0 + e) * H * kS] = yv[e];
        };

        // The Gram stage of chunk cj (its decay inputs gj, bj, lane = position), in the
        // time these warps would otherwise wait for the prep warps: pad the rows past
        // the end of the sequence with zeros (an identity step), then fill buffer cj & 1
        // of A^T and M.
        const int sw = warp - kStateWarp0, st_tid = 32 * sw + lane;
        auto gram_chunk = [&](int cj, float gj, float bj) {
            const int b = cj & 1, valid = min(kC, n_tokens - cj * kC);
            if (!st_wait(&bars.raw_full[b], cj >> 1, WD_STAGE_COPY)) return false;
            float *rk = reinterpret_cast<float *>(smem + kOffRaw + b * kRawBuf);
            if (valid < kC) {
                const int pad = (kC - valid) * kS;
                for (int i = st_tid; i < 2 * pad; i += kStateThreads) {
                    const int arr = i / pad, rem = i % pad;
                    rk[arr * kC * kRawRowF + (valid + rem / kS) * kRawRowF + rem % kS] = 0.f;
                }
                named_barrier_sync(kStateBarrier, kStateThreads);
            }
            float last;
            const float gam = chunk_gam_from(gj, lane, last);
            chunk_gram(rk, rk + kC * kRawRowF, reinterpret_cast<float *>(smem + kOffA + b * kAtBytes),
                       reinterpret_cast<float *>(smem + kOffM + b * kMBytes), gam, bj, sw, lane);
            st_signal(&bars.gram_ready[b]);
            return true;
        };

#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
            uint32_t r[16];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 x = ld4(srow + c0 + 16 * blk + e);
                r[e] = f2u(x.x); r[e + 1] = f2u(x.y); r[e + 2] = f2u(x.z); r[e + 3] = f2u(x.w);
            }
            tc::tmem_st16(trow + kColSacc + c0 + 16 * blk, r);
        }
        tc::tmem_st_wait();
        float g_cur = 0.f, b_cur = 0.f;  // decay inputs of chunk ci, lane = position
        if (lane < min(kC, n_tokens)) {
            g_cur = g[(row0 + lane) * H + vh];
            b_cur = beta[(row0 + lane) * H + vh];
        }
        bool ok = gram_chunk(0, g_cur, b_cur);
        for (int ci = 0; ci < n_chunks && ok; ++ci) {
            float last;
            (void)chunk_gam_from(g_cur, lane, last);
            const float gn = expf(last);
            float g_nx = 0.f, b_nx = 0.f;  // the next chunk's, for its Gram stage below
            if ((ci + 1) * kC + lane < n_tokens) {
                g_nx = g[(row0 + (ci + 1) * kC + lane) * H + vh];
                b_nx = beta[(row0 + (ci + 1) * kC + lane) * H + vh];
            }
            if (ci > 0) {
                if (!(ok = st_wait(&bars.b_done, ci - 1))) break;
                tc::fence_after_sync();
            }
            // S -> (hi, lo), the A operand of the S products; the accumulator becomes
            // Gam_31 S, ready for this chunk's update
            split_state_row(trow, c0, gn);
            // the previous chunk's y leaves D_y before this chunk's MMAs overwrite it
            float yv[16];
            if (ci > 0) read_y(yv);
            st_signal(&bars.s_ready);
            if (ci > 0) write_y(ci - 1, yv);
            // the next chunk's Gram stage, while the prep warps finish this chunk
            if (ci + 1 < n_chunks && !(ok = gram_chunk(ci + 1, g_nx, b_nx))) break;
            g_cur = g_nx;
            b_cur = b_nx;

            // U^T = Ut^T - D_u, split (a_done comes after img_ready, so it also says Ut
            // is in place; the leader checks both)
            if (!(ok = st_wait(&bars.img_ready, ci))) break;
            if (!(ok = st_wait(&bars.a_done, ci))) break;
            tc::fence_after_sync();
            {
                uint32_t du[16], du2[16], hi[8], lo[8];
                float u[16];
                tc::tmem_ld16_nowait(trow + kColDuA + u0, du);
                tc::tmem_ld16_nowait(trow + kColDuB + u0, du2);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) u[e] = ut[(u0 + e) * kS + dv] - (u2f(du[e]) + u2f(du2[e]));
                split16_packed(u, hi, lo);
                // positions u0.. of this warp, two to a column
                tc::tmem_st8(trow + kColUhi + u0 / 2, hi);
                tc::tmem_st8(trow + kColUlo + u0 / 2, lo);
                tc::tmem_st_wait();
            }
            st_signal(&bars.u_ready);
        }
        if (ok && n_chunks > 0 && (ok = st_wait(&bars.b_done, n_chunks - 1))) {
            tc::fence_after_sync();
            float yv[16];
            read_y(yv);
            write_y(n_chunks - 1, yv);
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t r[16];
                tc::tmem_ld16_nowait(trow + kColSacc + c0 + 16 * blk, r);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4 *>(srow + c0 + 16 * blk + e) =
                        make_float4(u2f(r[e]), u2f(r[e + 1]), u2f(r[e + 2]), u2f(r[e + 3]));
            }
        }
    } else {
        // ------------------------------------------------------------ prep warps
        // All eight warps take every decision together (named_barrier_or), so none is
        // ever left waiting at a named barrier that another has abandoned.
        const int pt = tid - 32 * kPrepWarp0;  // 0..255
        float *utw = reinterpret_cast<float *>(smem + kOffUt);
        // true: leave the loop (a wait gave up somewhere)
        auto prep_wait = [&](uint64_t *bar, int parity, unsigned bit) {
            return !group_wait(pt == 0, kPrepBarrier, kPrepThreads, bar, parity, bit);
        };
        auto prep_sync = [&]() {
            return named_barrier_or(kPrepBarrier, kPrepThreads, *abort_flag != 0);
        };
        float g_next = 0.f, b_next = 0.f;  // decay inputs of the next chunk, lane = position
        if (lane < min(kC, n_tokens)) {
            g_next = g[(row0 + lane) * H + vh];
            b_next = beta[(row0 + lane) * H + vh];
        }
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int b = ci & 1, use = ci >> 1;
            const int t0 = ci * kC;
            float *rk = reinterpret_cast<float *>(smem + kOffRaw + b * kRawBuf);
            float *rq = rk + kC * kRawRowF;
            float *ws = reinterpret_cast<float *>(smem + kOffWs);
            const float *At = reinterpret_cast<const float *>(smem + kOffA + b * kAtBytes);
            const float *Msc = reinterpret_cast<const float *>(smem + kOffM + b * kMBytes);
            // per-position decay quantities, lane = position (each warp its own copy)
            float last;
            const float gam = chunk_gam_from(g_next, lane, last);
            const float Gam = expf(gam), wdec = expf(last - gam);
            const float bet = b_next;
            g_next = b_next = 0.f;
            if (t0 + kC + lane < n_tokens) {
                g_next = g[(row0 + t0 + kC + lane) * H + vh];
                b_next = beta[(row0 + t0 + kC + lane) * H + vh];
            }
            // the state warps have padded the raw rows and written A^T and M of this chunk
            if (prep_wait(&bars.gram_ready[b], use, WD_MMA)) break;
            // the Ut columns start from beta_t v_t: fetch v (zero past the end)
            const int col = pt & (kS - 1);
            const bool is_w = pt < kS;
            float x[kC];
            if (!is_w) {
                const float *vp = v + ((row0 + t0) * H + vh) * kS + col;
                const size_t vstride = static_cast<size_t>(H) * kS;
                const int valid = min(kC, n_tokens - t0);
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    x[t] = t < valid ? *vp : 0.f;
                    vp += vstride;
                }
            }

            // ---- forward substitution, one column per thread: W (warps 0..3), Ut (4..7).
            // Row t is base_t - sum_{s<t} A[t][s] x_s, accumulated in order of s; done
            // column-wise (x_s is final once the rows above are, and then updates every
            // row below it), so the dependent chain is 32 steps long, not 496. Ut goes
            // straight to its buffer, so first wait until the previous chunk is done with
            // it (its U is formed, which also means its W S product is done).
            // the per-position scale factors, written by one warp before the wait below
            // (whose barrier publishes them; the previous chunk's readers are long done)
            float *sc = reinterpret_cast<float *>(smem + kOffScale);
            if (pt < 32) {
                sc[lane] = bet * Gam;
                sc[kC + lane] = bet;
            }
            if (ci > 0 ? prep_wait(&bars.u_ready, ci - 1, WD_MMA) : prep_sync()) break;
            {
                const float *scp = sc + (is_w ? 0 : kC);  // warp-uniform choice
#pragma unroll
                for (int t = 0; t < kC; t += 4) {
                    const float4 f = ld4(scp + t);
                    if (is_w) {
                        x[t] = f.x * rk[t * kRawRowF + col];
                        x[t + 1] = f.y * rk[(t + 1) * kRawRowF + col];
                        x[t + 2] = f.z * rk[(t + 2) * kRawRowF + col];
                        x[t + 3] = f.w * rk[(t + 3) * kRawRowF + col];
                    } else {
                        x[t] = f.x * x[t];
                        x[t + 1] = f.y * x[t + 1];
                        x[t + 2] = f.z * x[t + 2];
                        x[t + 3] = f.w * x[t + 3];
                    }
                }
            }
#pragma unroll
            for (int s2 = 0; s2 < kC - 1; ++s2) {
#pragma unroll
                for (int m = (s2 + 1) / 4; m < kC / 4; ++m) {
                    const float4 a = ld4(At + s2 * kAtRow + 4 * m);
                    if (4 * m + 0 > s2) x[4 * m + 0] = fmaf(-a.x, x[s2], x[4 * m + 0]);
                    if (4 * m + 1 > s2) x[4 * m + 1] = fmaf(-a.y, x[s2], x[4 * m + 1]);
                    if (4 * m + 2 > s2) x[4 * m + 2] = fmaf(-a.z, x[s2], x[4 * m + 2]);
                    if (4 * m + 3 > s2) x[4 * m + 3] = fmaf(-a.w, x[s2], x[4 * m + 3]);
                }
            }
            {
                float *outp = is_w ? ws : utw;
                const int ostride = is_w ? kRawRowF : kS;
#pragma unroll
                for (int t = 0; t < kC; ++t) outp[t * ostride + col] = x[t];
            }
            named_barrier_sync(kPrepBarrier, kPrepThreads);
            // the images take 16-byte units of 8 bf16: 8 fp32 values a unit
            for (int idx = pt; idx < kUnits128x32; idx += kPrepThreads) {  // W, split
                const uint32_t o = idx * 16u;
                int c, k0;
                image_unit(o, kSbo128, c, k0);
                const float4 a = ld4(ws + c * kRawRowF + k0), b4 = ld4(ws + c * kRawRowF + k0 + 4);
                const float x[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
                split8_store(x, smem + kOffWhi + o, smem + kOffWlo + o);
            }
            // Gam_t q_t, split (the S products that read it finished before U was formed)
            for (int idx = pt; idx < kUnits128x32; idx += kPrepThreads) {
                const uint32_t o = idx * 16u;
                int t, k0;
                image_unit(o, kSbo128, t, k0);
                const float Gt = __shfl_sync(FULL_MASK, Gam, t);
                const float4 a = ld4(rq + t * kRawRowF + k0), b4 = ld4(rq + t * kRawRowF + k0 + 4);
                float x[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] *= Gt;
                split8_store(x, smem + kOffQhi + o, smem + kOffQlo + o);
            }
            // ---- w_c k_c and M, split, once the previous chunk's state update is done
            if (ci > 0 ? prep_wait(&bars.b_done, ci - 1, WD_MMA) : prep_sync()) break;
            for (int u = pt; u < kUnits128x32; u += kPrepThreads) {
                int d, cc;
                wk_unit(u, d, cc);
                const uint32_t o = tc::kmajor_offset16(d, cc, kLbo, kSbo32);
                float x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    x[j] = __shfl_sync(FULL_MASK, wdec, cc + j) * rk[(cc + j) * kRawRowF + d];
                split8_store(x, smem + kOffKhi + o, smem + kOffKlo + o);
            }
            // M, split (read by the same MMAs as w K)
            for (int idx = pt; idx < kUnitsM; idx += kPrepThreads) {
                const uint32_t o = idx * 16u;
                int t, s0;
                image_unit(o, kSbo32, t, s0);
                const float4 a = ld4(Msc + t * kC + s0), b4 = ld4(Msc + t * kC + s0 + 4);
                const float x[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
                split8_store(x, smem + kOffMhi + o, smem + kOffMlo + o);
            }
            // the operands are read by the tensor cores (async proxy) and Ut by the
            // state warps
            fence_proxy_async_smem();
            named_barrier_sync(kPrepBarrier, kPrepThreads);
            if (pt == 0) {
                mbar_arrive(&bars.img_ready);
                mbar_arrive(&bars.raw_empty[b]);  // done with this chunk's raw rows
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace
}  // namespace gdn

namespace gdn {

// The bounded-wait self-test on this unit's watchdog flag (gdn_selftest_bounded_wait).
__global__ void wait_probe_kernel_chunked(int arm, unsigned long long limit_ns, float *out) {
    bounded_wait_probe(arm != 0, limit_ns, &g_watchdog_chunked, WD_STAGE_COPY, out);
}

gdn_status launch_wait_probe_chunked(bool arm, uint64_t limit_ns, float *out, cudaStream_t s) {
    wait_probe_kernel_chunked<<<1, 1, 0, s>>>(arm ? 1 : 0, limit_ns, out);
    return launch_status();
}

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

namespace gdn {

gdn_status launch_chunked_one_kernel(float *state, const float *q, const float *k,
                                     const float *v, const float *g, const float *beta, float *y,
                                     int n_seqs, SeqMap seqs, int n_k_heads, int n_v_heads,
                                     float scale, const int32_t *slots, int pool,
                                     int32_t *err_count, cudaStream_t s) {
    if (static_cast<long long>(n_seqs) * n_v_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    // per launch: the attribute belongs to the current device
    if (cudaFuncSetAttribute(chunked_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    chunked_scan_kernel<<<n_seqs * n_v_heads, kThreads, kSmemBytes, s>>>(
        state, q, k, v, g, beta, y, seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count);
    return launch_status();
}

}  // namespace gdn

extern "C" gdn_status gdn_recurrence_scan_chunked(float *state, const float *q, const float *k,
                                                  const float *v, const float *g,
                                                  const float *beta, float *y, int n_seqs,
                                                  int n_tokens, int n_k_heads, int n_v_heads,
                                                  int state_size, float scale,
                                                  const int32_t *slots, int pool,
                                                  int32_t *err_count, gdn_stream_t stream) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    if (n_seqs < 0 || n_tokens < 0) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    if (state_size != kS) return GDN_ERR_UNSUPPORTED;
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_ERR_ALIGN;
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    return launch_chunked_one_kernel(state, q, k, v, g, beta, y, n_seqs,
                                     uniform_seqs(n_seqs, n_tokens), n_k_heads, n_v_heads, scale,
                                     slots, pool, err_count, as_cuda(stream));
}
