// gdn_recurrence.cu -- the delta-rule recurrence on sm_103a: single-token decode
// over many sequences (HBM bound) and the multi-token sequential scan (latency /
// issue bound).
//
// Work split, both kernels: a warp owns R = 4 rows (v-index j) of one head's
// transposed state; lane L holds the contiguous cells [E*L, E*L+E) of each row
// (E = S/32), so a row moves as one 128-bit access per lane. The two dots per
// row and token are a 4-term in-lane chain plus a packed shuffle butterfly that
// serves R rows per shuffle: no shared-memory reduction tree, no barrier inside
// the token loop. Decode and scan call the same row step, so a scan over T tokens
// and T decode calls agree bit for bit (fm_kernel_ssm.m states the same property
// of its scan).
#include <atomic>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ unsigned g_watchdog;

constexpr int kWarps = 8;           // consumer warps per CTA
constexpr int kRowsPerWarp = 4;     // R
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 32 state rows

// Lanes that hold a finished readout for one of the R rows, and which row.
template <int R>
__device__ __forceinline__ bool y_writer(int lane, int &r) {
    constexpr int low = (R == 1) ? 31 : (R == 2) ? 15 : (R == 4) ? 7 : 3;
    r = ((lane >> 4) & 1) | (((lane >> 3) & 1) << 1) | (((lane >> 2) & 1) << 2);
    r &= (R - 1);
    return (lane & low) == 0;
}

// ---------------------------------------------------------------------------- decode
// Grid: one CTA per (sequence, v-head, block of 32 rows). Each warp pulls its 4
// contiguous state rows (4*S*4 bytes) with one bulk copy into shared memory while
// the lanes fetch k, q, v, g and beta; the update goes back to HBM with 128-bit
// stores. The state of a (slot, head) is S*S*4 contiguous bytes, so a CTA's tile is
// one contiguous run and every access is fully coalesced.
template <int E, bool FACTORED>
__global__ void __launch_bounds__(kWarps * 32) recurrence_decode_kernel(
    float *state, const float *__restrict__ q, const float *__restrict__ k,
    const float *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
    float *__restrict__ y, int n_k_heads, int n_v_heads, float scale,
    const int32_t *__restrict__ slots, int pool, int32_t *err_count, int reverse) {
    constexpr int S = 32 * E, R = kRowsPerWarp;
    constexpr int kBlocksPerHead = S / kRowsPerCta;
    // reverse: the tiles in descending order, so that a launch starts on the tiles the
    // previous one (ascending) wrote last, whose new state is still in L2
    const int blk = reverse ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *tile = reinterpret_cast<float *>(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + kRowsPerCta * S * sizeof(float));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blk % kBlocksPerHead;
    const int vh = (blk / kBlocksPerHead) % n_v_heads;
    const int n = blk / (kBlocksPerHead * n_v_heads);
    const int kh = vh % n_k_heads;
    const int slot = slots ? slots[n] : n;
    if (slot < 0 || slot >= pool) {
        if (err_count && vh == 0 && part == 0 && threadIdx.x == 0) atomicAdd(err_count, 1);
        return;
    }
    const int row0 = part * kRowsPerCta + warp * R;  // first row of this warp
    float *gstate = state + ((static_cast<size_t>(slot) * n_v_heads + vh) * S + row0) * S;
    float *wtile = tile + warp * R * S;
    uint64_t *bar = bars + warp;
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, R * S * sizeof(float));
        bulk_g2s(wtile, gstate, R * S * sizeof(float), bar);
    }
    float kk[E], qq[E], vv[R];
    load_vec<E>(kk, k + (static_cast<size_t>(n) * n_k_heads + kh) * S + lane * E);
    load_vec<E>(qq, q + (static_cast<size_t>(n) * n_k_heads + kh) * S + lane * E);
    const size_t hv = static_cast<size_t>(n) * n_v_heads + vh;
#pragma unroll
    for (int r = 0; r < R; ++r) vv[r] = v[hv * S + row0 + r];
    const float decay = expf(g[hv]);
    const float bt = beta[hv];
    __syncwarp();
    if (!mbar_wait(bar, 0)) {
        if (lane == 0) atomicOr(&g_watchdog, WD_STATE_COPY);
        mbar_wait(bar, 0);  // never leave with a copy still landing in shared memory
        return;
    }
    float row[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) load_vec<E>(row[r], wtile + r * S + lane * E);
    float yout;
    if constexpr (FACTORED) {
        const float kq = warp_allsum(lane_dot<E>(kk, qq));
        yout = row_step_factored<E, R>(row, kk, qq, vv, decay, bt, kq, scale, lane);
    } else {
        yout = __fmul_rn(scale, row_step<E, R>(row, kk, qq, vv, decay, bt, lane));
    }
#pragma unroll
    for (int r = 0; r < R; ++r) store_vec<E>(gstate + r * S + lane * E, row[r]);
    int r;
    if (y_writer<R>(lane, r)) y[hv * S + row0 + r] = yout;
}

// ---------------------------------------------------------------------------- scan
// The scan is bound by instruction issue, not memory: every state element is
// touched by 4 FP operations per token and the two dots per row and token must be
// reduced. Here a state row is held by a group of 4 lanes instead of a whole warp,
// so a warp carries 8 rows and each reduction needs only 2 shuffle levels.
//
// Lane g (0..3) of a row group holds the 8 chunks of E cells that lanes g, g+4, ...,
// g+28 hold in the decode kernels' layout (chunk m = cells [4E*m + E*g, ... + E)).
// The first three butterfly levels of the decode kernels (partners L^16, L^8,
// L^4) then pair chunks inside one lane, in the same order, and the last two
// (L^2, L^1) are shuffles inside the group: every sum, hence every state bit and
// output, is the decode kernels'. A scan over T tokens still equals T decode calls
// bit for bit.
constexpr int kScanRowsPerWarp = 8; // 8 groups of 4 lanes
constexpr int kScanTok = 16;        // tokens per staged chunk
constexpr int kScanDepth = 2;       // chunks in flight

// CTA shape and shared memory of the scan for S = 32 E. A CTA has 8 consumer warps
// (64 rows) wherever a head has that many rows, else 4, plus the producer warp: at
// S = 128, 2 CTAs per SM at 96 registers, each staging k and q once for 64 rows (a
// third less time than 4-warp CTAs at 4 per SM, same bits).
template <int E>
struct ScanSmem {
    static constexpr int S = 32 * E;
    static constexpr int kWarps = S >= 64 ? 8 : 4;           // consumer warps
    static constexpr int kRows = kWarps * kScanRowsPerWarp;  // state rows per CTA
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kMinBlocks = E >= 8 ? 1 : (E == 1 ? 4 : 2);
    static constexpr int kFloats = kScanTok * S;             // per array per stage
    static constexpr int vFloats = kScanTok * kRows;
    static constexpr size_t stage_bytes = (2 * kFloats + vFloats) * sizeof(float);
    static constexpr size_t bytes = kScanDepth * stage_bytes + 2 * kScanDepth * sizeof(uint64_t);
    static_assert(S % kRows == 0, "a head is a whole number of CTA row blocks");
};

// The 8 chunks of lane g of a row: chunk m starts at cell 4E*m + E*g.
template <int E>
__device__ __forceinline__ void load_group(float (&dst)[8][E], const float *row, int g) {
#pragma unroll
    for (int m = 0; m < 8; ++m) load_vec<E>(dst[m], row + 4 * E * m + E * g);
}

template <int E>
__device__ __forceinline__ void store_group(float *row, const float (&src)[8][E], int g) {
#pragma unroll
    for (int m = 0; m < 8; ++m) store_vec<E>(row + 4 * E * m + E * g, src[m]);
}

// Dot of a row with x (lane g's chunks read from shared memory at xs) over the
// whole row, in the decode kernels' exact order: per-chunk FMA chains, then chunks
// m and m+4, m and m+2, 0 and 1 (the partners L^16, L^8, L^4), then the group
// shuffles L^2 and L^1. Every lane of the group returns the same bits.
template <int E>
__device__ __forceinline__ float group_dot(const float (&r)[8][E], const float *xs, int g) {
    float p[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        float x[E];
        load_vec<E>(x, xs + 4 * E * m + E * g);
        p[m] = lane_dot<E>(r[m], x);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) p[m] = __fadd_rn(p[m], p[m + 4]);
#pragma unroll
    for (int m = 0; m < 2; ++m) p[m] = __fadd_rn(p[m], p[m + 2]);
    float acc = __fadd_rn(p[0], p[1]);
    acc = __fadd_rn(acc, __shfl_xor_sync(FULL_MASK, acc, 2));
    acc = __fadd_rn(acc, __shfl_xor_sync(FULL_MASK, acc, 1));
    return acc;
}

// Grid: one CTA per (sequence, v-head, block of 64 rows, or 32 at S = 32); 8 (or 4)
// consumer warps hold 8 rows each in registers for all tokens, plus one producer warp that stages the
// per-token k, q (S floats each) and this block's 32 v values through a 2-deep ring
// of shared-memory chunks with bulk copies, each chunk tracked by a "full" and an
// "empty" mbarrier. g and beta (one float per token and head) are read by the lanes
// a chunk ahead and broadcast with shuffles. The state reaches HBM once per call.
// RAGGED selects the ragged-batch form; the uniform one reads the sequence length and
// offset straight from the kernel parameters, which keeps them out of the registers the
// token loop needs.
template <int E, bool SNAP, bool RAGGED>
__global__ void __launch_bounds__(ScanSmem<E>::kThreads, ScanSmem<E>::kMinBlocks) recurrence_scan_kernel(
    float *state, const float *__restrict__ q, const float *__restrict__ k,
    const float *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
    float *__restrict__ y, const SeqMap seqs, int n_seqs_ragged, int n_k_heads, int n_v_heads,
    float scale, const int32_t *__restrict__ slots, int pool, int32_t *err_count,
    float *__restrict__ snaps) {
    constexpr int S = 32 * E, TC = kScanTok;
    using L = ScanSmem<E>;
    constexpr int kScanWarps = L::kWarps, kScanRows = L::kRows;
    constexpr int kBlocksPerHead = S / kScanRows;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw + kScanDepth * L::stage_bytes);
    uint64_t *empty = full + kScanDepth;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x % kBlocksPerHead;
    const int vh = (blockIdx.x / kBlocksPerHead) % n_v_heads;
    int n = blockIdx.x / (kBlocksPerHead * n_v_heads);
    if (RAGGED && n_seqs_ragged <= kLongestFirstMaxSeqs) {
        // a small ragged batch: the longest sequences' CTAs first
        __shared__ int pick;
        n = seq_by_length_rank(seqs, n_seqs_ragged, n, &pick);
    }
    const int kh = vh % n_k_heads;
    const int slot = slots ? slots[n] : n;
    size_t tok0;   // first position of sequence n in the token-major arrays
    int n_tokens;  // its length
    if (!RAGGED) {
        n_tokens = seqs.n_tokens;
        tok0 = static_cast<size_t>(n) * seqs.n_tokens;
    }
    if (slot < 0 || slot >= pool || (RAGGED && !seqs.range(n, tok0, n_tokens))) {
        if (err_count && vh == 0 && part == 0 && threadIdx.x == 0) atomicAdd(err_count, 1);
        return;
    }
    if (n_tokens == 0) return;  // uniform over the CTA: nothing to scan
    if (threadIdx.x == 0) {
        for (int s = 0; s < kScanDepth; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kScanWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int n_chunks = (n_tokens + TC - 1) / TC;
    const size_t kq_tok = static_cast<size_t>(n_k_heads) * S;   // q/k stride per token
    const size_t v_tok = static_cast<size_t>(n_v_heads) * S;    // v/y stride per token
    const float *kbase = k + (tok0 * n_k_heads + kh) * S;
    const float *qbase = q + (tok0 * n_k_heads + kh) * S;
    const float *vbase = v + (tok0 * n_v_heads + vh) * S + part * kScanRows;

    if (warp == kScanWarps) {
        // ---- producer warp: lane t copies token t of each chunk.
        int issued = 0;  // chunks whose copies were issued
        for (int c = 0; c < n_chunks; ++c) {
            const int s = c % kScanDepth, use = c / kScanDepth;
            if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1)) {
                if (lane == 0) atomicOr(&g_watchdog, WD_STAGE_FREE);
                break;
            }
            const int tc = min(TC, n_tokens - c * TC);
            unsigned char *st = smem_raw + s * L::stage_bytes;
            float *ks = reinterpret_cast<float *>(st);
            float *qs = ks + L::kFloats;
            float *vs = qs + L::kFloats;
            if (lane == 0)
                mbar_arrive_expect_tx(full + s, tc * (2 * S + kScanRows) * sizeof(float));
            __syncwarp();
            if (lane < tc) {
                const size_t t = static_cast<size_t>(c) * TC + lane;
                bulk_g2s(ks + lane * S, kbase + t * kq_tok, S * sizeof(float), full + s);
                bulk_g2s(qs + lane * S, qbase + t * kq_tok, S * sizeof(float), full + s);
                bulk_g2s(vs + lane * kScanRows, vbase + t * v_tok, kScanRows * sizeof(float),
                         full + s);
            }
            issued = c + 1;
        }
        // Do not leave while copies may still be landing in this CTA's shared memory,
        // also when a wait above gave up (each of these waits is bounded too).
        for (int c = max(0, issued - kScanDepth); c < issued; ++c)
            mbar_wait(full + c % kScanDepth, (c / kScanDepth) & 1);
        return;
    }

    // ---- consumer warps: lane = 4 * (row of the warp) + g
    const int rho = lane >> 2, gq = lane & 3;
    const int rl = warp * kScanRowsPerWarp + rho;  // row within the CTA's block
    const int j = part * kScanRows + rl;         // state row (v index)
    float *grow = state + ((static_cast<size_t>(slot) * n_v_heads + vh) * S + j) * S;
    float row[8][E];
    load_group<E>(row, grow, gq);
    const size_t gb_base = tok0 * n_v_heads + vh;
    float *yrow = y + (tok0 * n_v_heads + vh) * S + j;
    // snapshot after position t of sequence n: at packed position tok0 + t of snaps
    // ([N][T][H][S][S] for a uniform batch), the state layout of one slot
    const size_t snap_tok = static_cast<size_t>(n_v_heads) * S * S;
    float *srow = SNAP ? snaps + ((tok0 * n_v_heads + vh) * S + j) * S : nullptr;

    // g and beta of token (chunk*TC + lane), one chunk ahead.
    auto fetch_gb = [&](int c, float &dec, float &bt) {
        const int t = c * TC + lane;
        if (lane < TC && c < n_chunks && t < n_tokens) {
            dec = expf(g[gb_base + static_cast<size_t>(t) * n_v_heads]);
            bt = beta[gb_base + static_cast<size_t>(t) * n_v_heads];
        } else {
            dec = 1.0f;
            bt = 0.0f;
        }
    };
    float dec_cur, bt_cur, dec_nxt, bt_nxt;
    fetch_gb(0, dec_cur, bt_cur);
    bool ok = true;
    for (int c = 0; c < n_chunks; ++c) {
        const int s = c % kScanDepth;
        fetch_gb(c + 1, dec_nxt, bt_nxt);
        if (!mbar_wait(full + s, (c / kScanDepth) & 1)) {
            if (lane == 0) atomicOr(&g_watchdog, WD_STAGE_COPY);
            ok = false;
            break;
        }
        const unsigned char *st = smem_raw + s * L::stage_bytes;
        const float *ks = reinterpret_cast<const float *>(st);
        const float *qs = ks + L::kFloats;
        const float *vs = qs + L::kFloats;
        const int tc = min(TC, n_tokens - c * TC);
        // unrolled by 3: a warp issues in order, and this lets it start the next tokens'
        // products while a token's readout is still in its shuffles (deeper unrolling
        // spills at this register budget)
#pragma unroll 3
        for (int t = 0; t < tc; ++t) {
            // the row step of the decode kernels, in the group layout
            const float decay = __shfl_sync(FULL_MASK, dec_cur, t);
            const float bt = __shfl_sync(FULL_MASK, bt_cur, t);
            // k and q chunks are read from shared memory where they are used, so the
            // warp keeps only its state rows live across the token
            const float *kt = ks + t * S;
            const float vj = vs[t * kScanRows + rl];
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int e = 0; e < E; ++e) row[m][e] = __fmul_rn(row[m][e], decay);
            const float pred = group_dot<E>(row, kt, gq);
            const float delta = __fmul_rn(__fsub_rn(vj, pred), bt);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                float kc[E];
                load_vec<E>(kc, kt + 4 * E * m + E * gq);
#pragma unroll
                for (int e = 0; e < E; ++e) row[m][e] = __fmaf_rn(kc[e], delta, row[m][e]);
            }
            const float ysum = group_dot<E>(row, qs + t * S, gq);
            const size_t tok = static_cast<size_t>(c) * TC + t;
            if (gq == 0) yrow[tok * v_tok] = __fmul_rn(scale, ysum);
            if constexpr (SNAP) store_group<E>(srow + tok * snap_tok, row, gq);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
        dec_cur = dec_nxt;
        bt_cur = bt_nxt;
    }
    if (!ok) return;  // leave the state untouched rather than write a partial scan
    store_group<E>(grow, row, gq);
}

// Opts a kernel in to more than 48 KiB of dynamic shared memory.
template <typename Kern>
gdn_status set_smem(Kern kern, size_t bytes) {
    if (bytes <= 48 * 1024) return GDN_OK;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_LAUNCH;
}

template <int E, bool FACTORED>
gdn_status launch_decode(float *state, const float *q, const float *k, const float *v,
                         const float *g, const float *beta, float *y, int n_seqs, int n_k_heads,
                         int n_v_heads, float scale, const int32_t *slots, int pool,
                         int32_t *err_count, cudaStream_t s) {
    constexpr int S = 32 * E;
    const size_t smem = kRowsPerCta * S * sizeof(float) + kWarps * sizeof(uint64_t);
    GDN_TRY(set_smem(recurrence_decode_kernel<E, FACTORED>, smem));
    const long long blocks = static_cast<long long>(n_seqs) * n_v_heads * (S / kRowsPerCta);
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    // Consecutive decode steps visit the tiles in alternating directions: a step leaves the
    // state it wrote last dirty in L2 and the next one, walking the other way, reads that
    // state first instead of evicting it unread. The results do not depend on the order.
    static std::atomic<unsigned> launches{0};
    const int reverse = static_cast<int>(launches.fetch_add(1, std::memory_order_relaxed) & 1u);
    recurrence_decode_kernel<E, FACTORED><<<static_cast<unsigned>(blocks), kWarps * 32, smem, s>>>(
        state, q, k, v, g, beta, y, n_k_heads, n_v_heads, scale, slots, pool, err_count, reverse);
    return launch_status();
}

template <int E, bool SNAP, bool RAGGED>
gdn_status launch_scan_form(float *state, const float *q, const float *k, const float *v,
                            const float *g, const float *beta, float *y, int n_seqs, SeqMap seqs,
                            int n_k_heads, int n_v_heads, float scale, const int32_t *slots,
                            int pool, int32_t *err_count, float *snaps, cudaStream_t s) {
    constexpr int S = 32 * E;
    const size_t smem = ScanSmem<E>::bytes;
    GDN_TRY(set_smem(recurrence_scan_kernel<E, SNAP, RAGGED>, smem));
    const long long blocks = static_cast<long long>(n_seqs) * n_v_heads * (S / ScanSmem<E>::kRows);
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    recurrence_scan_kernel<E, SNAP, RAGGED><<<static_cast<unsigned>(blocks), ScanSmem<E>::kThreads, smem, s>>>(
        state, q, k, v, g, beta, y, seqs, n_seqs, n_k_heads, n_v_heads, scale, slots, pool,
        err_count, snaps);
    return launch_status();
}

template <int E, bool SNAP>
gdn_status launch_scan(float *state, const float *q, const float *k, const float *v,
                       const float *g, const float *beta, float *y, int n_seqs, SeqMap seqs,
                       int n_k_heads, int n_v_heads, float scale, const int32_t *slots, int pool,
                       int32_t *err_count, float *snaps, cudaStream_t s) {
    if (seqs.cu)
        return launch_scan_form<E, SNAP, true>(state, q, k, v, g, beta, y, n_seqs, seqs,
                                               n_k_heads, n_v_heads, scale, slots, pool,
                                               err_count, snaps, s);
    return launch_scan_form<E, SNAP, false>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads,
                                            n_v_heads, scale, slots, pool, err_count, snaps, s);
}

gdn_status check_recurrence_args(const float *state, const float *q, const float *k,
                                 const float *v, const float *g, const float *beta,
                                 const float *y, int n_seqs, int n_tokens, int n_k_heads,
                                 int n_v_heads, int state_size, const int32_t *slots, int pool) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    if (n_seqs < 0 || n_tokens < 0) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_ERR_ALIGN;
    return GDN_OK;
}

}  // namespace

// The bounded-wait self-test on this unit's watchdog flag (gdn_selftest_bounded_wait).
__global__ void wait_probe_kernel_recurrence(int arm, unsigned long long limit_ns, float *out) {
    bounded_wait_probe(arm != 0, limit_ns, &g_watchdog, WD_STAGE_COPY, out);
}

gdn_status launch_wait_probe_recurrence(bool arm, uint64_t limit_ns, float *out, cudaStream_t s) {
    wait_probe_kernel_recurrence<<<1, 1, 0, s>>>(arm ? 1 : 0, limit_ns, out);
    return launch_status();
}

unsigned read_and_clear_watchdog_recurrence(cudaStream_t s) {
    unsigned flags = 0;
    const unsigned zero = 0;
    cudaMemcpyFromSymbolAsync(&flags, g_watchdog, sizeof(flags), 0, cudaMemcpyDeviceToHost, s);
    cudaMemcpyToSymbolAsync(g_watchdog, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return flags;
}

namespace {

template <bool FACTORED>
gdn_status decode_entry(float *state, const float *q, const float *k, const float *v,
                        const float *g, const float *beta, float *y, int n_seqs, int n_k_heads,
                        int n_v_heads, int state_size, float scale, const int32_t *slots, int pool,
                        int32_t *err_count, gdn_stream_t stream) {
    GDN_TRY(check_recurrence_args(state, q, k, v, g, beta, y, n_seqs, 1, n_k_heads, n_v_heads,
                                  state_size, slots, pool));
    if (n_seqs == 0) return GDN_OK;
    const cudaStream_t s = as_cuda(stream);
    switch (state_size) {
        case 32: return launch_decode<1, FACTORED>(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, s);
        case 64: return launch_decode<2, FACTORED>(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, s);
        case 128: return launch_decode<4, FACTORED>(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, s);
        default: return launch_decode<8, FACTORED>(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, s);
    }
}

template <bool SNAP>
gdn_status scan_launch(float *state, const float *q, const float *k, const float *v,
                       const float *g, const float *beta, float *y, int n_seqs, SeqMap seqs,
                       int n_k_heads, int n_v_heads, int state_size, float scale,
                       const int32_t *slots, int pool, int32_t *err_count, float *snaps,
                       cudaStream_t s) {
    switch (state_size) {
        case 32: return launch_scan<1, SNAP>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, snaps, s);
        case 64: return launch_scan<2, SNAP>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, snaps, s);
        case 128: return launch_scan<4, SNAP>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, snaps, s);
        default: return launch_scan<8, SNAP>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads, n_v_heads, scale, slots, pool, err_count, snaps, s);
    }
}

template <bool SNAP>
gdn_status scan_entry(float *state, const float *q, const float *k, const float *v,
                      const float *g, const float *beta, float *y, int n_seqs, int n_tokens,
                      int n_k_heads, int n_v_heads, int state_size, float scale,
                      const int32_t *slots, int pool, int32_t *err_count, float *snaps,
                      gdn_stream_t stream) {
    GDN_TRY(check_recurrence_args(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads,
                                  n_v_heads, state_size, slots, pool));
    if (SNAP && snaps == nullptr) return GDN_ERR_NULL;
    if (SNAP && !aligned16(snaps)) return GDN_ERR_ALIGN;
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    return scan_launch<SNAP>(state, q, k, v, g, beta, y, n_seqs, uniform_seqs(n_seqs, n_tokens),
                             n_k_heads, n_v_heads, state_size, scale, slots, pool, err_count,
                             snaps, as_cuda(stream));
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

gdn_status gdn_recurrence_decode(float *state, const float *q, const float *k, const float *v,
                                 const float *g, const float *beta, float *y, int n_seqs,
                                 int n_k_heads, int n_v_heads, int state_size, float scale,
                                 const int32_t *slots, int pool, int32_t *err_count,
                                 gdn_stream_t stream) {
    return decode_entry<false>(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads,
                               state_size, scale, slots, pool, err_count, stream);
}

gdn_status gdn_recurrence_decode_2pass(float *state, const float *q, const float *k,
                                       const float *v, const float *g, const float *beta,
                                       float *y, int n_seqs, int n_k_heads, int n_v_heads,
                                       int state_size, float scale, const int32_t *slots,
                                       int pool, int32_t *err_count, gdn_stream_t stream) {
    return decode_entry<true>(state, q, k, v, g, beta, y, n_seqs, n_k_heads, n_v_heads,
                              state_size, scale, slots, pool, err_count, stream);
}

gdn_status gdn_recurrence_scan(float *state, const float *q, const float *k, const float *v,
                               const float *g, const float *beta, float *y, int n_seqs,
                               int n_tokens, int n_k_heads, int n_v_heads, int state_size,
                               float scale, const int32_t *slots, int pool, int32_t *err_count,
                               gdn_stream_t stream) {
    return scan_entry<false>(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads, n_v_heads,
                             state_size, scale, slots, pool, err_count, nullptr, stream);
}

gdn_status gdn_recurrence_scan_snapshots(float *state, const float *q, const float *k,
                                         const float *v, const float *g, const float *beta,
                                         float *y, float *snaps, int n_seqs, int n_tokens,
                                         int n_k_heads, int n_v_heads, int state_size,
                                         float scale, const int32_t *slots, int pool,
                                         int32_t *err_count, gdn_stream_t stream) {
    return scan_entry<true>(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads, n_v_heads,
                            state_size, scale, slots, pool, err_count, snaps, stream);
}

}  // extern "C"

// ============================================================================ ragged batches
namespace gdn {

gdn_status launch_scan_seqs(float *state, const float *q, const float *k, const float *v,
                            const float *g, const float *beta, float *y, int n_seqs, SeqMap seqs,
                            int n_k_heads, int n_v_heads, int state_size, float scale,
                            const int32_t *slots, int pool, int32_t *err_count, float *snaps,
                            cudaStream_t s) {
    if (snaps)
        return scan_launch<true>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads, n_v_heads,
                                 state_size, scale, slots, pool, err_count, snaps, s);
    return scan_launch<false>(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads, n_v_heads,
                              state_size, scale, slots, pool, err_count, nullptr, s);
}

gdn_status check_varlen(const int32_t *cu_seqlens, int n_seqs, int total_tokens, int max_tokens) {
    if (!cu_seqlens) return GDN_ERR_NULL;
    if (n_seqs < 0 || total_tokens < 0 || max_tokens < 0) return GDN_ERR_SHAPE;
    return GDN_OK;
}

}  // namespace gdn

extern "C" gdn_status gdn_recurrence_scan_varlen(float *state, const float *q, const float *k,
                                                 const float *v, const float *g,
                                                 const float *beta, float *y,
                                                 const int32_t *cu_seqlens, int n_seqs,
                                                 int total_tokens, int max_tokens,
                                                 int n_k_heads, int n_v_heads, int state_size,
                                                 float scale, const int32_t *slots, int pool,
                                                 int32_t *err_count, gdn_stream_t stream) {
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    GDN_TRY(check_recurrence_args(state, q, k, v, g, beta, y, n_seqs, max_tokens, n_k_heads,
                                  n_v_heads, state_size, slots, pool));
    if (n_seqs == 0 || total_tokens == 0 || max_tokens == 0) return GDN_OK;
    return launch_scan_seqs(state, q, k, v, g, beta, y, n_seqs,
                            SeqMap{cu_seqlens, max_tokens, total_tokens}, n_k_heads, n_v_heads,
                            state_size, scale, slots, pool, err_count, nullptr, as_cuda(stream));
}
