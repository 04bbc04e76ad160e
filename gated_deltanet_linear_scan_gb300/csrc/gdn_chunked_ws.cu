// gdn_chunked_ws.cu -- the chunked scan in two phases, with a caller workspace.
//
// The algebra is the one of gdn_chunked.cu (the WY/UT regrouping of the delta-rule
// recurrence in chunks of 32 positions; fm_kernel_ssm.m, sequential-scan section,
// names the chunked prefill path and keeps the sequential scan as its reference).
// There, one CTA per (sequence, v-head) does everything for its chunks one after
// the other, and the per-chunk CUDA-core work that does not depend on the state
// (the Gram products and the forward substitution) sets the pace. Here that work
// moves into its own fully parallel kernel:
//
//   chunk_prepare_kernel   one CTA per (chunk, sequence, k-head): the Gram products
//                          of the chunk's k and q rows (shared by the k-head's GQA
//                          v-heads), then per v-head the decay prefix, A and M, and
//                          the forward substitutions (I + A) W = diag(beta Gam) K,
//                          (I + A) Ut = diag(beta) V; W, Ut and M go to the workspace.
//   chunk_state_kernel     one CTA per (sequence, v-head), sequential over chunks:
//                          only the state-dependent part, U = Ut - W S, y and the
//                          state update, on the tensor cores (3xBF16), with W, Ut and M
//                          read back from the workspace.
//
// Both kernels run the arithmetic of gdn_chunked.cu in the same order, so the two
// forms give the same bits. A workspace that holds fewer chunks than the sequence
// has is used in waves (prepare a wave of chunks, advance the state over it, ...);
// the state goes through its fp32 home between waves, which changes no bits either.
#include "gdn_chunk_common.cuh"
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace chunk;

__device__ unsigned g_watchdog_chunked_ws;
constexpr unsigned WD_MMA = 8u;  // a hand-off between the roles of the state kernel

// Workspace block of one (chunk, sequence, v-head), fp32: W [32][128] (rows = positions,
// columns = dk), Ut [32][128] (columns = dv), M [32][32]; chunk-major over a wave: block
// ((c * n_seqs + n) * H + vh) for wave chunk c of a uniform batch.
constexpr int kBlkW = 0, kBlkUt = kC * kS, kBlkM = 2 * kC * kS;
constexpr int kBlkFloats = 2 * kC * kS + kC * kC;
constexpr size_t kBlkBytes = static_cast<size_t>(kBlkFloats) * sizeof(float);

// A ragged batch is prepared in one wave, its blocks indexed by chunk slot: chunk c of
// sequence n takes slot cu[n] / 32 + n + c. The slots of consecutive sequences never
// collide (floor((a + L) / 32) + 1 >= floor(a / 32) + ceil(L / 32)) and stay below
// total / 32 + n_seqs, so the workspace needs (total / 32 + n_seqs) slots of blocks
// whatever the lengths are, and a slot maps back to its sequence by a search over the
// sequences' first slots.
__device__ __forceinline__ long long chunk_slot_base(const int32_t *cu, int n) {
    return static_cast<long long>(cu[n]) / kC + n;
}

__host__ __device__ __forceinline__ long long ragged_chunk_slots(long long total, int n_seqs) {
    return total / kC + n_seqs;
}

// ============================================================================ phase 1
constexpr int kPThreads = 256;
constexpr int kAtRow = kC + 4;  // A^T rows: 36 floats, float4 aligned
constexpr uint32_t kAtBytes = kC * kAtRow * 4;
constexpr uint32_t kVBytes = kC * kS * 4;  // the v rows of one v-head, unpadded
// shared memory: k and q rows (padded), the v rows of two v-heads, A^T, 3 mbarriers
constexpr uint32_t kPOffK = 0, kPOffQ = kRawArr, kPOffV = 2 * kRawArr;
constexpr uint32_t kPOffAt = kPOffV + 2 * kVBytes, kPOffBar = kPOffAt + kAtBytes;
constexpr uint32_t kPOffScale = kPOffBar + 4 * sizeof(uint64_t);  // beta Gam[32], beta[32]
constexpr size_t kPSmemBytes = kPOffScale + 2 * kC * sizeof(float);
static_assert(kPOffBar % 8 == 0, "mbarrier alignment");

// grid = n_wave_chunks * n_seqs * n_k_heads; CTA (cw, n, kh) prepares chunk c_begin + cw of
// sequence n for the v-heads rr * Hk + kh. Warp 0 moves the chunk's k and q rows and the
// v rows of the first two v-heads by 16-byte cp.async at the start (the v rows of v-head
// rr + 2 into the buffer of rr once rr is done), so a CTA waits on memory about once.
__global__ void __launch_bounds__(kPThreads, 3) chunk_prepare_kernel(
    const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
    const float *__restrict__ g, const float *__restrict__ beta, float *__restrict__ ws,
    int n_seqs, const SeqMap seqs, int n_k_heads, int n_v_heads, int c_begin, int n_wave_chunks) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = n_v_heads, Hk = n_k_heads;
    int kh, n, chunk;
    size_t seq0, blk_row;  // first position of sequence n; workspace block row of the chunk
    int n_tokens;
    if (seqs.cu == nullptr) {  // uniform batch: grid (wave chunk, k-head, sequence)
        const int cw = blockIdx.x % n_wave_chunks, rest = blockIdx.x / n_wave_chunks;
        kh = rest % Hk;
        n = rest / Hk;
        seqs.range(n, seq0, n_tokens);
        chunk = c_begin + cw;
        blk_row = static_cast<size_t>(cw) * n_seqs + n;
    } else {  // ragged batch: grid (chunk slot, k-head); slots no chunk owns return
        const int cs = blockIdx.x % n_wave_chunks;
        kh = blockIdx.x / n_wave_chunks;
        n = warp_seq_of_slot(seqs.cu, n_seqs, kC, cs);  // each warp finds it; the same n
        if (n < 0 || !seqs.range(n, seq0, n_tokens)) return;  // uniform over the CTA
        chunk = static_cast<int>(cs - chunk_slot_base(seqs.cu, n));
        if (chunk * kC >= n_tokens) return;
        blk_row = static_cast<size_t>(cs);
    }
    const int t0 = chunk * kC, valid = min(kC, n_tokens - t0);
    const size_t row0 = seq0 + t0;  // (n, t0) in the token-major arrays
    const int ratio = H / Hk;
    float *rk = reinterpret_cast<float *>(smem + kPOffK);
    float *rq = reinterpret_cast<float *>(smem + kPOffQ);
    float *At = reinterpret_cast<float *>(smem + kPOffAt);
    uint64_t *bar_kq = reinterpret_cast<uint64_t *>(smem + kPOffBar);
    uint64_t *bar_v = bar_kq + 1;  // [2]

    // v rows of v-head rr into buffer rr & 1 (warp 0): row r's 512 bytes in one warp
    // instruction (16 bytes a lane), then each lane arrives once its copies land
    auto issue_v = [&](int rr) {
        const int vh = rr * Hk + kh;
#pragma unroll 1
        for (int r = 0; r < valid; ++r)
            cp_async16(smem + kPOffV + (rr & 1) * kVBytes + r * kS * 4 + 16 * lane,
                       v + ((row0 + r) * H + vh) * kS + 4 * lane);
        cp_async_arrive_noinc(bar_v + (rr & 1));
    };
    if (tid == 0) {
        mbar_init(bar_kq, 32);  // one arrival per lane of warp 0
        mbar_init(bar_v, 32);
        mbar_init(bar_v + 1, 32);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll 1
        for (int r = 0; r < valid; ++r) {
            const size_t row = ((row0 + r) * Hk + kh) * kS + 4 * lane;
            cp_async16(rk + r * kRawRowF + 4 * lane, k + row);
            cp_async16(rq + r * kRawRowF + 4 * lane, q + row);
        }
        cp_async_arrive_noinc(bar_kq);
        issue_v(0);
        if (ratio > 1) issue_v(1);
    }
    // rows past the end of the sequence are zero (not copied)
    for (int i = tid; i < 2 * (kC - valid) * kS; i += kPThreads) {
        const int arr = i / ((kC - valid) * kS), rem = i % ((kC - valid) * kS);
        (arr ? rq : rk)[(valid + rem / kS) * kRawRowF + rem % kS] = 0.f;
    }
    // g and beta of the first v-head (lane = position), loaded while the copies land; each
    // v-head's loop then loads the next one's, so no iteration waits on global memory
    auto load_gb = [&](int rr, float &gl, float &bl) {
        gl = 0.f;
        bl = 0.f;
        if (rr < ratio && lane < valid) {
            const int vh = rr * Hk + kh;
            gl = g[(row0 + lane) * H + vh];
            bl = beta[(row0 + lane) * H + vh];
        }
    };
    float gl_next, bl_next;
    load_gb(0, gl_next, bl_next);
    bool ok = mbar_wait(bar_kq, 0);
    __syncthreads();
    int t, s0;
    float kk[4], qk[4];
    gram_products(rk, rq, warp, lane, t, s0, kk, qk);

    const int col = tid & (kS - 1);
    const bool is_w = tid < kS;
    for (int rr = 0; rr < ratio; ++rr) {
        const int vh = rr * Hk + kh;
        float *blk = ws + (blk_row * H + vh) * kBlkFloats;
        const float gl = gl_next, bl = bl_next;  // lane = position
        load_gb(rr + 1, gl_next, bl_next);
        float last;
        const float gam = chunk_gam_from(gl, lane, last);
        const float Gam = expf(gam);
        {
            // A^T[s][t] = beta_t exp(gam_t - gam_s) (k_t . k_s) (s < t); M[t][s] likewise
            // with q_t (s <= t); the same expressions as the one-kernel form
            const float gam_t = __shfl_sync(FULL_MASK, gam, t);
            const float bet_t = __shfl_sync(FULL_MASK, bl, t);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = s0 + 8 * j;
                const float gam_s = __shfl_sync(FULL_MASK, gam, s);
                const float e = s <= t ? expf(gam_t - gam_s) : 0.f;
                At[s * kAtRow + t] = s < t ? bet_t * (e * kk[j]) : 0.f;
                blk[kBlkM + t * kC + s] = e * qk[j];
            }
        }
        // the substitution's per-position scale factors, one warp writing them
        float *sc = reinterpret_cast<float *>(smem + kPOffScale);
        if (warp == 0) {
            sc[lane] = bl * Gam;
            sc[kC + lane] = bl;
        }
        __syncthreads();  // A^T of this v-head is complete, and the scale factors

        // forward substitution, one column per thread: W (threads 0..127), Ut (128..255),
        // column-wise (x_s is final once the rows above are, then updates every row below)
        float x[kC];
        if (is_w) {
#pragma unroll
            for (int p = 0; p < kC; ++p) x[p] = rk[p * kRawRowF + col];
        } else {
            ok = mbar_wait(bar_v + (rr & 1), (rr >> 1) & 1) && ok;
            const float *rv = reinterpret_cast<const float *>(smem + kPOffV + (rr & 1) * kVBytes);
#pragma unroll
            for (int p = 0; p < kC; ++p) x[p] = p < valid ? rv[p * kS + col] : 0.f;
        }
        {
            const float *scp = sc + (is_w ? 0 : kC);  // warp-uniform choice
#pragma unroll
            for (int p = 0; p < kC; p += 4) {
                const float4 f = ld4(scp + p);
                x[p] = f.x * x[p];
                x[p + 1] = f.y * x[p + 1];
                x[p + 2] = f.z * x[p + 2];
                x[p + 3] = f.w * x[p + 3];
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
        float *outp = blk + (is_w ? kBlkW : kBlkUt) + col;
#pragma unroll
        for (int p = 0; p < kC; ++p) outp[p * kS] = x[p];
        __syncthreads();  // done with A^T and with this v-head's v rows
        if (warp == 0 && rr + 2 < ratio) issue_v(rr + 2);
    }
    if (!ok) {
        // a copy wait gave up: flag it, and never leave with a copy still landing
        atomicOr(&g_watchdog_chunked_ws, WD_STAGE_COPY);
        mbar_wait(bar_kq, 0);
        for (int j = 0; j < 2 && j < ratio; ++j)
            mbar_wait(bar_v + j, ((ratio - 1 - j) / 2) & 1);  // last use of buffer j
    }
}

// ============================================================================ phase 2
// shared memory (bytes): the operand images of two chunks, then a ring of two chunk
// stages (the raw k and q rows, and the W and M rows from the workspace, each row padded
// so that a float4 column walk over 8 rows covers all banks). Both images are double-buffered, so the prep warps build chunk ci + 1's
// (buffer (ci + 1) & 1) while the tensor cores still read chunk ci's: image buffer 0 is
// the layout of gdn_chunk_common.cuh at 0 (128-row image, then w K | M); buffer 1 is the
// w K | M image at kOffKM1 and the 128-row image at kOffWQ1.
constexpr uint32_t kKMBytes = kImgBytes - kOffKhi;  // 20 KB: one w K | M image, hi and lo
constexpr uint32_t kWQBytes = kOffKhi;              // 32 KB: one 128-row image, hi and lo
constexpr uint32_t kOffKM1 = kImgBytes;             // second w K | M buffer
constexpr uint32_t kOffWQ1 = kOffKM1 + kKMBytes;    // second 128-row image
constexpr int kMRowF = kC + 4;                      // M rows in a stage: 36 floats
constexpr uint32_t kStW = 2 * kRawArr, kStM = 3 * kRawArr;  // within a stage
constexpr uint32_t kRawBuf = kStM + kC * kMRowF * 4;        // one stage: 55,296 bytes
constexpr uint32_t kOffRaw = kOffWQ1 + kWQBytes;
constexpr uint32_t kOffPTab = kOffRaw + 2 * kRawBuf;  // Gam[32], w_c[32] of the prep's chunk
constexpr uint32_t kOffBars = kOffPTab + 2 * kC * 4;
static_assert(kOffKM1 == kOffKhi + kKMBytes, "second w K | M buffer follows the first");
static_assert(kOffWQ1 % 1024 == 0 && kOffRaw % 16 == 0, "buffer alignment");

struct Bars {
    uint64_t raw_full[2], raw_empty[2];
    uint64_t img_ready[2], buf_free[2], s_ready, u_ready;
    uint64_t a_done, b_done, fin;
    uint32_t taddr;
    int abort;
};
constexpr size_t kSmemBytes = kOffBars + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "fits the opt-in shared memory of one CTA");
static_assert(kOffBars % 8 == 0, "mbarrier alignment");

constexpr int kProducerWarp = 0, kMmaWarp = 1;
constexpr int kStateWarp0 = 2, kStateWarps = 8;
constexpr int kPrepWarp0 = kStateWarp0 + kStateWarps, kPrepWarps = 8;
constexpr int kThreads = 32 * (kPrepWarp0 + kPrepWarps);  // 576
constexpr int kPrepThreads = 32 * kPrepWarps;
constexpr int kStateThreads = 32 * kStateWarps;
constexpr int kPrepBarrier = 1, kStateBarrier = 2;
// 16-byte image units (8 bf16) of W and of M a prep thread converts per chunk
constexpr int kWUnits = kC * kS / 8 / kPrepThreads, kMUnits = kC * kC / 8;
static_assert(kWUnits * kPrepThreads * 8 == kC * kS && kMUnits <= kPrepThreads, "unit split");

// 8 words r[o ..] to p, one 256-bit store; p 32-byte aligned.
__device__ __forceinline__ void st_global_v8(float *p, const uint32_t (&r)[16], int o) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "r"(r[o]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]),
                    "r"(r[o + 4]), "r"(r[o + 5]), "r"(r[o + 6]), "r"(r[o + 7])
                 : "memory");
}

// Columns c0 .. c0 + 63 of the state accumulator's lane at trow (one thread's row of S^T,
// fp32) to dst[c0 ..], 16-byte aligned, in passes of 16 columns. A warp's lanes hold 32
// rows 512 bytes apart, so each store instruction touches 32 lines: 256-bit stores
// (where dst is 32-byte aligned) halve the instructions and requests of 128-bit ones.
__device__ __forceinline__ void copy_state_row(uint32_t trow, int c0, float *dst) {
    const bool wide = (reinterpret_cast<uintptr_t>(dst) & 31u) == 0;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t r[16];
        tc::tmem_ld16_nowait(trow + kColSacc + c0 + 16 * blk, r);
        tc::tmem_ld_wait();
        float *d = dst + c0 + 16 * blk;
        if (wide) {
            st_global_v8(d, r, 0);
            st_global_v8(d + 8, r, 8);
        } else {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(d + e) =
                    make_float4(u2f(r[e]), u2f(r[e + 1]), u2f(r[e + 2]), u2f(r[e + 3]));
        }
    }
}

// State snapshots: every `every` chunks, the state after the chunk that ends there.
// Snapshot j of a sequence is the state after its position (j + 1) * every * kC - 1,
// laid out as one state slot (H * kS * kS floats) of p. Uniform batch (base == nullptr):
// `count` a sequence, sequence n's at slots n * count + j. Ragged batch: sequence n's
// floor(len / (every * kC)) snapshots at slots base[n] + j of a pool of `pool` slots; a
// negative base, or a range past the pool, writes none of them (and is counted).
// p == nullptr: none.
struct SnapOut {
    float *p;
    int every, count;
    const int32_t *base;
    int pool;

    // the first chunk, from chunk cb on, that a snapshot precedes (a positive multiple
    // of every)
    __device__ __forceinline__ int first(int cb) const {
        const int m = (cb + every - 1) / every;
        return (m > 1 ? m : 1) * every;
    }
    // Row dv of v-head vh in snapshot slot 0 of sequence n (of n_tok positions), and the
    // number of its snapshots to write; false for a ragged range that does not fit.
    __device__ __forceinline__ bool place(int n, int n_tok, int vh, int H, int dv, float *&row0,
                                          int &n_snap) const {
        long long slot0;
        if (base == nullptr) {
            slot0 = static_cast<long long>(n) * count;
            n_snap = count;
        } else {
            slot0 = base[n];
            n_snap = n_tok / (every * kC);
            if (n_snap == 0 || slot0 < 0 || slot0 + n_snap > pool) {
                const bool fits = n_snap == 0;
                n_snap = 0;
                row0 = nullptr;
                return fits;
            }
        }
        row0 = p + (static_cast<size_t>(slot0) * H + vh) * (kS * kS) + static_cast<size_t>(dv) * kS;
        return true;
    }
};

// One CTA per (sequence, v-head); grid = n_seqs * n_v_heads. Advances the state over
// chunks c_begin .. c_begin + n_wave_chunks - 1, whose workspace blocks are prepared.
// kSnap (snap.p set): it also writes the snapshots that fall in them; a separate
// instantiation, so that the plain form keeps its registers.
// Roles as in the one-kernel form: producer (k, q rows), MMA issuer, state warps (the
// split of S, U = Ut - D_u, y, no Gram stage), prep warps (operand images only).
template <bool kSnap>
__global__ void __launch_bounds__(kThreads, 1) chunk_state_kernel(
    float *__restrict__ state, const float *__restrict__ q, const float *__restrict__ k,
    const float *__restrict__ g, const float *__restrict__ ws, float *__restrict__ y,
    int n_seqs, const SeqMap seqs, int n_k_heads, int n_v_heads, int c_begin, int n_wave_chunks,
    float scale, const int32_t *__restrict__ slots, int pool, int32_t *err_count,
    const SnapOut snap) {
    extern __shared__ __align__(16) unsigned char smem[];
    Bars &bars = *reinterpret_cast<Bars *>(smem + kOffBars);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = n_v_heads, Hk = n_k_heads;
    const int vh = blockIdx.x % H, kh = vh % Hk;
    int n = blockIdx.x / H;
    if (seqs.cu && n_seqs <= kLongestFirstMaxSeqs) {
        // a small ragged batch: the longest sequences' CTAs first, so the longest chain
        // of chunks starts at once instead of wherever its index puts it
        __shared__ int pick;
        n = seq_by_length_rank(seqs, n_seqs, n, &pick);
    }
    const int slot = slots ? slots[n] : n;
    size_t row0;   // (n, t = 0) in the token-major arrays
    int n_tokens;  // positions of sequence n
    if (slot < 0 || slot >= pool || !seqs.range(n, row0, n_tokens)) {
        // uniform over the CTA, before any barrier
        if (vh == 0 && tid == 0 && err_count) atomicAdd(err_count, 1);
        return;
    }
    float *snap_row0 = nullptr;  // this thread's row of the sequence's snapshot slot 0
    int snap_n = 0;              // snapshots of the sequence to write
    // (tid & 127 is a state thread's row dv: quarter * 32 + lane)
    if (kSnap && !snap.place(n, n_tokens, vh, H, tid & 127, snap_row0, snap_n) && vh == 0 &&
        tid == 0 && err_count)
        atomicAdd(err_count, 1);  // the scan runs; its snapshots are not written
    // uniform batch: this wave's chunks, block rows ci * n_seqs + n; ragged batch: all of
    // the sequence's chunks in one wave, block rows from its first chunk slot on
    const int nw = seqs.cu ? (n_tokens + kC - 1) / kC : n_wave_chunks;
    if (nw == 0) return;  // an empty sequence: the state keeps its bits
    const size_t blk_row0 = seqs.cu ? static_cast<size_t>(chunk_slot_base(seqs.cu, n)) : n;
    const size_t blk_step = seqs.cu ? 1 : static_cast<size_t>(n_seqs);
    auto chunk_t0 = [&](int ci) { return (c_begin + ci) * kC; };
    auto blk_of = [&](int ci) {
        return ws + ((blk_row0 + ci * blk_step) * H + vh) * kBlkFloats;
    };

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.raw_full[i], 32);  // one arrival per producer lane
            mbar_init(&bars.raw_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.img_ready[i], 1);  // chunk ci's images are in buffer ci & 1
            mbar_init(&bars.buf_free[i], 1);   // the MMAs of chunk ci are done with it
        }
        mbar_init(&bars.s_ready, 1);
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

    // Bounded waits, as in the one-kernel form: a wait that gives up raises the
    // watchdog flag and sets `abort`; every role leaves its loop and all threads meet
    // at the final barrier.
    auto wait1 = [&](uint64_t *bar, int parity, unsigned bit) {
        if (*abort_flag) return false;
        if (mbar_wait_sleep(bar, parity & 1, 128)) return true;
        atomicOr(&g_watchdog_chunked_ws, bit);
        *abort_flag = 1;
        return false;
    };
    auto waitw = [&](uint64_t *bar, int parity, unsigned bit) {
        int ok = 0;
        if (lane == 0) ok = wait1(bar, parity, bit);
        return __shfl_sync(FULL_MASK, ok, 0) != 0;
    };
    auto group_wait = [&](bool leader, int barrier_id, int threads, uint64_t *bar, int parity,
                          unsigned bit) {
        bool failed = false;
        if (leader) failed = !wait1(bar, parity, bit);
        return !named_barrier_or(barrier_id, threads, failed || *abort_flag);
    };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        for (int ci = 0; ci < nw; ++ci) {
            const int b = ci & 1, use = ci >> 1;
            if (use > 0 && !waitw(&bars.raw_empty[b], use - 1, WD_STAGE_FREE)) break;
            const int t0 = chunk_t0(ci), valid = min(kC, n_tokens - t0);
            unsigned char *raw = smem + kOffRaw + b * kRawBuf;
            // row r of k and of q: lane l moves bytes 16 l .. 16 l + 15 (one 512-byte row a
            // warp instruction); then the chunk's W rows and M rows from its workspace
            // block (all 32 of each are written there); each lane then arrives on raw_full
            // once its copies land
            for (int r = 0; r < valid; ++r) {
                const size_t row = ((row0 + t0 + r) * Hk + kh) * kS + 4 * lane;
                cp_async16(raw + r * kRawRow + 16 * lane, k + row);
                cp_async16(raw + kRawArr + r * kRawRow + 16 * lane, q + row);
            }
            const float *blk = blk_of(ci);
            for (int r = 0; r < kC; ++r)
                cp_async16(raw + kStW + r * kRawRow + 16 * lane, blk + kBlkW + r * kS + 4 * lane);
            for (int i = 0; i < kC / 4; ++i) {  // 4 rows of M (128 bytes each) a warp instruction
                const int r = 4 * i + (lane >> 3), c4 = 4 * (lane & 7);
                cp_async16(raw + kStM + (r * kMRowF + c4) * 4, blk + kBlkM + r * kC + c4);
            }
            cp_async_arrive_noinc(&bars.raw_full[b]);
            issued = ci + 1;
        }
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
            const uint64_t d_wq0 = desc(kOffWQ, kSbo128), d_wq1 = desc(kOffWQ1, kSbo128);
            constexpr uint64_t kStep = (2 * kLbo) >> 4;
            for (int ci = 0; ci < nw; ++ci) {
                if (!wait1(&bars.img_ready[ci & 1], ci >> 1, WD_MMA)) break;
                const uint64_t d_wq = ci & 1 ? d_wq1 : d_wq0;
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
                // [S^T | D_y] += U^T [w K | M]^T: hi hi + hi lo + lo hi, from buffer ci & 1
                const uint32_t km = (ci & 1) * kKMBytes;
                const uint64_t d_hi = desc(kOffKhi + km, kSbo32), d_lo = desc(kOffKlo + km, kSbo32);
                for (int p = 0; p < 3; ++p) {
                    const uint32_t a = p == 2 ? kColUlo : kColUhi;
                    const uint64_t bd = p == 1 ? d_lo : d_hi;
                    for (int ks = 0; ks < kC / 16; ++ks)
                        tc::mma_bf16_ts(tmem + kColSacc, tmem + a + 8 * ks, bd + kStep * ks, id160,
                                        true);
                }
                tc::mma_commit(&bars.b_done);
                tc::mma_commit(&bars.buf_free[ci & 1]);
            }
            tc::mma_commit(&bars.fin);  // tensor memory stays allocated until all MMAs end
            mbar_wait_sleep(&bars.fin, 0, 128);
        }
    } else if (warp < kPrepWarp0) {
        // ------------------------------------------------------------ state warps
        const int quarter = warp & 3, half = (warp - kStateWarp0) >> 2;
        const int dv = quarter * 32 + lane;
        const int c0 = half * 64, u0 = half * 16;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        float *srow = state + ((static_cast<size_t>(slot) * H + vh) * kS + dv) * kS;
        const bool leader = warp == kStateWarp0 && lane == 0;
        auto st_wait = [&](uint64_t *bar, int parity, unsigned bit = WD_MMA) {
            return group_wait(leader, kStateBarrier, kStateThreads, bar, parity, bit);
        };
        auto st_signal = [&](uint64_t *bar) {
            tc::fence_before_sync();
            named_barrier_sync(kStateBarrier, kStateThreads);
            if (leader) mbar_arrive(bar);
        };
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
            const int t0 = chunk_t0(cj), valid = min(kC, n_tokens - t0);
            float *yp = y + ((row0 + t0) * H + vh) * kS + dv;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (u0 + e < valid) yp[static_cast<size_t>(u0 + e) * H * kS] = yv[e];
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
        float g_cur = 0.f;  // log-decays of chunk ci, lane = position
        if (chunk_t0(0) + lane < n_tokens) g_cur = g[(row0 + chunk_t0(0) + lane) * H + vh];
        bool ok = true;
        int snap_cg = kSnap ? snap.first(c_begin) : 0;  // the next chunk a snapshot precedes
        const size_t snap_stride = static_cast<size_t>(H) * kS * kS;
        for (int ci = 0; ci < nw && ok; ++ci) {
            // this chunk's Ut (dv = this thread's lane of tensor memory, positions u0..)
            float utv[16];
            {
                const float *up = blk_of(ci) + kBlkUt + u0 * kS + dv;
#pragma unroll
                for (int e = 0; e < 16; ++e) utv[e] = up[e * kS];
            }
            float last;
            (void)chunk_gam_from(g_cur, lane, last);
            const float gn = expf(last);
            float g_nx = 0.f;
            if (ci + 1 < nw && chunk_t0(ci + 1) + lane < n_tokens)
                g_nx = g[(row0 + chunk_t0(ci + 1) + lane) * H + vh];
            if (ci > 0) {
                if (!(ok = st_wait(&bars.b_done, ci - 1))) break;
                tc::fence_after_sync();
            }
            // S here is the state after the previous chunk: a snapshot when that chunk
            // ends a snapshot interval
            if (kSnap && c_begin + ci == snap_cg) {
                const int j = snap_cg / snap.every - 1;
                if (j < snap_n) copy_state_row(trow, c0, snap_row0 + j * snap_stride);
                snap_cg += snap.every;
            }
            // S -> (hi, lo), the A operand of the S products; the accumulator becomes
            // Gam_31 S, ready for this chunk's update
            split_state_cols<64>(trow, c0, gn);
            float yv[16];
            if (ci > 0) read_y(yv);
            st_signal(&bars.s_ready);
            if (ci > 0) write_y(ci - 1, yv);
            g_cur = g_nx;

            // U^T = Ut^T - D_u, split
            if (!(ok = st_wait(&bars.a_done, ci))) break;
            tc::fence_after_sync();
            {
                uint32_t du[16], du2[16], hi[8], lo[8];
                float u[16];
                tc::tmem_ld16_nowait(trow + kColDuA + u0, du);
                tc::tmem_ld16_nowait(trow + kColDuB + u0, du2);
                tc::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) u[e] = utv[e] - (u2f(du[e]) + u2f(du2[e]));
                split16_packed(u, hi, lo);
                // positions u0.. of this warp, two to a column
                tc::tmem_st8(trow + kColUhi + u0 / 2, hi);
                tc::tmem_st8(trow + kColUlo + u0 / 2, lo);
                tc::tmem_st_wait();
            }
            st_signal(&bars.u_ready);
        }
        if (ok && nw > 0 && (ok = st_wait(&bars.b_done, nw - 1))) {
            tc::fence_after_sync();
            float yv[16];
            read_y(yv);
            write_y(nw - 1, yv);
            copy_state_row(trow, c0, srow);
            // the final state is the last snapshot too when the sequence ends on one
            if (kSnap && c_begin + nw == snap_cg && snap_cg * kC == n_tokens) {
                const int j = snap_cg / snap.every - 1;
                if (j < snap_n) copy_state_row(trow, c0, snap_row0 + j * snap_stride);
            }
        }
    } else {
        // ------------------------------------------------------------ prep warps
        const int pt = tid - 32 * kPrepWarp0;  // 0..255
        float g_next = 0.f;
        if (chunk_t0(0) + lane < n_tokens) g_next = g[(row0 + chunk_t0(0) + lane) * H + vh];
        // true: leave the loop. The leader waits for the chunk's k and q rows and, from
        // the third chunk on, for image buffer cj & 1 to be free (the MMAs of chunk
        // cj - 2 are done with it).
        auto prep_wait_chunk = [&](int cj) {
            bool failed = false;
            if (pt == 0)
                failed = !wait1(&bars.raw_full[cj & 1], cj >> 1, WD_STAGE_COPY) ||
                         (cj > 1 && !wait1(&bars.buf_free[cj & 1], (cj >> 1) - 1, WD_MMA));
            return named_barrier_or(kPrepBarrier, kPrepThreads, failed || *abort_flag);
        };
        for (int ci = 0; ci < nw; ++ci) {
            const int b = ci & 1;
            const int t0 = chunk_t0(ci), valid = min(kC, n_tokens - t0);
            const float *rk = reinterpret_cast<const float *>(smem + kOffRaw + b * kRawBuf);
            const float *rq = rk + kC * kRawRowF;
            const float *sw = reinterpret_cast<const float *>(smem + kOffRaw + b * kRawBuf + kStW);
            const float *sm = reinterpret_cast<const float *>(smem + kOffRaw + b * kRawBuf + kStM);
            // 8 fp32 values from p, one 16-byte image unit (8 bf16) of a part
            auto ld8 = [](const float *p, float (&x)[8]) {
                const float4 a = ld4(p), b4 = ld4(p + 4);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                x[4] = b4.x; x[5] = b4.y; x[6] = b4.z; x[7] = b4.w;
            };
            // the chunk's Gam_t and w_t for the image units: the first prep warp forms them
            // (lane = position) and writes them before the wait below, whose barrier
            // publishes them (the previous chunk's readers are past the barrier that ended
            // their iteration)
            float *tab = reinterpret_cast<float *>(smem + kOffPTab);
            if (pt < 32) {
                float last;
                const float gam = chunk_gam_from(g_next, lane, last);
                tab[lane] = expf(gam);
                tab[kC + lane] = expf(last - gam);
                g_next = 0.f;
                if (ci + 1 < nw && chunk_t0(ci + 1) + lane < n_tokens)
                    g_next = g[(row0 + chunk_t0(ci + 1) + lane) * H + vh];
            }
            if (prep_wait_chunk(ci)) break;
            // W and Gam_t q_t, split (rows past the end of the sequence count as zero), into
            // image buffer ci & 1
            unsigned char *wq = smem + (b ? kOffWQ1 : kOffWQ);
#pragma unroll
            for (int j = 0; j < kWUnits; ++j) {
                const uint32_t o = (pt + j * kPrepThreads) * 16u;
                int c, k0;
                float x[8];
                image_unit(o, kSbo128, c, k0);
                ld8(sw + c * kRawRowF + k0, x);
                split8_store(x, wq + kOffWhi + o, wq + kOffWlo + o);
            }
#pragma unroll
            for (int j = 0; j < kWUnits; ++j) {
                const uint32_t o = (pt + j * kPrepThreads) * 16u;
                int t, k0;
                image_unit(o, kSbo128, t, k0);
                const float Gt = tab[t];
                float x[8];
                if (t < valid) {
                    const float4 a = ld4(rq + t * kRawRowF + k0), b4 = ld4(rq + t * kRawRowF + k0 + 4);
                    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                    x[4] = b4.x; x[5] = b4.y; x[6] = b4.z; x[7] = b4.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] *= Gt;
                split8_store(x, wq + kOffQhi + o, wq + kOffQlo + o);
            }
            // w_c k_c and M, split, into buffer ci & 1
            unsigned char *kmb = smem + b * kKMBytes;
#pragma unroll
            for (int j = 0; j < kWUnits; ++j) {
                int d, cc;
                wk_unit(pt + j * kPrepThreads, d, cc);
                const uint32_t o = tc::kmajor_offset16(d, cc, kLbo, kSbo32);
                float x[8], wd[8];
                ld8(tab + kC + cc, wd);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    x[j] = wd[j] * (cc + j < valid ? rk[(cc + j) * kRawRowF + d] : 0.f);
                split8_store(x, kmb + kOffKhi + o, kmb + kOffKlo + o);
            }
            if (pt < kMUnits) {
                int t, s0;
                float x[8];
                image_unit(pt * 16u, kSbo32, t, s0);
                ld8(sm + t * kMRowF + s0, x);
                split8_store(x, kmb + kOffMhi + pt * 16u, kmb + kOffMlo + pt * 16u);
            }
            fence_proxy_async_smem();
            named_barrier_sync(kPrepBarrier, kPrepThreads);
            if (pt == 0) {
                mbar_arrive(&bars.img_ready[b]);
                mbar_arrive(&bars.raw_empty[b]);  // done with this chunk's stage
            }
            // this chunk's state split, columns c0 + 32 .. c0 + 63 of this warp's lane
            // quarter, once the previous chunk's state update is done (the first chunk's
            // split is the state warps' alone)

        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

size_t bytes_per_chunk(int n_seqs, int n_v_heads) {
    return static_cast<size_t>(n_seqs) * static_cast<size_t>(n_v_heads) * kBlkBytes;
}

// Checks shared by the entry points; n_seqs > 0 and n_tokens > 0 on GDN_OK.
gdn_status check_common(int n_seqs, int n_tokens, int n_k_heads, int n_v_heads, int state_size) {
    if (n_seqs < 0 || n_tokens < 0) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    if (state_size != kS) return GDN_ERR_UNSUPPORTED;
    if (static_cast<long long>(n_seqs) * n_v_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// A chunk range [cb, cb + nc) of the call and a workspace that holds it.
gdn_status check_range(int n_seqs, int n_tokens, int n_k_heads, int n_v_heads, int cb, int nc,
                       const void *workspace, size_t workspace_bytes) {
    const int n_chunks = (n_tokens + kC - 1) / kC;
    if (cb < 0 || nc < 0 || cb > n_chunks || nc > n_chunks - cb) return GDN_ERR_SHAPE;
    if (nc == 0) return GDN_OK;
    if (!workspace) return GDN_ERR_NULL;
    if (!aligned16(workspace)) return GDN_ERR_ALIGN;
    if (workspace_bytes / bytes_per_chunk(n_seqs, n_v_heads) < static_cast<size_t>(nc))
        return GDN_ERR_SHAPE;
    if (static_cast<long long>(nc) * n_seqs * n_k_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Uniform batch: chunks cb .. cb + nc - 1 of every sequence. Ragged batch (seqs.cu set,
// cb = 0): every chunk slot, nc = ragged_chunk_slots().
gdn_status launch_prepare(const float *q, const float *k, const float *v, const float *g,
                          const float *beta, float *ws, int n_seqs, SeqMap seqs, int n_k_heads,
                          int n_v_heads, int cb, int nc, cudaStream_t s) {
    // per launch: the attribute belongs to the current device
    if (cudaFuncSetAttribute(chunk_prepare_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPSmemBytes)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const long long blocks =
        static_cast<long long>(nc) * (seqs.cu ? 1 : n_seqs) * n_k_heads;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    chunk_prepare_kernel<<<static_cast<unsigned>(blocks), kPThreads, kPSmemBytes, s>>>(
        q, k, v, g, beta, ws, n_seqs, seqs, n_k_heads, n_v_heads, cb, nc);
    return launch_status();
}

gdn_status launch_advance(float *state, const float *q, const float *k, const float *g,
                          const float *ws, float *y, int n_seqs, SeqMap seqs, int n_k_heads,
                          int n_v_heads, float scale, int cb, int nc, const int32_t *slots,
                          int pool, int32_t *err_count, cudaStream_t s,
                          SnapOut snap = SnapOut{nullptr, 1, 0, nullptr, 0}) {
    // per launch: the attribute belongs to the current device
    auto *kernel = snap.p ? chunk_state_kernel<true> : chunk_state_kernel<false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    // slot errors are counted once, with the first chunk
    kernel<<<n_seqs * n_v_heads, kThreads, kSmemBytes, s>>>(
        state, q, k, g, ws, y, n_seqs, seqs, n_k_heads, n_v_heads, cb, nc, scale, slots, pool,
        cb == 0 ? err_count : nullptr, snap);
    return launch_status();
}

}  // namespace

// The bounded-wait self-test on this unit's watchdog flag (gdn_selftest_bounded_wait).
__global__ void wait_probe_kernel_chunked_ws(int arm, unsigned long long limit_ns, float *out) {
    bounded_wait_probe(arm != 0, limit_ns, &g_watchdog_chunked_ws, WD_STAGE_COPY, out);
}

gdn_status launch_wait_probe_chunked_ws(bool arm, uint64_t limit_ns, float *out, cudaStream_t s) {
    wait_probe_kernel_chunked_ws<<<1, 1, 0, s>>>(arm ? 1 : 0, limit_ns, out);
    return launch_status();
}

unsigned read_and_clear_watchdog_chunked_ws(cudaStream_t s) {
    unsigned flags = 0;
    const unsigned zero = 0;
    cudaMemcpyFromSymbolAsync(&flags, g_watchdog_chunked_ws, sizeof(flags), 0,
                              cudaMemcpyDeviceToHost, s);
    cudaMemcpyToSymbolAsync(g_watchdog_chunked_ws, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return flags;
}

size_t ragged_chunked_ws_size(int n_seqs, long long total, int n_v_heads) {
    if (n_seqs < 1 || n_v_heads < 1 || total < 0) return 0;
    return static_cast<size_t>(ragged_chunk_slots(total, n_seqs)) * n_v_heads * kBlkBytes;
}

size_t chunked_seqs_ws_size(int n_seqs, SeqMap seqs, int n_v_heads) {
    if (n_seqs < 1 || n_v_heads < 1) return 0;
    if (seqs.cu == nullptr)
        return static_cast<size_t>((seqs.n_tokens + kC - 1) / kC) * bytes_per_chunk(n_seqs, n_v_heads);
    return ragged_chunked_ws_size(n_seqs, seqs.total, n_v_heads);
}

// The two-phase chunked scan of a ragged batch in one wave, its workspace checked.
static gdn_status chunked_ragged_ws(float *state, const float *q, const float *k, const float *v,
                                    const float *g, const float *beta, float *y, int n_seqs,
                                    SeqMap seqs, int n_k_heads, int n_v_heads, float scale,
                                    const int32_t *slots, int pool, int32_t *err_count,
                                    float *ws, SnapOut snap, cudaStream_t s) {
    const long long n_slots = ragged_chunk_slots(seqs.total, n_seqs);
    if (n_slots > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const int nc = static_cast<int>(n_slots);
    GDN_TRY(launch_prepare(q, k, v, g, beta, ws, n_seqs, seqs, n_k_heads, n_v_heads, 0, nc, s));
    return launch_advance(state, q, k, g, ws, y, n_seqs, seqs, n_k_heads, n_v_heads, scale, 0, nc,
                          slots, pool, err_count, s, snap);
}

gdn_status launch_chunked_seqs(float *state, const float *q, const float *k, const float *v,
                               const float *g, const float *beta, float *y, int n_seqs,
                               SeqMap seqs, int n_k_heads, int n_v_heads, float scale,
                               const int32_t *slots, int pool, int32_t *err_count,
                               void *workspace, size_t workspace_bytes, cudaStream_t s) {
    const size_t need = chunked_seqs_ws_size(n_seqs, seqs, n_v_heads);
    if (workspace == nullptr || need == 0 || workspace_bytes < need || !aligned16(workspace))
        return launch_chunked_one_kernel(state, q, k, v, g, beta, y, n_seqs, seqs, n_k_heads,
                                         n_v_heads, scale, slots, pool, err_count, s);
    const long long slots_or_chunks =
        seqs.cu ? ragged_chunk_slots(seqs.total, n_seqs) : (seqs.n_tokens + kC - 1) / kC;
    if (slots_or_chunks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    float *ws = static_cast<float *>(workspace);
    const int nc = static_cast<int>(slots_or_chunks);
    GDN_TRY(launch_prepare(q, k, v, g, beta, ws, n_seqs, seqs, n_k_heads, n_v_heads, 0, nc, s));
    return launch_advance(state, q, k, g, ws, y, n_seqs, seqs, n_k_heads, n_v_heads, scale, 0, nc,
                          slots, pool, err_count, s);
}

}  // namespace gdn

using namespace gdn;
using namespace gdn::chunk;

extern "C" size_t gdn_recurrence_scan_chunked_ws_size(int n_seqs, int n_tokens, int n_v_heads,
                                                      int state_size) {
    if (n_seqs < 1 || n_tokens < 1 || n_v_heads < 1 || state_size != kS) return 0;
    const size_t n_chunks = (static_cast<size_t>(n_tokens) + kC - 1) / kC;
    return n_chunks * bytes_per_chunk(n_seqs, n_v_heads);
}

extern "C" gdn_status gdn_chunked_prepare(const float *q, const float *k, const float *v,
                                          const float *g, const float *beta, void *workspace,
                                          size_t workspace_bytes, int n_seqs, int n_tokens,
                                          int n_k_heads, int n_v_heads, int state_size,
                                          int chunk_begin, int n_chunks, gdn_stream_t stream) {
    if (!q || !k || !v || !g || !beta) return GDN_ERR_NULL;
    GDN_TRY(check_common(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size));
    if (n_seqs == 0 || n_tokens == 0) return n_chunks == 0 && chunk_begin == 0 ? GDN_OK : GDN_ERR_SHAPE;
    GDN_TRY(check_range(n_seqs, n_tokens, n_k_heads, n_v_heads, chunk_begin, n_chunks, workspace,
                        workspace_bytes));
    if (n_chunks == 0) return GDN_OK;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_ERR_ALIGN;
    return launch_prepare(q, k, v, g, beta, static_cast<float *>(workspace), n_seqs,
                          uniform_seqs(n_seqs, n_tokens), n_k_heads, n_v_heads, chunk_begin,
                          n_chunks, as_cuda(stream));
}

extern "C" gdn_status gdn_chunked_advance(float *state, const float *q, const float *k,
                                          const float *g, const void *workspace,
                                          size_t workspace_bytes, float *y, int n_seqs,
                                          int n_tokens, int n_k_heads, int n_v_heads,
                                          int state_size, float scale, int chunk_begin,
                                          int n_chunks, const int32_t *slots, int pool,
                                          int32_t *err_count, gdn_stream_t stream) {
    if (!state || !q || !k || !g || !y) return GDN_ERR_NULL;
    GDN_TRY(check_common(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (n_seqs == 0 || n_tokens == 0) return n_chunks == 0 && chunk_begin == 0 ? GDN_OK : GDN_ERR_SHAPE;
    GDN_TRY(check_range(n_seqs, n_tokens, n_k_heads, n_v_heads, chunk_begin, n_chunks, workspace,
                        workspace_bytes));
    if (n_chunks == 0) return GDN_OK;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k)) return GDN_ERR_ALIGN;
    return launch_advance(state, q, k, g, static_cast<const float *>(workspace), y, n_seqs,
                          uniform_seqs(n_seqs, n_tokens), n_k_heads, n_v_heads, scale,
                          chunk_begin, n_chunks, slots, pool, err_count, as_cuda(stream));
}

namespace {

// A uniform batch in waves of as many chunks as the workspace holds; the arguments are
// checked by the caller, n_seqs and n_tokens are positive.
gdn_status scan_uniform_waves(float *state, const float *q, const float *k, const float *v,
                              const float *g, const float *beta, float *y, int n_seqs,
                              int n_tokens, int n_k_heads, int n_v_heads, float scale,
                              const int32_t *slots, int pool, int32_t *err_count,
                              void *workspace, size_t workspace_bytes, SnapOut snap,
                              cudaStream_t s) {
    const int n_chunks = (n_tokens + kC - 1) / kC;
    const size_t fit = workspace_bytes / bytes_per_chunk(n_seqs, n_v_heads);
    if (fit < 1) return GDN_ERR_SHAPE;
    const int wave = fit < static_cast<size_t>(n_chunks) ? static_cast<int>(fit) : n_chunks;
    if (static_cast<long long>(wave) * n_seqs * n_k_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    float *ws = static_cast<float *>(workspace);
    for (int cb = 0; cb < n_chunks; cb += wave) {
        const int nc = n_chunks - cb < wave ? n_chunks - cb : wave;
        const SeqMap seqs = uniform_seqs(n_seqs, n_tokens);
        GDN_TRY(launch_prepare(q, k, v, g, beta, ws, n_seqs, seqs, n_k_heads, n_v_heads, cb, nc,
                               s));
        GDN_TRY(launch_advance(state, q, k, g, ws, y, n_seqs, seqs, n_k_heads, n_v_heads, scale,
                               cb, nc, slots, pool, err_count, s, snap));
    }
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_recurrence_scan_chunked_ws(float *state, const float *q, const float *k,
                                                     const float *v, const float *g,
                                                     const float *beta, float *y, int n_seqs,
                                                     int n_tokens, int n_k_heads, int n_v_heads,
                                                     int state_size, float scale,
                                                     const int32_t *slots, int pool,
                                                     int32_t *err_count, void *workspace,
                                                     size_t workspace_bytes, gdn_stream_t stream) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    GDN_TRY(check_common(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    if (!workspace) return GDN_ERR_NULL;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(workspace))
        return GDN_ERR_ALIGN;
    return scan_uniform_waves(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads, n_v_heads,
                              scale, slots, pool, err_count, workspace, workspace_bytes,
                              SnapOut{nullptr, 1, 0, nullptr, 0}, as_cuda(stream));
}

extern "C" int gdn_chunked_snapshot_count(int n_tokens, int snap_every) {
    if (n_tokens < 0 || snap_every < 1) return -1;
    return static_cast<int>(n_tokens / (static_cast<long long>(kC) * snap_every));
}

extern "C" gdn_status gdn_recurrence_scan_chunked_snapshots(
    float *state, const float *q, const float *k, const float *v, const float *g,
    const float *beta, float *y, float *snaps, int snap_every, int n_seqs, int n_tokens,
    int n_k_heads, int n_v_heads, int state_size, float scale, const int32_t *slots, int pool,
    int32_t *err_count, void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    GDN_TRY(check_common(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (snap_every < 1) return GDN_ERR_SHAPE;
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    const int n_snaps = gdn_chunked_snapshot_count(n_tokens, snap_every);
    if (n_snaps > 0 && !snaps) return GDN_ERR_NULL;
    if (!workspace) return GDN_ERR_NULL;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(workspace) || (n_snaps > 0 && !aligned16(snaps)))
        return GDN_ERR_ALIGN;
    return scan_uniform_waves(state, q, k, v, g, beta, y, n_seqs, n_tokens, n_k_heads, n_v_heads,
                              scale, slots, pool, err_count, workspace, workspace_bytes,
                              SnapOut{n_snaps > 0 ? snaps : nullptr, snap_every, n_snaps, nullptr, 0},
                              as_cuda(stream));
}

extern "C" size_t gdn_recurrence_scan_chunked_varlen_ws_size(int n_seqs, int total_tokens,
                                                             int n_v_heads, int state_size) {
    if (state_size != kS) return 0;
    return ragged_chunked_ws_size(n_seqs, total_tokens, n_v_heads);
}

extern "C" gdn_status gdn_recurrence_scan_chunked_varlen(
    float *state, const float *q, const float *k, const float *v, const float *g,
    const float *beta, float *y, const int32_t *cu_seqlens, int n_seqs, int total_tokens,
    int max_tokens, int n_k_heads, int n_v_heads, int state_size, float scale,
    const int32_t *slots, int pool, int32_t *err_count, void *workspace, size_t workspace_bytes,
    gdn_stream_t stream) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    GDN_TRY(check_common(n_seqs, max_tokens, n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_ERR_ALIGN;
    if (workspace && !aligned16(workspace)) return GDN_ERR_ALIGN;
    if (n_seqs == 0 || total_tokens == 0 || max_tokens == 0) return GDN_OK;
    return launch_chunked_seqs(state, q, k, v, g, beta, y, n_seqs,
                               SeqMap{cu_seqlens, max_tokens, total_tokens}, n_k_heads, n_v_heads,
                               scale, slots, pool, err_count, workspace,
                               workspace ? workspace_bytes : 0, as_cuda(stream));
}

extern "C" gdn_status gdn_recurrence_scan_chunked_snapshots_varlen(
    float *state, const float *q, const float *k, const float *v, const float *g,
    const float *beta, float *y, float *snaps, const int32_t *snap_base, int snap_pool,
    int snap_every, const int32_t *cu_seqlens, int n_seqs, int total_tokens, int max_tokens,
    int n_k_heads, int n_v_heads, int state_size, float scale, const int32_t *slots, int pool,
    int32_t *err_count, void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    if (!state || !q || !k || !v || !g || !beta || !y) return GDN_ERR_NULL;
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    GDN_TRY(check_common(n_seqs, max_tokens, n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (snap_every < 1 || snap_pool < 0) return GDN_ERR_SHAPE;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_ERR_ALIGN;
    if (n_seqs == 0 || total_tokens == 0 || max_tokens == 0) return GDN_OK;
    // no sequence of at most max_tokens positions reaches a snapshot: the plain scan
    const bool any = max_tokens / (static_cast<long long>(kC) * snap_every) > 0;
    if (any && (!snaps || !snap_base)) return GDN_ERR_NULL;
    if (!workspace) return GDN_ERR_NULL;
    if ((any && !aligned16(snaps)) || !aligned16(workspace)) return GDN_ERR_ALIGN;
    if (workspace_bytes < ragged_chunked_ws_size(n_seqs, total_tokens, n_v_heads))
        return GDN_ERR_SHAPE;
    return chunked_ragged_ws(state, q, k, v, g, beta, y, n_seqs,
                             SeqMap{cu_seqlens, max_tokens, total_tokens}, n_k_heads, n_v_heads,
                             scale, slots, pool, err_count, static_cast<float *>(workspace),
                             SnapOut{any ? snaps : nullptr, snap_every, 0, snap_base, snap_pool},
                             as_cuda(stream));
}
