// gdn_block.cu -- the whole Gated-DeltaNet block for one decode token per
// sequence, fused into one sm_103a kernel so every state byte crosses HBM once.
//
// Mapping. A thread-block cluster serves one (sequence, k-head kh) group: the
// GQA ratio r = H/Hk v-heads vh = rr*Hk + kh (ssm_gated_delta.cu: interleaved
// tiling; gated_delta_net_decode.metal: k_head = v_head % n_k_heads) share kh's
// q/k conv channels. Each v-head may be split over `split` CTAs of S/split rows,
// so the cluster has r*split CTAs. Every CTA
//   1. issues one bulk (TMA) copy per warp for its state rows into shared memory;
//   2. meanwhile recomputes conv1d+SiLU of kh's 2S q/k channels from the old
//      conv_state, L2-normalises q and k, convolves the v channels of its own
//      rows (rolling their conv_state, which it alone owns), and evaluates the
//      decay gate and beta for its head;
//   3. runs the row step (decay, pred, delta, rank-1 write, read-after-write
//      readout) on its rows and streams the new state back to HBM;
//   4. applies the gated RMSNorm to its head's readout. When a head is split,
//      the per-CTA sums of squares are exchanged through distributed shared
//      memory.
// The q/k conv_state of kh is rolled exactly once, by cluster rank 0, after a
// cluster barrier guarantees every CTA of the group has read the old values.
#include <atomic>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ unsigned g_watchdog;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kR = 4;   // rows per warp per pass
constexpr int kTaps = 3;  // conv_kernel - 1 (the fused block is built for K = 4)

struct BlockParams {
    const float *qkv, *conv_w;
    float *conv_state;
    const float *alpha, *b, *dt, *a, *z, *norm_w;
    float *state, *out;
    const int32_t *slots;
    int32_t *err_count;
    int n_k_heads, n_v_heads, ratio, split, pool;
    float scale, l2_eps, norm_eps;
};

template <int E>
struct BlockSmem {
    static constexpr int S = 32 * E;
    // Offsets in floats for a CTA of rb rows.
    __host__ __device__ static size_t qk(int rb) { return static_cast<size_t>(rb) * S; }
    __host__ __device__ static size_t vbuf(int rb) { return qk(rb) + 2 * S; }
    __host__ __device__ static size_t ybuf(int rb) { return vbuf(rb) + rb; }
    __host__ __device__ static size_t scal(int rb) { return ybuf(rb) + rb; }       // 8 floats
    __host__ __device__ static size_t bars(int rb) { return scal(rb) + 8; }        // in floats, 8B aligned
    __host__ __device__ static size_t bytes(int rb) {
        return bars(rb) * sizeof(float) + kWarps * sizeof(uint64_t);
    }
};

// Conv1d + SiLU of one channel for one token, history oldest-first; the same
// operation order as the standalone conv kernel (current tap, then the history).
__device__ __forceinline__ float conv_channel(float x, const float4 w, float h0, float h1,
                                              float h2) {
    float pre = __fmul_rn(x, w.w);
    pre = __fmaf_rn(h0, w.x, pre);
    pre = __fmaf_rn(h1, w.y, pre);
    pre = __fmaf_rn(h2, w.z, pre);
    return silu(pre);
}

template <int E>
__global__ void __launch_bounds__(kThreads) block_decode_kernel(const BlockParams p) {
    constexpr int S = 32 * E;
    constexpr int kQKPerThread = (2 * S + kThreads - 1) / kThreads;
    using L = BlockSmem<E>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *sm = reinterpret_cast<float *>(smem_raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hk = p.n_k_heads, H = p.n_v_heads;
    const int csize = p.ratio * p.split;
    const int rank = static_cast<int>(cluster_ctarank());
    const int group = blockIdx.x / csize;
    const int n = group / Hk, kh = group % Hk;
    const int rr = rank / p.split, part = rank % p.split;
    const int vh = rr * Hk + kh;
    const int rb = S / p.split;            // rows of this CTA
    const int rows_per_warp = rb / kWarps;  // a multiple of kR
    const int row0 = part * rb;
    const int key_dim = Hk * S;
    const size_t conv_dim = static_cast<size_t>(2 * key_dim + H * S);
    const int slot = p.slots ? p.slots[n] : n;
    const bool valid = slot >= 0 && slot < p.pool;

    float *tile = sm;
    float *qk = sm + L::qk(rb);
    float *vbuf = sm + L::vbuf(rb);
    float *ybuf = sm + L::ybuf(rb);
    float *scal = sm + L::scal(rb);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::bars(rb)) + warp;

    const size_t head = static_cast<size_t>(slot) * H + vh;
    float *gstate = p.state + (head * S + row0 + warp * rows_per_warp) * S;
    float *wtile = tile + warp * rows_per_warp * S;
    const uint32_t tile_bytes = rows_per_warp * S * sizeof(float);

    // 1. state rows of this warp: one bulk copy, tracked by the warp's mbarrier.
    if (lane == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        if (valid) {
            mbar_arrive_expect_tx(bar, tile_bytes);
            bulk_g2s(wtile, gstate, tile_bytes, bar);
        }
    }

    // The gate input z and the norm weight of this CTA's rows (rb <= 128 < kThreads: at
    // most one each per thread), fetched now so their latency hides behind the state.
    static_assert(kThreads >= 128, "one output row per thread");
    const size_t ob = (static_cast<size_t>(n) * H + vh) * S + row0;
    float z_pre = 0.0f, w_pre = 0.0f;
    if (valid && tid < rb) {
        z_pre = p.z[ob + tid];
        w_pre = p.norm_w[row0 + tid];
    }

    // 2a. conv1d+SiLU of kh's q and k channels (old history read here).
    float nh[kQKPerThread][kTaps];
    const float *xrow = p.qkv + static_cast<size_t>(n) * conv_dim;
    if (valid) {
#pragma unroll
        for (int i = 0; i < kQKPerThread; ++i) {
            const int c = tid + i * kThreads;
            if (c < 2 * S) {
                const size_t ch = (c < S) ? static_cast<size_t>(kh) * S + c
                                          : static_cast<size_t>(key_dim) + kh * S + (c - S);
                const float x = xrow[ch];
                const float *hs = p.conv_state + (static_cast<size_t>(slot) * conv_dim + ch) * kTaps;
                const float h0 = hs[0], h1 = hs[1], h2 = hs[2];
                const float4 w = *reinterpret_cast<const float4 *>(p.conv_w + ch * 4);
                qk[c] = conv_channel(x, w, h0, h1, h2);
                nh[i][0] = h1; nh[i][1] = h2; nh[i][2] = x;
            }
        }
        // 2b. v channels of this CTA's rows: exclusively owned, rolled right away.
        for (int c = tid; c < rb; c += kThreads) {
            const size_t ch = static_cast<size_t>(2 * key_dim) + static_cast<size_t>(vh) * S + row0 + c;
            const float x = xrow[ch];
            float *hs = p.conv_state + (static_cast<size_t>(slot) * conv_dim + ch) * kTaps;
            const float h0 = hs[0], h1 = hs[1], h2 = hs[2];
            const float4 w = *reinterpret_cast<const float4 *>(p.conv_w + ch * 4);
            vbuf[c] = conv_channel(x, w, h0, h1, h2);
            hs[0] = h1; hs[1] = h2; hs[2] = x;
        }
        // 2c. decay gate and beta of this v-head.
        if (tid == 0) {
            const size_t nh_idx = static_cast<size_t>(n) * H + vh;
            const float gval = p.a[vh] * softplus_guarded(p.alpha[nh_idx] + p.dt[vh]);
            scal[0] = expf(gval);
            scal[1] = 1.0f / (1.0f + expf(-p.b[nh_idx]));
        }
    } else if (tid == 0 && kh == 0 && rank == 0 && p.err_count) {
        atomicAdd(p.err_count, 1);  // once per skipped sequence
    }
    // Phase 1 of the cluster barrier: this CTA has read kh's old q/k history.
    cluster_arrive_release();
    __syncthreads();

    // 2d. L2 norms of q (warp 0) and k (warp 1): x / max(||x||, eps).
    if (valid && warp < 2) {
        float x[E];
        load_vec<E>(x, qk + warp * S + lane * E);
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = __fmaf_rn(x[e], x[e], ss);
        ss = warp_allsum(ss);
        if (lane == 0) scal[2 + warp] = 1.0f / fmaxf(sqrtf(ss), p.l2_eps);
    }
    __syncthreads();

    // 3. the recurrence on this CTA's rows.
    bool ok = valid;
    if (valid) {
        float kk[E], qq[E];
        load_vec<E>(qq, qk + lane * E);
        load_vec<E>(kk, qk + S + lane * E);
        const float inv_q = scal[2], inv_k = scal[3];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            qq[e] *= inv_q;
            kk[e] *= inv_k;
        }
        const float decay = scal[0], bt = scal[1];
        __syncwarp();
        if (!mbar_wait(bar, 0)) {
            if (lane == 0) atomicOr(&g_watchdog, WD_STATE_COPY);
            ok = false;
        } else {
            int yr;
            const bool writer = [&] {
                yr = ((lane >> 4) & 1) | (((lane >> 3) & 1) << 1);
                return (lane & 7) == 0;
            }();
            for (int ps = 0; ps < rows_per_warp; ps += kR) {
                const int rl = warp * rows_per_warp + ps;  // first local row of this pass
                float row[kR][E], vv[kR];
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    load_vec<E>(row[r], tile + (rl + r) * S + lane * E);
                    vv[r] = vbuf[rl + r];
                }
                const float ysum = row_step<E, kR>(row, kk, qq, vv, decay, bt, lane);
#pragma unroll
                for (int r = 0; r < kR; ++r) store_vec<E>(gstate + (ps + r) * S + lane * E, row[r]);
                if (writer) ybuf[rl + yr] = __fmul_rn(p.scale, ysum);
            }
        }
    }
    if (!ok && valid) {
        // Never leave with a bulk copy still landing in this CTA's shared memory.
        mbar_wait(bar, 0);
    }
    __syncthreads();

    // 4. gated RMSNorm of this head's readout.
    if (warp == 0) {
        float ss = 0.0f;
        if (rb == S) {
            // Whole head here: the lane layout of the standalone gated-norm kernel,
            // so the two give the same bits.
            float yv[E];
            load_vec<E>(yv, ybuf + lane * E);
#pragma unroll
            for (int e = 0; e < E; ++e) ss = __fmaf_rn(yv[e], yv[e], ss);
        } else {
            for (int c = lane; c < rb; c += 32) ss = __fmaf_rn(ybuf[c], ybuf[c], ss);
        }
        ss = warp_allsum(ss);
        if (lane == 0) scal[4] = ss;
    }
    __syncthreads();         // the partial is visible to every warp of this CTA
    cluster_wait_acquire();  // phase 1 complete: every CTA has read the old q/k history
    float ss_total;
    if (p.split > 1) {
        cluster_arrive_release();  // phase 2: this CTA's partial is in shared memory
        cluster_wait_acquire();
        ss_total = 0.0f;
        for (int pp = 0; pp < p.split; ++pp)
            ss_total += ld_shared_cluster(scal + 4, static_cast<uint32_t>(rr * p.split + pp));
        cluster_arrive_release();  // phase 3: done reading the other CTAs' shared memory
    } else {
        ss_total = scal[4];
    }
    if (ok) {
        const float inv_rms = 1.0f / sqrtf(ss_total / static_cast<float>(S) + p.norm_eps);
        if (tid < rb) {
            p.out[ob + tid] = ybuf[tid] * inv_rms * w_pre * silu(z_pre);
        }
    }
    // Roll kh's q/k history, now that no CTA of the group will read it again.
    if (rank == 0 && valid) {
#pragma unroll
        for (int i = 0; i < kQKPerThread; ++i) {
            const int c = tid + i * kThreads;
            if (c < 2 * S) {
                const size_t ch = (c < S) ? static_cast<size_t>(kh) * S + c
                                          : static_cast<size_t>(key_dim) + kh * S + (c - S);
                float *hs = p.conv_state + (static_cast<size_t>(slot) * conv_dim + ch) * kTaps;
                hs[0] = nh[i][0]; hs[1] = nh[i][1]; hs[2] = nh[i][2];
            }
        }
    }
    if (p.split > 1) cluster_wait_acquire();  // keep shared memory alive for remote readers
}

// ============================================================================ persistent form
// For many sequences the cluster-per-group kernel leaves HBM idle between a CTA's
// load, compute and store phases. The persistent form keeps one CTA per SM alive
// for the whole step. Each CTA owns whole (sequence, k-head) groups, so it alone
// reads and rolls a group's q/k history (no cluster needed). Its warps have fixed
// roles and talk only through mbarriers, so no role ever waits at a CTA-wide
// barrier for another:
//   producer  (1 warp)  streams each group's state in units of 64 rows through a
//             ring of shared-memory stages (bulk copies, full/empty barriers) and
//             fetches the next group's qkv, conv history, conv weights and z into
//             a double buffer;
//   prologue  (4 warps) conv1d+SiLU of the group's channel slices (q and k, each
//             with its L2 norm, and one v slice per head) plus the gate and
//             beta, rolling the conv history, ahead of the row steps;
//   rows      (16 warps) the row steps, 4 rows per warp per unit;
//   epilogue  (2 warps) the gated RMSNorm of the finished group, a head each.
// Per-group operands and values rotate through three buffers: the producer refills
// buffer i%3 for group i once the epilogue of group i-3 has released it, so unit
// loads never wait on a recent group's prologue or epilogue.
constexpr int kPRowWarps = 16;
constexpr int kPProWarps = 4;
constexpr int kPEpiWarps = 2;
constexpr int kPProducer = kPRowWarps;      // warp index of the first warp of each role
constexpr int kPPro0 = kPRowWarps + 1;
constexpr int kPEpi0 = kPPro0 + kPProWarps;
constexpr int kPThreads = (kPRowWarps + 1 + kPProWarps + kPEpiWarps) * 32;
constexpr int kPUnitRows = kPRowWarps * kR;  // 64 state rows per ring stage
constexpr int kPMaxStages = 8;
constexpr int kPBufs = 3;  // depth of the per-group operand buffers and slots
constexpr int kPEarlyUnits = 1;  // state units issued before the first group's operands
constexpr int kPSmemBudget = 227 * 1024;

struct PLayout {
    int S, r, stages;
    size_t unit_bytes, gbuf_bytes, slot_floats, ring, gbuf, slot, bars, total;
    __host__ __device__ PLayout(int S_, int r_, int stages_) : S(S_), r(r_), stages(stages_) {
        unit_bytes = static_cast<size_t>(kPUnitRows) * S * sizeof(float);
        // per group: qkv slices, conv history, conv weights of the 2 + r channel
        // slices (q, k, one v per head), and z of the r heads
        gbuf_bytes = static_cast<size_t>((2 + r) * S * 8 + r * S) * sizeof(float);
        // per group slot: q^, k^ (normalised), v, y, decay, beta (padded to 16 B)
        slot_floats = (static_cast<size_t>(2 * S + 2 * r * S + 2 * r) + 3) / 4 * 4;
        ring = 0;
        gbuf = ring + stages * unit_bytes;
        slot = gbuf + kPBufs * gbuf_bytes;
        bars = slot + kPBufs * slot_floats * sizeof(float);
        // sfull/sempty[stages], gfull/gempty/cfull/yfull/cfree[kPBufs]; then the
        // per-stage and per-buffer issue counts and the abort flag
        total = bars + (2 * stages + 5 * kPBufs) * sizeof(uint64_t) +
                (stages + kPBufs + 1) * sizeof(int);
    }
};

// First conv channel of slice 0 = q of kh, 1 = k of kh, 2 + rr = v of v-head rr*Hk + kh.
__host__ __device__ inline size_t p_channel0(int slice, int kh, int S, int Hk) {
    const size_t key_dim = static_cast<size_t>(Hk) * S;
    if (slice == 0) return static_cast<size_t>(kh) * S;
    if (slice == 1) return key_dim + static_cast<size_t>(kh) * S;
    return 2 * key_dim + (static_cast<size_t>(slice - 2) * Hk + kh) * S;
}

// Conv1d+SiLU of E consecutive channels held by one lane (buffers in shared memory:
// x [E], history [3E], weights [4E]); writes the rolled history of those channels
// (3E consecutive floats) to global memory.
template <int E>
__device__ __forceinline__ void p_conv_lane(const float *X, const float *Hh, const float *W,
                                            float *hist_out, float (&val)[E]) {
    float x[E], h[3 * E];
    load_vec<E>(x, X);
    load_vec<3 * E>(h, Hh);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float4 w = *reinterpret_cast<const float4 *>(W + 4 * e);
        val[e] = conv_channel(x[e], w, h[3 * e], h[3 * e + 1], h[3 * e + 2]);
        h[3 * e] = h[3 * e + 1];
        h[3 * e + 1] = h[3 * e + 2];
        h[3 * e + 2] = x[e];
    }
    store_vec<3 * E>(hist_out, h);
}

template <int E>
__global__ void __launch_bounds__(kPThreads, 1) block_decode_persistent_kernel(const BlockParams p,
                                                                               int n_groups,
                                                                               int stages,
                                                                               int reverse) {
    constexpr int S = 32 * E;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int r = p.ratio;
    const PLayout L(S, r, stages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hk = p.n_k_heads, H = p.n_v_heads;
    const size_t conv_dim = static_cast<size_t>(2 * Hk * S + H * S);
    const int n_slices = 2 + r;
    const int units_per_head = S / kPUnitRows;
    const int units_per_group = r * units_per_head;

    uint64_t *sfull = reinterpret_cast<uint64_t *>(smem_raw + L.bars);
    uint64_t *sempty = sfull + stages;
    uint64_t *gfull = sempty + stages;
    uint64_t *gempty = gfull + kPBufs;
    uint64_t *cfull = gempty + kPBufs;   // prologue -> row warps
    uint64_t *yfull = cfull + kPBufs;    // row warps -> epilogue
    uint64_t *cfree = yfull + kPBufs;    // epilogue -> prologue
    int *s_issued = reinterpret_cast<int *>(cfree + kPBufs);  // [stages] uses issued per stage
    int *g_issued = s_issued + stages;                         // [kPBufs], then the abort flag
    volatile int *abort_flag = reinterpret_cast<volatile int *>(g_issued + kPBufs);

    if (tid == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(sfull + i, 1);
            mbar_init(sempty + i, kPRowWarps);
            s_issued[i] = 0;
        }
        for (int i = 0; i < kPBufs; ++i) {
            mbar_init(gfull + i, 1);
            mbar_init(gempty + i, kPProWarps + kPEpiWarps);
            mbar_init(cfull + i, kPProWarps);
            mbar_init(yfull + i, kPRowWarps);
            mbar_init(cfree + i, kPEpiWarps);
            g_issued[i] = 0;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // A wait that gives up raises the watchdog flag and sets `abort`; every role
    // then leaves its loop, and all threads meet at the final barrier.
    auto wait = [&](uint64_t *bar, int parity, unsigned bit) {
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity & 1)) return true;
        if (lane == 0) atomicOr(&g_watchdog, bit);
        *abort_flag = 1;
        return false;
    };
    auto slot_of = [&](int n) { return p.slots ? p.slots[n] : n; };
    auto valid_slot = [&](int slot) { return slot >= 0 && slot < p.pool; };
    auto gbuf_at = [&](int gb) { return reinterpret_cast<float *>(smem_raw + L.gbuf + gb * L.gbuf_bytes); };
    auto slot_at = [&](int cs) {
        return reinterpret_cast<float *>(smem_raw + L.slot + cs * L.slot_floats * sizeof(float));
    };
    // slot layout
    auto QH = [&](float *c) { return c; };
    auto KH = [&](float *c) { return c + S; };
    auto VV = [&](float *c) { return c + 2 * S; };
    auto YY = [&](float *c) { return c + 2 * S + r * S; };
    auto DEC = [&](float *c) { return c + 2 * S + 2 * r * S; };
    auto BET = [&](float *c) { return c + 2 * S + 2 * r * S + r; };

    int gi = 0;  // index of the valid group, shared by all roles
    // reverse: the groups in descending order, so that a launch starts on the groups the
    // previous one (ascending) wrote last, whose new state is still in L2
    for (int gf = blockIdx.x; gf < n_groups; gf += gridDim.x) {
        const int g = reverse ? n_groups - 1 - gf : gf;
        const int n = g / Hk, kh = g % Hk;
        const int slot = slot_of(n);
        if (!valid_slot(slot)) {
            if (warp == kPPro0 && lane == 0 && kh == 0 && p.err_count) atomicAdd(p.err_count, 1);
            continue;
        }
        const int use = gi / kPBufs, b = gi % kPBufs;  // gbuf and group slot rotate together
        ++gi;
        if (*abort_flag) break;
        float *gbuf = gbuf_at(b);
        float *X = gbuf, *Hh = X + n_slices * S, *W = Hh + 3 * n_slices * S;
        float *Z = W + 4 * n_slices * S;
        float *cslot = slot_at(b);

        if (warp == kPProducer) {
            // -------------------------------------------------------- producer
            bool ok = true;
            auto issue_unit = [&](int u) {
                const int unit = (gi - 1) * units_per_group + u;
                const int st = unit % stages, su = unit / stages;
                if (su > 0 && !wait(sempty + st, su - 1, WD_STAGE_FREE)) return false;
                if (lane == 0) {
                    const int rr = u / units_per_head, row0 = (u % units_per_head) * kPUnitRows;
                    const float *src =
                        p.state + ((static_cast<size_t>(slot) * H + rr * Hk + kh) * S + row0) * S;
                    mbar_arrive_expect_tx(sfull + st, static_cast<uint32_t>(L.unit_bytes));
                    bulk_g2s(smem_raw + L.ring + st * L.unit_bytes, src,
                             static_cast<uint32_t>(L.unit_bytes), sfull + st);
                    s_issued[st] = su + 1;
                }
                __syncwarp();
                return true;
            };
            // The CTA's first group: its first state unit goes out ahead of the operand
            // copies. At start-up that unit's arrival, not the prologue, gates the row
            // warps; one unit (4.9 MB over the GPU) delays the operands little, a whole
            // ring (19.5 MB) delays them more than it gains.
            const int early = gi == 1 ? (kPEarlyUnits < units_per_group ? kPEarlyUnits
                                                                        : units_per_group)
                                      : 0;
            for (int u = 0; u < early && ok; ++u) ok = issue_unit(u);
            if (!ok) break;
            if (use > 0 && !wait(gempty + b, use - 1, WD_STAGE_FREE)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(gfull + b, static_cast<uint32_t>(L.gbuf_bytes));
                g_issued[b] = use + 1;
            }
            __syncwarp();
            const int n_copies = 3 * n_slices + r;
            for (int c = lane; c < n_copies; c += 32) {
                if (c < n_slices) {
                    bulk_g2s(X + c * S, p.qkv + n * conv_dim + p_channel0(c, kh, S, Hk),
                             S * sizeof(float), gfull + b);
                } else if (c < 2 * n_slices) {
                    const int sl = c - n_slices;
                    bulk_g2s(Hh + sl * 3 * S,
                             p.conv_state + (slot * conv_dim + p_channel0(sl, kh, S, Hk)) * kTaps,
                             3 * S * sizeof(float), gfull + b);
                } else if (c < 3 * n_slices) {
                    const int sl = c - 2 * n_slices;
                    bulk_g2s(W + sl * 4 * S, p.conv_w + p_channel0(sl, kh, S, Hk) * 4,
                             4 * S * sizeof(float), gfull + b);
                } else {
                    const int rr = c - 3 * n_slices;
                    bulk_g2s(Z + rr * S, p.z + (static_cast<size_t>(n) * H + rr * Hk + kh) * S,
                             S * sizeof(float), gfull + b);
                }
            }
            for (int u = early; u < units_per_group && ok; ++u) ok = issue_unit(u);
            if (!ok) break;
        } else if (warp >= kPPro0 && warp < kPEpi0) {
            // -------------------------------------------------------- prologue
            const int pw = warp - kPPro0;
            // the gate inputs first, so their latency overlaps the convolutions
            const bool gate_lane = (pw == kPProWarps - 1) && lane < r;
            float g_alpha = 0.f, g_b = 0.f, g_dt = 0.f, g_a = 0.f;
            if (gate_lane) {
                const int vh = lane * Hk + kh;
                const size_t nh = static_cast<size_t>(n) * H + vh;
                g_alpha = p.alpha[nh];
                g_b = p.b[nh];
                g_dt = p.dt[vh];
                g_a = p.a[vh];
            }
            if (!wait(gfull + b, use, WD_STAGE_COPY)) break;
            if (use > 0 && !wait(cfree + b, use - 1, WD_STAGE_FREE)) break;
            // slice 0 = q, 1 = k (each L2-normalised), 2 + rr = v of head rr; lane L
            // takes channels [E*L, E*L+E) of the slice
            for (int sl = pw; sl < n_slices; sl += kPProWarps) {
                float val[E];
                const int c0 = sl * S + lane * E;
                p_conv_lane<E>(X + c0, Hh + 3 * c0, W + 4 * c0,
                               p.conv_state +
                                   (slot * conv_dim + p_channel0(sl, kh, S, Hk) + lane * E) * kTaps,
                               val);
                if (sl < 2) {  // x / max(||x||, eps)
                    float ss = 0.0f;
#pragma unroll
                    for (int e = 0; e < E; ++e) ss = __fmaf_rn(val[e], val[e], ss);
                    ss = warp_allsum(ss);
                    const float inv = 1.0f / fmaxf(sqrtf(ss), p.l2_eps);
#pragma unroll
                    for (int e = 0; e < E; ++e) val[e] *= inv;
                    store_vec<E>((sl ? KH(cslot) : QH(cslot)) + lane * E, val);
                } else {
                    store_vec<E>(VV(cslot) + (sl - 2) * S + lane * E, val);
                }
            }
            if (gate_lane) {
                DEC(cslot)[lane] = expf(g_a * softplus_guarded(g_alpha + g_dt));
                BET(cslot)[lane] = 1.0f / (1.0f + expf(-g_b));
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(gempty + b);  // done with X, H, W of this buffer
                mbar_arrive(cfull + b);
            }
        } else if (warp >= kPEpi0) {
            // -------------------------------------------------------- epilogue
            if (!wait(yfull + b, use, WD_STAGE_COPY)) break;
            if (!wait(gfull + b, use, WD_STAGE_COPY)) break;  // z of this group
            for (int rr = warp - kPEpi0; rr < r; rr += kPEpiWarps) {
                float yv[E], zv[E], wv[E], o[E];
                load_vec<E>(yv, YY(cslot) + rr * S + lane * E);
                load_vec<E>(zv, Z + rr * S + lane * E);
                load_vec<E>(wv, p.norm_w + lane * E);
                float ss = 0.0f;
#pragma unroll
                for (int e = 0; e < E; ++e) ss = __fmaf_rn(yv[e], yv[e], ss);
                ss = warp_allsum(ss);
                const float inv_rms = 1.0f / sqrtf(ss / static_cast<float>(S) + p.norm_eps);
#pragma unroll
                for (int e = 0; e < E; ++e) o[e] = yv[e] * inv_rms * wv[e] * silu(zv[e]);
                store_vec<E>(p.out + (static_cast<size_t>(n) * H + rr * Hk + kh) * S + lane * E, o);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(gempty + b);  // done with z
                mbar_arrive(cfree + b);   // slot reusable
            }
        } else {
            // -------------------------------------------------------- row warps
            if (!wait(cfull + b, use, WD_STAGE_COPY)) break;
            float kk[E], qq[E];
            load_vec<E>(qq, QH(cslot) + lane * E);
            load_vec<E>(kk, KH(cslot) + lane * E);
            int yr;
            const bool writer = [&] {
                yr = ((lane >> 4) & 1) | (((lane >> 3) & 1) << 1);
                return (lane & 7) == 0;
            }();
            bool ok = true;
            for (int u = 0; u < units_per_group; ++u) {
                const int unit = (gi - 1) * units_per_group + u;
                const int st = unit % stages, su = unit / stages;
                if (!wait(sfull + st, su, WD_STATE_COPY)) { ok = false; break; }
                const int rr = u / units_per_head;
                const int j0 = (u % units_per_head) * kPUnitRows + warp * kR;
                const int vh = rr * Hk + kh;
                const float *tile =
                    reinterpret_cast<const float *>(smem_raw + L.ring + st * L.unit_bytes) + warp * kR * S;
                float row[kR][E], vv[kR];
#pragma unroll
                for (int q = 0; q < kR; ++q) load_vec<E>(row[q], tile + q * S + lane * E);
                load_vec<kR>(vv, VV(cslot) + rr * S + j0);
                const float ysum =
                    row_step<E, kR>(row, kk, qq, vv, DEC(cslot)[rr], BET(cslot)[rr], lane);
                float *gst = p.state + ((static_cast<size_t>(slot) * H + vh) * S + j0) * S;
#pragma unroll
                for (int q = 0; q < kR; ++q) store_vec<E>(gst + q * S + lane * E, row[q]);
                if (writer) YY(cslot)[rr * S + j0 + yr] = __fmul_rn(p.scale, ysum);
                __syncwarp();
                if (lane == 0) mbar_arrive(sempty + st);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(yfull + b);
        }
    }
    // Never leave while a bulk copy may still be landing in shared memory.
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < stages; ++i)
            if (s_issued[i] > 0) mbar_wait(sfull + i, (s_issued[i] - 1) & 1);
        for (int i = 0; i < kPBufs; ++i)
            if (g_issued[i] > 0) mbar_wait(gfull + i, (g_issued[i] - 1) & 1);
    }
}

int sm_count() {
    static std::atomic<int> cached{0};
    int v = cached.load();
    if (v == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (v <= 0) v = 1;
        cached.store(v);
    }
    return v;
}

// Persistent form: one CTA per SM when there are at least two (sequence, k-head)
// groups per SM and the ring of 64-row stages fits in shared memory.
template <int E>
gdn_status launch_block_persistent(BlockParams p, int n_seqs, cudaStream_t s, bool &used) {
    constexpr int S = 32 * E;
    static_assert(S == 64 || S == 128, "the persistent form streams 64-row stages");
    used = false;
    const int ratio = p.n_v_heads / p.n_k_heads;
    const long long groups = static_cast<long long>(n_seqs) * p.n_k_heads;
    const int sms = sm_count();
    if (groups < 2LL * sms || groups > 0x7fffffffLL) return GDN_OK;
    int stages = kPMaxStages;
    while (stages >= 2 && PLayout(S, ratio, stages).total > static_cast<size_t>(kPSmemBudget)) --stages;
    if (stages < 2) return GDN_OK;
    p.ratio = ratio;
    p.split = 1;
    const size_t smem = PLayout(S, ratio, stages).total;
    if (cudaFuncSetAttribute(block_decode_persistent_kernel<E>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    used = true;
    // Consecutive decode steps walk the groups in alternating directions. A step leaves
    // the state it wrote last (tens of MB) dirty in L2; the next step, walking the other
    // way, reads that state first, from L2, instead of evicting it unread. The results do
    // not depend on the order (each group is independent).
    static std::atomic<unsigned> launches{0};
    const int reverse = static_cast<int>(launches.fetch_add(1, std::memory_order_relaxed) & 1u);
    block_decode_persistent_kernel<E><<<sms, kPThreads, smem, s>>>(p, static_cast<int>(groups), stages,
                                                                    reverse);
    return launch_status();
}

template <int E>
gdn_status launch_block(BlockParams p, int n_seqs, cudaStream_t s) {
    constexpr int S = 32 * E;
    if constexpr (E == 2 || E == 4) {
        bool used = false;
        const gdn_status pst = launch_block_persistent<E>(p, n_seqs, s, used);
        if (used || pst != GDN_OK) return pst;
    }
    const int ratio = p.n_v_heads / p.n_k_heads;
    // Smallest split that keeps the tile within shared memory, doubled while the
    // grid is short of two CTAs per SM; a CTA keeps at least 32 rows and a
    // cluster at most 8 CTAs.
    const int max_split = E < 8 / ratio ? E : 8 / ratio;
    int split = (S == 256) ? 2 : 1;
    while (split < max_split && static_cast<long long>(n_seqs) * p.n_v_heads * split < 2LL * sm_count())
        split *= 2;
    if (split > max_split || ratio > 8) return GDN_ERR_UNSUPPORTED;
    p.ratio = ratio;
    p.split = split;
    const int rb = S / split;
    const size_t smem = BlockSmem<E>::bytes(rb);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(block_decode_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return GDN_ERR_LAUNCH;
    }
    const long long blocks = static_cast<long long>(n_seqs) * p.n_k_heads * ratio * split;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ratio * split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, block_decode_kernel<E>, p) != cudaSuccess) return GDN_ERR_LAUNCH;
    return launch_status();
}

}  // namespace

// The bounded-wait self-test on this unit's watchdog flag (gdn_selftest_bounded_wait).
__global__ void wait_probe_kernel_block(int arm, unsigned long long limit_ns, float *out) {
    bounded_wait_probe(arm != 0, limit_ns, &g_watchdog, WD_STAGE_COPY, out);
}

gdn_status launch_wait_probe_block(bool arm, uint64_t limit_ns, float *out, cudaStream_t s) {
    wait_probe_kernel_block<<<1, 1, 0, s>>>(arm ? 1 : 0, limit_ns, out);
    return launch_status();
}

unsigned read_and_clear_watchdog_block(cudaStream_t s) {
    unsigned flags = 0;
    const unsigned zero = 0;
    cudaMemcpyFromSymbolAsync(&flags, g_watchdog, sizeof(flags), 0, cudaMemcpyDeviceToHost, s);
    cudaMemcpyToSymbolAsync(g_watchdog, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return flags;
}

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_block_decode(const float *qkv, const float *conv_w, float *conv_state,
                                       const float *alpha, const float *b, const float *dt,
                                       const float *a, const float *z, const float *norm_w,
                                       float *state, float *out, int n_seqs, int n_k_heads,
                                       int n_v_heads, int state_size, int conv_kernel,
                                       float scale, float l2_eps, float norm_eps,
                                       const int32_t *slots, int pool, int32_t *err_count,
                                       gdn_stream_t stream) {
    if (!qkv || !conv_w || !conv_state || !alpha || !b || !dt || !a || !z || !norm_w || !state ||
        !out)
        return GDN_ERR_NULL;
    if (n_seqs < 0) return GDN_ERR_SHAPE;
    if (conv_kernel < 2 || conv_kernel > 8) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (conv_kernel != 4) return GDN_ERR_UNSUPPORTED;
    if (n_v_heads / n_k_heads > 8) return GDN_ERR_UNSUPPORTED;
    if (!aligned16(qkv) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(state) ||
        !aligned16(z) || !aligned16(out) || !aligned16(norm_w))
        return GDN_ERR_ALIGN;
    if (n_seqs == 0) return GDN_OK;
    BlockParams p{qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, slots, err_count,
                  n_k_heads, n_v_heads, 0, 0, pool, scale, l2_eps, norm_eps};
    const cudaStream_t s = as_cuda(stream);
    switch (state_size) {
        case 32: return launch_block<1>(p, n_seqs, s);
        case 64: return launch_block<2>(p, n_seqs, s);
        case 128: return launch_block<4>(p, n_seqs, s);
        default: return launch_block<8>(p, n_seqs, s);
    }
}
