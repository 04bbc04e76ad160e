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
        const size_t ob = (static_cast<size_t>(n) * H + vh) * S + row0;
        for (int c = tid; c < rb; c += kThreads) {
            const float zv = p.z[ob + c];
            p.out[ob + c] = ybuf[c] * inv_rms * p.norm_w[row0 + c] * silu(zv);
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

template <int E>
gdn_status launch_block(BlockParams p, int n_seqs, cudaStream_t s) {
    constexpr int S = 32 * E;
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
    if (!aligned16(qkv) || !aligned16(conv_w) || !aligned16(state) || !aligned16(z) ||
        !aligned16(out) || !aligned16(norm_w))
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
