// gdn_prefill.cu -- the block over n_tokens positions per sequence (prefill): the
// conv scan fused with the q/k split + L2-norm, the decay gate, beta, the scan of
// the recurrence (sequential or chunked) and the gated RMSNorm, chained on one
// stream. Intermediates (q, k, v, g, beta) live in a workspace the caller provides
// (the library allocates nothing); the scan writes y straight into `out`, which the
// gated norm then rewrites in place.
//
// Follows the batched (prefill) variants of ssm_gated_delta.cu: decay gate, conv
// scan, q/k norm with the v passthrough, then the recurrence scan, per position.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr size_t kAlignFloats = 64;  // 256-byte sub-buffers

size_t round_up(size_t n) { return (n + kAlignFloats - 1) / kAlignFloats * kAlignFloats; }

// Intermediates of a call over `rows` positions in all (n_seqs * n_tokens for a uniform
// batch, the packed total for a ragged one).
struct PrefillLayout {
    size_t q, k, v, g, beta, total_floats;
    PrefillLayout(long long rows_ll, int hk, int h, int s) {
        const size_t rows = static_cast<size_t>(rows_ll);
        q = 0;
        k = q + round_up(rows * hk * s);
        v = k + round_up(rows * hk * s);
        g = v + round_up(rows * h * s);
        beta = g + round_up(rows * h);
        total_floats = beta + round_up(rows * h);
    }
};

// The conv scan and the q/k split + L2-norm in one pass: one warp per (head slice of S
// channels, block of positions, sequence), kConvNormWarps consecutive slices to a CTA.
// Lane L holds channels [E L, E L + E) of its slice, the split-norm kernel's lane layout,
// so a q or k head vector is normalised in registers with one butterfly, and each load
// and store moves E consecutive channels (one 16-byte access at E = 4). The conv is the
// conv scan's arithmetic (current tap, then the history oldest-first; the block at
// position 0 alone reads and rewrites conv_state) and the norm the split-norm kernel's,
// so the results are those two kernels' bit for bit, without their [n][t][C]
// intermediate in HBM.
constexpr int kConvNormWarps = 4;

template <int E>
__host__ __device__ constexpr int conv_norm_positions() { return E >= 8 ? 16 : 32; }
static_assert(conv_norm_positions<8>() == 16 && conv_norm_positions<4>() == 32,
              "the ragged grid check in prefill_impl assumes these block sizes");

// Grid, uniform batch: (group of slices, block of P positions, sequence). Ragged batch:
// (group of slices, block slot); block b of sequence n takes slot cu[n] / P + n + b (the
// chunk-slot scheme of the chunked scan: slots of consecutive sequences never collide
// and number at most total / P + n_seqs), so no CTA is launched for positions past a
// sequence's end.
template <int E, int K, bool RAGGED>
__global__ void __launch_bounds__(32 * kConvNormWarps) conv_split_norm_kernel(
    const float *__restrict__ qkv, const float *__restrict__ w, float *conv_state,
    float *__restrict__ q, float *__restrict__ k, float *__restrict__ v, const SeqMap seqs,
    int n_seqs, int n_k_heads, int n_v_heads, float eps, const int32_t *__restrict__ slots,
    int pool, int32_t *err_count) {
    constexpr int S = 32 * E, TAPS = K - 1, P = conv_norm_positions<E>();
    constexpr int B = E >= 8 ? 2 : 4;  // positions a load group holds
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hk = n_k_heads, H = n_v_heads;
    int n, t0;
    size_t seq0;   // first position of sequence n in the token-major arrays
    int n_tokens;  // its length
    if (!RAGGED) {
        n = blockIdx.z;
        t0 = blockIdx.y * P;
        seqs.range(n, seq0, n_tokens);
        const int slot_n = slots ? slots[n] : n;
        if (slot_n < 0 || slot_n >= pool) {  // uniform over the CTA
            if (err_count && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
                atomicAdd(err_count, 1);
            return;
        }
    } else {
        if (err_count && blockIdx.x == 0 && blockIdx.y == 0) {  // each skipped sequence once
            for (int m = threadIdx.x; m < n_seqs; m += blockDim.x) {
                const int slot_m = slots ? slots[m] : m;
                size_t a;
                int len;
                if (slot_m < 0 || slot_m >= pool || !seqs.range(m, a, len)) atomicAdd(err_count, 1);
            }
        }
        const long long cs = blockIdx.y;
        n = warp_seq_of_slot(seqs.cu, n_seqs, P, cs);  // each warp finds it; the same n
        if (n < 0 || !seqs.range(n, seq0, n_tokens)) return;  // uniform over the CTA
        const int slot_n = slots ? slots[n] : n;
        if (slot_n < 0 || slot_n >= pool) return;
        t0 = static_cast<int>(cs - (static_cast<long long>(seqs.cu[n]) / P + n)) * P;
    }
    const int sl = blockIdx.x * kConvNormWarps + warp;  // this warp's head slice
    if (sl >= 2 * Hk + H) return;  // uniform over the warp; no CTA barrier follows
    const int slot = slots ? slots[n] : n;
    const int t1 = min(n_tokens, t0 + P);
    if (t0 >= n_tokens) return;  // past the end of a shorter sequence: uniform over the CTA
    const size_t conv_dim = static_cast<size_t>(2 * Hk + H) * S;
    const size_t ch0 = static_cast<size_t>(sl) * S + E * lane;  // this lane's first channel
    float wc[K][E];
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
        for (int t = 0; t < K; ++t) wc[t][e] = w[(ch0 + e) * K + t];
    // the lane's channels' histories, channel-major: hs[e * TAPS + t]
    float *hs = conv_state + (static_cast<size_t>(slot) * conv_dim + ch0) * TAPS;
    const float *x_ptr = qkv + seq0 * conv_dim + ch0;
    float hist[TAPS][E];
#pragma unroll
    for (int t = 0; t < TAPS; ++t) {
        const int pos = t0 - TAPS + t;
        if (pos >= 0) {
            load_vec<E>(hist[t], x_ptr + static_cast<size_t>(pos) * conv_dim);
        } else {  // t0 == 0: the old state
#pragma unroll
            for (int e = 0; e < E; ++e) hist[t][e] = hs[e * TAPS + t];
        }
    }
    const bool is_qk = sl < 2 * Hk;  // uniform over the warp
    float *dst = is_qk ? (sl < Hk ? q : k) + (seq0 * Hk + (sl % Hk)) * S + E * lane
                       : v + (seq0 * H + (sl - 2 * Hk)) * S + E * lane;
    const size_t dst_step = static_cast<size_t>(is_qk ? Hk : H) * S;  // floats a position
    // position p from its input x: the conv, SiLU, the L2-norm of a q or k head vector,
    // the store, then x joins the history
    auto position = [&](const float (&x)[E], int p) {
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float pre = __fmul_rn(x[e], wc[K - 1][e]);
#pragma unroll
            for (int t = 0; t < TAPS; ++t) pre = __fmaf_rn(hist[t][e], wc[t][e], pre);
            o[e] = silu(pre);
        }
        if (is_qk) {
            float ss = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) ss = __fmaf_rn(o[e], o[e], ss);
            ss = warp_allsum(ss);
            const float inv = 1.0f / fmaxf(sqrtf(ss), eps);
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] *= inv;
        }
        store_vec<E>(dst + static_cast<size_t>(p) * dst_step, o);
#pragma unroll
        for (int t = 0; t + 1 < TAPS; ++t)
#pragma unroll
            for (int e = 0; e < E; ++e) hist[t][e] = hist[t + 1][e];
#pragma unroll
        for (int e = 0; e < E; ++e) hist[TAPS - 1][e] = x[e];
    };
    // whole groups of B positions without per-position checks, so that the independent
    // work of neighbouring positions can interleave, with the next group's loads issued
    // before the current group's work (two register buffers in turn); then the
    // sequence's last few positions
    int pb = t0;
    {
        float xa[B][E], xb[B][E];
        auto load_group = [&](float (&xg)[B][E], int p0) {
#pragma unroll
            for (int j = 0; j < B; ++j) load_vec<E>(xg[j], x_ptr + static_cast<size_t>(p0 + j) * conv_dim);
        };
        bool have = pb + B <= t1;  // uniform over the warp, as every condition below
        if (have) load_group(xa, pb);
        while (have) {
            const bool next_b = pb + 2 * B <= t1;
            if (next_b) load_group(xb, pb + B);
#pragma unroll
            for (int j = 0; j < B; ++j) position(xa[j], pb + j);
            pb += B;
            if (!next_b) break;
            const bool next_a = pb + 2 * B <= t1;
            if (next_a) load_group(xa, pb + B);
#pragma unroll
            for (int j = 0; j < B; ++j) position(xb[j], pb + j);
            pb += B;
            have = next_a;
        }
    }
    if (pb < t1) {
        float xs[B][E];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (pb + j < t1) {
                load_vec<E>(xs[j], x_ptr + static_cast<size_t>(pb + j) * conv_dim);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) xs[j][e] = 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (pb + j >= t1) break;  // uniform over the warp
            position(xs[j], pb + j);
        }
    }
    if (t0 == 0) {
        // the new state: the last K-1 inputs of (old state, this call's inputs); entry t
        // is input n_tokens - TAPS + t, or old entry n_tokens + t where that is negative
        // (the old state is read before this lane rewrites it; no other thread touches it)
        float nw[TAPS][E];
#pragma unroll
        for (int t = 0; t < TAPS; ++t) {
            const int pos = n_tokens - TAPS + t;
            if (pos >= 0) {
                load_vec<E>(nw[t], x_ptr + static_cast<size_t>(pos) * conv_dim);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) nw[t][e] = hs[e * TAPS + pos + TAPS];
            }
        }
#pragma unroll
        for (int t = 0; t < TAPS; ++t)
#pragma unroll
            for (int e = 0; e < E; ++e) hs[e * TAPS + t] = nw[t][e];
    }
}

template <int E, int K>
gdn_status launch_conv_split_norm_k(const float *qkv, const float *w, float *conv_state, float *q,
                                    float *k, float *v, int n_seqs, SeqMap seqs, int Hk, int H,
                                    float eps, const int32_t *slots, int pool, int32_t *err_count,
                                    cudaStream_t s) {
    constexpr int P = conv_norm_positions<E>();
    const unsigned groups = (2 * Hk + H + kConvNormWarps - 1) / kConvNormWarps;
    if (seqs.cu == nullptr) {
        const dim3 grid(groups, (seqs.n_tokens + P - 1) / P, n_seqs);
        conv_split_norm_kernel<E, K, false><<<grid, 32 * kConvNormWarps, 0, s>>>(
            qkv, w, conv_state, q, k, v, seqs, n_seqs, Hk, H, eps, slots, pool, err_count);
    } else {
        const long long block_slots = seqs.total / P + n_seqs;
        if (block_slots > 65535) return GDN_ERR_UNSUPPORTED;
        const dim3 grid(groups, static_cast<unsigned>(block_slots), 1);
        conv_split_norm_kernel<E, K, true><<<grid, 32 * kConvNormWarps, 0, s>>>(
            qkv, w, conv_state, q, k, v, seqs, n_seqs, Hk, H, eps, slots, pool, err_count);
    }
    return launch_status();
}

template <int E>
gdn_status launch_conv_split_norm(int conv_kernel, const float *qkv, const float *w,
                                  float *conv_state, float *q, float *k, float *v, int n_seqs,
                                  SeqMap seqs, int Hk, int H, float eps, const int32_t *slots,
                                  int pool, int32_t *err_count, cudaStream_t s) {
    switch (conv_kernel) {
        case 2: return launch_conv_split_norm_k<E, 2>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
        case 3: return launch_conv_split_norm_k<E, 3>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
        case 4: return launch_conv_split_norm_k<E, 4>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
        case 5: return launch_conv_split_norm_k<E, 5>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
        case 6: return launch_conv_split_norm_k<E, 6>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
        case 7: return launch_conv_split_norm_k<E, 7>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
        default: return launch_conv_split_norm_k<E, 8>(qkv, w, conv_state, q, k, v, n_seqs, seqs, Hk, H, eps, slots, pool, err_count, s);
    }
}


// The decay gate and beta of the block's rows in one pass, thread per (row, head):
// g = a[h] * softplus(alpha + dt[h]) (fm_kernel_ssm.m, "Decay gate"; ssm_gated_delta.cu,
// fc_ssm_decay_gate_nx) and beta = sigmoid(b) (ssm_gated_delta.cu, fc_sigmoid), with the
// operations of gdn_decay_gate and gdn_beta_sigmoid, so the same bits.
constexpr int kGateThreads = 256;
__global__ void __launch_bounds__(kGateThreads) gate_beta_kernel(
    const float *__restrict__ alpha, const float *__restrict__ dt, const float *__restrict__ a,
    const float *__restrict__ b, float *__restrict__ g, float *__restrict__ beta, int n_heads,
    long long total) {
    const long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (idx >= total) return;
    const int h = static_cast<int>(idx % n_heads);
    g[idx] = a[h] * softplus_guarded(alpha[idx] + dt[h]);
    beta[idx] = 1.0f / (1.0f + expf(-b[idx]));
}

// The conv history after every position, for speculative-decoding rollback: the K-1
// raw inputs ending at position t, oldest first (snaps [n][t][C][K-1], the conv_state
// layout of one slot per position), positions before the call read from the old
// conv_state. Runs before the conv pass rolls conv_state; copies only.
constexpr int kHistThreads = 256;

__global__ void __launch_bounds__(kHistThreads) conv_history_snapshots_kernel(
    const float *__restrict__ qkv, const float *__restrict__ conv_state,
    float *__restrict__ snaps, const SeqMap seqs, int conv_dim, int taps,
    const int32_t *__restrict__ slots, int pool) {
    const int c = blockIdx.x * kHistThreads + threadIdx.x, t = blockIdx.y, n = blockIdx.z;
    const int slot = slots ? slots[n] : n;
    size_t row;  // first position of sequence n
    int n_tokens;
    // a skipped sequence is counted by the conv pass
    if (c >= conv_dim || slot < 0 || slot >= pool || !seqs.range(n, row, n_tokens)) return;
    if (t >= n_tokens) return;
    float *dst = snaps + ((row + t) * conv_dim + c) * taps;
    for (int j = 0; j < taps; ++j) {
        const int pos = t - (taps - 1) + j;
        dst[j] = pos >= 0 ? qkv[(row + pos) * conv_dim + c]
                          : conv_state[(static_cast<size_t>(slot) * conv_dim + c) * taps + taps + pos];
    }
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_block_prefill_workspace_size(int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                                        int state_size) {
    if (n_seqs < 0 || n_tokens < 0 || n_k_heads < 1 || n_v_heads < 1 || state_size < 1) return 0;
    return PrefillLayout(static_cast<long long>(n_seqs) * n_tokens, n_k_heads, n_v_heads,
                         state_size).total_floats * sizeof(float);
}

size_t gdn_block_prefill_chunked_workspace_size(int n_seqs, int n_tokens, int n_k_heads,
                                                int n_v_heads, int state_size) {
    const size_t base =
        gdn_block_prefill_workspace_size(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size);
    if (base == 0 || state_size != 128) return base;
    return (base + 15) / 16 * 16 +
           gdn_recurrence_scan_chunked_ws_size(n_seqs, n_tokens, n_v_heads, state_size);
}

}  // extern "C"

namespace {

// The prefill block with either scan: the sequential one (bit for bit the fused
// decode step, position after position) or the chunked tensor-core one, over a
// uniform batch (seqs.cu NULL: n_seqs x seqs.n_tokens positions) or a ragged one
// (seqs.total packed positions; seqs.n_tokens bounds one sequence's length).
gdn_status prefill_impl(const float *qkv, const float *conv_w, float *conv_state,
                        const float *alpha, const float *b, const float *dt, const float *a,
                        const float *z, const float *norm_w, float *state, float *out,
                        int n_seqs, SeqMap seqs, int n_k_heads, int n_v_heads, int state_size,
                        int conv_kernel, float scale, float l2_eps, float norm_eps,
                        const int32_t *slots, int pool, int32_t *err_count, void *workspace,
                        size_t workspace_bytes, gdn_stream_t stream, bool chunked,
                        float *snaps = nullptr, float *conv_snaps = nullptr) {
    if (!qkv || !conv_w || !conv_state || !alpha || !b || !dt || !a || !z || !norm_w || !state ||
        !out)
        return GDN_ERR_NULL;
    const bool snapshots = snaps != nullptr;  // the snapshot form passes both, non-NULL
    const int n_tokens = seqs.n_tokens;       // positions of a sequence (ragged: at most)
    if (n_seqs < 0 || n_tokens < 0 || seqs.total < 0) return GDN_ERR_SHAPE;
    if (conv_kernel < 2 || conv_kernel > 8) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    if (chunked && state_size != 128) return GDN_ERR_UNSUPPORTED;
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(qkv) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(state) ||
        !aligned16(z) || !aligned16(out) || !aligned16(norm_w))
        return GDN_ERR_ALIGN;
    if (n_seqs == 0 || n_tokens == 0 || seqs.total == 0) return GDN_OK;
    const long long rows = seqs.total;  // positions in all
    const PrefillLayout L(rows, n_k_heads, n_v_heads, state_size);
    if (!workspace) return GDN_ERR_NULL;
    if (workspace_bytes < L.total_floats * sizeof(float)) return GDN_ERR_SHAPE;
    if (!aligned16(workspace)) return GDN_ERR_ALIGN;
    if (rows * n_v_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const int S = state_size, H = n_v_heads, Hk = n_k_heads;
    float *ws = static_cast<float *>(workspace);
    float *q = ws + L.q, *k = ws + L.k, *v = ws + L.v;
    float *g = ws + L.g, *beta = ws + L.beta;
    if ((n_tokens + 31) / 32 > 65535 || n_seqs > 65535) return GDN_ERR_UNSUPPORTED;
    if (snapshots && n_tokens > 65535) return GDN_ERR_UNSUPPORTED;  // positions on grid.y
    if (seqs.cu) {  // the ragged grids, checked before anything is enqueued
        const long long per_block = S >= 256 ? 16 : 32;  // conv_norm_positions
        if (rows / per_block + n_seqs > 65535) return GDN_ERR_UNSUPPORTED;
        if (chunked && (rows / 32 + n_seqs) * n_k_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    }

    // A skipped sequence is counted once, by the conv pass; nothing of it is written
    // to conv_state, state or out.
    const cudaStream_t cs = as_cuda(stream);
    if (snapshots) {
        const int C = (2 * Hk + H) * S;
        const dim3 grid((C + kHistThreads - 1) / kHistThreads, n_tokens, n_seqs);
        conv_history_snapshots_kernel<<<grid, kHistThreads, 0, cs>>>(
            qkv, conv_state, conv_snaps, seqs, C, conv_kernel - 1, slots, pool);
        GDN_TRY(launch_status());
    }
    switch (S) {
        case 32: GDN_TRY(launch_conv_split_norm<1>(conv_kernel, qkv, conv_w, conv_state, q, k, v, n_seqs, seqs, Hk, H, l2_eps, slots, pool, err_count, cs)); break;
        case 64: GDN_TRY(launch_conv_split_norm<2>(conv_kernel, qkv, conv_w, conv_state, q, k, v, n_seqs, seqs, Hk, H, l2_eps, slots, pool, err_count, cs)); break;
        case 128: GDN_TRY(launch_conv_split_norm<4>(conv_kernel, qkv, conv_w, conv_state, q, k, v, n_seqs, seqs, Hk, H, l2_eps, slots, pool, err_count, cs)); break;
        default: GDN_TRY(launch_conv_split_norm<8>(conv_kernel, qkv, conv_w, conv_state, q, k, v, n_seqs, seqs, Hk, H, l2_eps, slots, pool, err_count, cs)); break;
    }
    {
        const long long total = rows * H;
        gate_beta_kernel<<<static_cast<unsigned>((total + kGateThreads - 1) / kGateThreads),
                           kGateThreads, 0, cs>>>(alpha, dt, a, b, g, beta, H, total);
        GDN_TRY(launch_status());
    }
    if (chunked && seqs.cu == nullptr) {
        // the two-phase form in the bytes past the intermediates, if they hold one chunk
        const size_t base = (L.total_floats * sizeof(float) + 15) / 16 * 16;
        const size_t one_chunk = gdn_recurrence_scan_chunked_ws_size(n_seqs, 1, H, S);
        if (workspace_bytes >= base + one_chunk) {
            GDN_TRY(gdn_recurrence_scan_chunked_ws(state, q, k, v, g, beta, out, n_seqs, n_tokens,
                                                   Hk, H, S, scale, slots, pool, nullptr,
                                                   static_cast<char *>(workspace) + base,
                                                   workspace_bytes - base, stream));
        } else {
            GDN_TRY(gdn_recurrence_scan_chunked(state, q, k, v, g, beta, out, n_seqs, n_tokens,
                                                Hk, H, S, scale, slots, pool, nullptr, stream));
        }
    } else if (chunked) {
        // ragged: the two-phase form if the bytes past the intermediates hold every chunk
        const size_t base = (L.total_floats * sizeof(float) + 15) / 16 * 16;
        GDN_TRY(launch_chunked_seqs(state, q, k, v, g, beta, out, n_seqs, seqs, Hk, H, scale,
                                    slots, pool, nullptr,
                                    workspace_bytes > base ? static_cast<char *>(workspace) + base
                                                           : nullptr,
                                    workspace_bytes > base ? workspace_bytes - base : 0, cs));
    } else {
        GDN_TRY(launch_scan_seqs(state, q, k, v, g, beta, out, n_seqs, seqs, Hk, H, S, scale,
                                 slots, pool, nullptr, snapshots ? snaps : nullptr, cs));
    }
    return launch_gated_norm_seqs(out, norm_w, z, out, rows * H, S, norm_eps, H, n_seqs, seqs,
                                  slots, pool, cs);
}

}  // namespace

extern "C" {

gdn_status gdn_block_prefill(const float *qkv, const float *conv_w, float *conv_state,
                             const float *alpha, const float *b, const float *dt, const float *a,
                             const float *z, const float *norm_w, float *state, float *out,
                             int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                             int state_size, int conv_kernel, float scale, float l2_eps,
                             float norm_eps, const int32_t *slots, int pool, int32_t *err_count,
                             void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    return prefill_impl(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                        uniform_seqs(n_seqs, n_tokens), n_k_heads, n_v_heads, state_size,
                        conv_kernel, scale, l2_eps,
                        norm_eps, slots, pool, err_count, workspace, workspace_bytes, stream, false);
}

gdn_status gdn_block_prefill_snapshots(const float *qkv, const float *conv_w,
                                       float *conv_state, const float *alpha, const float *b,
                                       const float *dt, const float *a, const float *z,
                                       const float *norm_w, float *state, float *out,
                                       float *snaps, float *conv_snaps, int n_seqs,
                                       int n_tokens, int n_k_heads, int n_v_heads,
                                       int state_size, int conv_kernel, float scale,
                                       float l2_eps, float norm_eps, const int32_t *slots,
                                       int pool, int32_t *err_count, void *workspace,
                                       size_t workspace_bytes, gdn_stream_t stream) {
    if (!snaps || !conv_snaps) return GDN_ERR_NULL;
    if (!aligned16(snaps)) return GDN_ERR_ALIGN;
    return prefill_impl(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                        uniform_seqs(n_seqs, n_tokens), n_k_heads, n_v_heads, state_size,
                        conv_kernel, scale, l2_eps,
                        norm_eps, slots, pool, err_count, workspace, workspace_bytes, stream, false,
                        snaps, conv_snaps);
}

gdn_status gdn_block_prefill_chunked(const float *qkv, const float *conv_w, float *conv_state,
                                     const float *alpha, const float *b, const float *dt,
                                     const float *a, const float *z, const float *norm_w,
                                     float *state, float *out, int n_seqs, int n_tokens,
                                     int n_k_heads, int n_v_heads, int state_size,
                                     int conv_kernel, float scale, float l2_eps, float norm_eps,
                                     const int32_t *slots, int pool, int32_t *err_count,
                                     void *workspace, size_t workspace_bytes,
                                     gdn_stream_t stream) {
    return prefill_impl(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                        uniform_seqs(n_seqs, n_tokens), n_k_heads, n_v_heads, state_size,
                        conv_kernel, scale, l2_eps,
                        norm_eps, slots, pool, err_count, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

// ============================================================================ ragged batches
// The prefill block over sequences of different lengths packed token-major: sequence
// n owns positions cu_seqlens[n] .. cu_seqlens[n+1] - 1 of every [total][...] array.
// Each kernel finds its sequence's range through the same SeqMap as the uniform
// calls, so a sequence gets the bits it would get in a call of its own.
extern "C" {

size_t gdn_block_prefill_varlen_workspace_size(int n_seqs, int total_tokens, int n_k_heads,
                                               int n_v_heads, int state_size) {
    if (n_seqs < 0 || total_tokens < 0 || n_k_heads < 1 || n_v_heads < 1 || state_size < 1)
        return 0;
    return PrefillLayout(total_tokens, n_k_heads, n_v_heads, state_size).total_floats *
           sizeof(float);
}

size_t gdn_block_prefill_chunked_varlen_workspace_size(int n_seqs, int total_tokens,
                                                       int n_k_heads, int n_v_heads,
                                                       int state_size) {
    const size_t base = gdn_block_prefill_varlen_workspace_size(n_seqs, total_tokens, n_k_heads,
                                                                n_v_heads, state_size);
    if (base == 0 || state_size != 128 || n_seqs < 1) return base;
    return (base + 15) / 16 * 16 + ragged_chunked_ws_size(n_seqs, total_tokens, n_v_heads);
}

gdn_status gdn_block_prefill_varlen(const float *qkv, const float *conv_w, float *conv_state,
                                    const float *alpha, const float *b, const float *dt,
                                    const float *a, const float *z, const float *norm_w,
                                    float *state, float *out, const int32_t *cu_seqlens,
                                    int n_seqs, int total_tokens, int max_tokens, int n_k_heads,
                                    int n_v_heads, int state_size, int conv_kernel, float scale,
                                    float l2_eps, float norm_eps, const int32_t *slots, int pool,
                                    int32_t *err_count, void *workspace, size_t workspace_bytes,
                                    gdn_stream_t stream) {
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    return prefill_impl(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                        SeqMap{cu_seqlens, max_tokens, total_tokens}, n_k_heads, n_v_heads,
                        state_size, conv_kernel, scale, l2_eps, norm_eps, slots, pool, err_count,
                        workspace, workspace_bytes, stream, false);
}

gdn_status gdn_block_prefill_chunked_varlen(const float *qkv, const float *conv_w,
                                            float *conv_state, const float *alpha,
                                            const float *b, const float *dt, const float *a,
                                            const float *z, const float *norm_w, float *state,
                                            float *out, const int32_t *cu_seqlens, int n_seqs,
                                            int total_tokens, int max_tokens, int n_k_heads,
                                            int n_v_heads, int state_size, int conv_kernel,
                                            float scale, float l2_eps, float norm_eps,
                                            const int32_t *slots, int pool, int32_t *err_count,
                                            void *workspace, size_t workspace_bytes,
                                            gdn_stream_t stream) {
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    return prefill_impl(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                        SeqMap{cu_seqlens, max_tokens, total_tokens}, n_k_heads, n_v_heads,
                        state_size, conv_kernel, scale, l2_eps, norm_eps, slots, pool, err_count,
                        workspace, workspace_bytes, stream, true);
}

gdn_status gdn_block_prefill_snapshots_varlen(
    const float *qkv, const float *conv_w, float *conv_state, const float *alpha, const float *b,
    const float *dt, const float *a, const float *z, const float *norm_w, float *state, float *out,
    float *snaps, float *conv_snaps, const int32_t *cu_seqlens, int n_seqs, int total_tokens,
    int max_tokens, int n_k_heads, int n_v_heads, int state_size, int conv_kernel, float scale,
    float l2_eps, float norm_eps, const int32_t *slots, int pool, int32_t *err_count,
    void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    if (!snaps || !conv_snaps) return GDN_ERR_NULL;
    if (!aligned16(snaps)) return GDN_ERR_ALIGN;
    return prefill_impl(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out, n_seqs,
                        SeqMap{cu_seqlens, max_tokens, total_tokens}, n_k_heads, n_v_heads,
                        state_size, conv_kernel, scale, l2_eps, norm_eps, slots, pool, err_count,
                        workspace, workspace_bytes, stream, false, snaps, conv_snaps);
}

}  // extern "C"

// ============================================================================ no allocation
// An allocation-free form of gdn_block_prefill for callers that cannot allocate
// device memory: a plugin that only ever receives the input and output buffers of
// the engine hosting it, or a serving loop that must not allocate in the middle
// of a step (a device allocation can synchronise the whole device). Its workspace
// is a fixed array in device memory that every GPU loading this library holds
// until the process exits.
#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = GDN_PREFILL_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// In host code this name is only a stand-in for the array, not its device address.
static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

// Device address of g_prefill_scratch on the current device, looked up on the
// first call per device (with that device current) and remembered.
gdn_status scratch_on_current_device(void **out) {
    static std::mutex lock;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_LAUNCH;
    std::lock_guard<std::mutex> guard(lock);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || p == nullptr)
            return GDN_ERR_LAUNCH;
        addr[dev] = p;
    }
    *out = addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_block_prefill_noalloc(
    const float *qkv, const float *conv_w, float *conv_state, const float *alpha, const float *b,
    const float *dt, const float *a, const float *z, const float *norm_w, float *state, float *out,
    int n_seqs, int n_tokens, int n_k_heads, int n_v_heads, int state_size, int conv_kernel,
    float scale, float l2_eps, float norm_eps, const int32_t *slots, int pool, int32_t *err_count,
    gdn_stream_t stream) {
    if (n_seqs < 0 || n_tokens < 0 || n_k_heads < 1 || n_v_heads < 1 || state_size < 1)
        return GDN_ERR_SHAPE;
    const size_t need = PrefillLayout(static_cast<long long>(n_seqs) * n_tokens, n_k_heads,
                                      n_v_heads, state_size).total_floats * sizeof(float);
    if (need > kNoAllocScratchBytes) return GDN_ERR_UNSUPPORTED;  // beyond the fixed scratch
    void *scratch = nullptr;
    GDN_TRY(scratch_on_current_device(&scratch));
    // Nothing needs clearing: every scratch value that can reach an output is written
    // earlier in the same call (rows of a skipped sequence are read but never used).
    return gdn_block_prefill(qkv, conv_w, conv_state, alpha, b, dt, a, z, norm_w, state, out,
                             n_seqs, n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel,
                             scale, l2_eps, norm_eps, slots, pool, err_count, scratch,
                             kNoAllocScratchBytes, stream);
}
