// gdn_misc.cu -- the small per-token steps of the block as standalone kernels:
// decay gate, beta sigmoid, causal conv1d + SiLU (single token and scan), q/k
// split + L2-norm, gated RMSNorm; plus the status helpers of the C ABI.
//
// These steps move a few bytes per channel and are HBM/latency bound; they use
// one thread per element (conv: per channel, history in registers across tokens)
// or one warp per head vector with a shuffle reduction.
#include <cstdio>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// fm_kernel_ssm.m, "Decay gate"; ssm_gated_delta.cu, fc_ssm_decay_gate_nx: one
// thread per (row, head).
__global__ void __launch_bounds__(kThreads) decay_gate_kernel(const float *__restrict__ alpha,
                                                               const float *__restrict__ dt,
                                                               const float *__restrict__ a,
                                                               float *g, int n_heads,
                                                               long long total) {
    const long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (idx >= total) return;
    const int h = static_cast<int>(idx % n_heads);
    g[idx] = a[h] * softplus_guarded(alpha[idx] + dt[h]);
}

// ssm_gated_delta.cu, fc_sigmoid.
__global__ void __launch_bounds__(kThreads) sigmoid_kernel(const float *__restrict__ b,
                                                            float *beta, long long n) {
    const long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (i < n) beta[i] = 1.0f / (1.0f + expf(-b[i]));
}

// Causal depthwise conv1d + SiLU over n_tokens positions, fm_kernel_ssm.m "Causal
// depthwise conv1d + SiLU" and its scan form. The history holds RAW inputs, so the
// window of position p is just inputs p-K+1 .. p (the old conv_state standing in
// for p < 0): positions are independent, and the scan runs in blocks of
// kConvTokens positions, one thread per (sequence, V consecutive channels, block),
// each carrying its K-1 taps in registers across its block. V = 4 where the channel
// count and the qkv and out pointers allow 16-byte accesses, else 1. The block of
// position 0 alone reads the old conv_state and writes the new one (the last K-1 raw
// inputs), so the in-place update cannot race. The accumulation is the current tap
// first, then the history oldest-first, per channel whatever V is; every position is
// computed with the same operations as a single-token call, so a scan and n
// single-token calls agree bit for bit.
constexpr int kConvTokens = 64;
static_assert(kConvTokens >= 8, "a block's history must reach back no further than position 0");

template <int K, bool SNAP, int V>
__global__ void __launch_bounds__(kThreads) conv1d_silu_kernel(
    const float *__restrict__ qkv, const float *__restrict__ w, float *conv_state,
    float *__restrict__ out, int n_tokens, int conv_dim, const int32_t *__restrict__ slots,
    int pool, int32_t *err_count, float *__restrict__ snaps) {
    constexpr int TAPS = K - 1, B = 16 / V;  // B: positions a load group holds
    const int n = blockIdx.y;
    const int c0 = (blockIdx.x * kThreads + threadIdx.x) * V;  // this thread's first channel
    const int t0 = blockIdx.z * kConvTokens;
    const int t1 = min(n_tokens, t0 + kConvTokens);
    const int slot = slots ? slots[n] : n;
    if (slot < 0 || slot >= pool) {
        if (err_count && blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            atomicAdd(err_count, 1);
        return;
    }
    if (c0 >= conv_dim) return;  // V divides conv_dim
    float wc[K][V];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int t = 0; t < K; ++t) wc[t][v] = w[static_cast<size_t>(c0 + v) * K + t];
    // the thread's channels' histories, channel-major: hs[v * TAPS + t]
    float *hs = conv_state + (static_cast<size_t>(slot) * conv_dim + c0) * TAPS;
    const float *x_ptr = qkv + static_cast<size_t>(n) * n_tokens * conv_dim + c0;
    float *o_ptr = out + static_cast<size_t>(n) * n_tokens * conv_dim + c0;
    // inputs at positions t0-K+1 .. t0-1 (the old state for negative positions)
    float hist[TAPS][V];
#pragma unroll
    for (int t = 0; t < TAPS; ++t) {
        const int pos = t0 - TAPS + t;
        if (pos >= 0) {
            load_vec<V>(hist[t], x_ptr + static_cast<size_t>(pos) * conv_dim);
        } else {  // t0 == 0
#pragma unroll
            for (int v = 0; v < V; ++v) hist[t][v] = hs[v * TAPS + t];
        }
    }
    auto position = [&](const float (&x)[V], int p) {
        float o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float pre = __fmul_rn(x[v], wc[K - 1][v]);
#pragma unroll
            for (int t = 0; t < TAPS; ++t) pre = __fmaf_rn(hist[t][v], wc[t][v], pre);
            o[v] = silu(pre);
        }
        store_vec<V>(o_ptr + static_cast<size_t>(p) * conv_dim, o);
#pragma unroll
        for (int t = 0; t + 1 < TAPS; ++t)
#pragma unroll
            for (int v = 0; v < V; ++v) hist[t][v] = hist[t + 1][v];
#pragma unroll
        for (int v = 0; v < V; ++v) hist[TAPS - 1][v] = x[v];
        if constexpr (SNAP) {  // the history after token p: snaps[n][p][C][K-1]
            float *sn = snaps + ((static_cast<size_t>(n) * n_tokens + p) * conv_dim + c0) * TAPS;
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int t = 0; t < TAPS; ++t) sn[v * TAPS + t] = hist[t][v];
        }
    };
    // whole groups of B positions without per-position checks, the next group's loads
    // issued before the current group's work (two register buffers in turn); then the
    // block's last few positions
    int pb = t0;
    {
        float xa[B][V], xb[B][V];
        auto load_group = [&](float (&xg)[B][V], int p0) {
#pragma unroll
            for (int j = 0; j < B; ++j) load_vec<V>(xg[j], x_ptr + static_cast<size_t>(p0 + j) * conv_dim);
        };
        bool have = pb + B <= t1;
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
        float xs[B][V];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (pb + j < t1) {
                load_vec<V>(xs[j], x_ptr + static_cast<size_t>(pb + j) * conv_dim);
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) xs[j][v] = 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (pb + j >= t1) break;
            position(xs[j], pb + j);
        }
    }
    if (t0 == 0) {
        // the new state: the last K-1 inputs of (old state, this call's inputs); entry t
        // is input n_tokens - TAPS + t, or old entry n_tokens + t where that is negative
        // (the old state is read before this thread rewrites it; no other thread touches it)
        float nw[TAPS][V];
#pragma unroll
        for (int t = 0; t < TAPS; ++t) {
            const int pos = n_tokens - TAPS + t;
            if (pos >= 0) {
                load_vec<V>(nw[t], x_ptr + static_cast<size_t>(pos) * conv_dim);
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) nw[t][v] = hs[v * TAPS + pos + TAPS];
            }
        }
#pragma unroll
        for (int t = 0; t < TAPS; ++t)
#pragma unroll
            for (int v = 0; v < V; ++v) hs[v * TAPS + t] = nw[t][v];
    }
}

// q/k split + L2-norm (ssm_gated_delta.cu, fc_ssm_qknorm_gqa_nx, without the GQA
// copies): one CTA per row, one warp per head vector, lane L holding elements
// [E*L, E*L+E); v is copied through.
template <int E>
__global__ void __launch_bounds__(kThreads) qkv_split_norm_kernel(
    const float *__restrict__ conv_out, float *__restrict__ q, float *__restrict__ k,
    float *__restrict__ v, int n_k_heads, int n_v_heads, float eps) {
    constexpr int S = 32 * E;
    const int row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int key_dim = n_k_heads * S;
    const size_t conv_dim = static_cast<size_t>(2 * key_dim + n_v_heads * S);
    const float *src = conv_out + row * conv_dim;
    for (int hv = warp; hv < 2 * n_k_heads; hv += kThreads / 32) {
        float x[E];
        load_vec<E>(x, src + static_cast<size_t>(hv) * S + lane * E);
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = __fmaf_rn(x[e], x[e], ss);
        ss = warp_allsum(ss);
        const float inv = 1.0f / fmaxf(sqrtf(ss), eps);
#pragma unroll
        for (int e = 0; e < E; ++e) x[e] *= inv;
        float *dst = (hv < n_k_heads ? q : k) +
                     (static_cast<size_t>(row) * n_k_heads + (hv % n_k_heads)) * S + lane * E;
        store_vec<E>(dst, x);
    }
    const float4 *vs = reinterpret_cast<const float4 *>(src + 2 * key_dim);
    float4 *vd = reinterpret_cast<float4 *>(v + static_cast<size_t>(row) * n_v_heads * S);
    for (int i = threadIdx.x; i < n_v_heads * S / 4; i += kThreads) vd[i] = vs[i];
}

// Gated RMSNorm, fm_kernel_ssm.m "Gated RMSNorm" and ssm_gated_delta.cu Kernel 3:
// one warp per head row, one shuffle reduction, weight shared across heads.
// Row r is head r % heads of position r / heads. With `slots` or a ragged batch, the
// rows of a sequence whose slot is outside [0, pool) or whose range is not valid,
// and (ragged) rows of positions no sequence owns, are left untouched.
template <int E>
__global__ void __launch_bounds__(kThreads) gated_norm_kernel(const float *y,
                                                               const float *__restrict__ w,
                                                               const float *__restrict__ z,
                                                               float *out, long long rows,
                                                               float eps, int heads, int n_seqs,
                                                               const SeqMap seqs,
                                                               const int32_t *__restrict__ slots,
                                                               int pool) {
    constexpr int D = 32 * E;
    const long long row = blockIdx.x * static_cast<long long>(kThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    // the row's operands first: their latency overlaps the lookup of its sequence
    float yv[E], zv[E], wv[E];
    load_vec<E>(yv, y + row * D + lane * E);
    load_vec<E>(zv, z + row * D + lane * E);
    load_vec<E>(wv, w + lane * E);
    if (slots || seqs.cu) {
        const long long pos = row / heads;
        int n;
        if (seqs.cu) {
            n = warp_seq_of_position(seqs.cu, n_seqs, pos);  // row (and pos) is per warp
            size_t t0;
            int len;
            if (n < 0 || !seqs.range(n, t0, len) || pos >= static_cast<long long>(t0) + len) return;
        } else {
            n = static_cast<int>(pos / seqs.n_tokens);
        }
        if (slots) {
            const int slot = slots[n];
            if (slot < 0 || slot >= pool) return;
        }
    }
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = __fmaf_rn(yv[e], yv[e], ss);
    ss = warp_allsum(ss);
    const float inv_rms = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = yv[e] * inv_rms * wv[e] * silu(zv[e]);
    store_vec<E>(out + row * D + lane * E, o);
}

template <int K>
gdn_status launch_conv(const float *qkv, const float *w, float *conv_state, float *out,
                       int n_seqs, int n_tokens, int conv_dim, const int32_t *slots, int pool,
                       int32_t *err_count, float *snaps, cudaStream_t s) {
    // four channels a thread where the channel rows allow 16-byte accesses
    const bool wide = conv_dim % 4 == 0 && aligned16(qkv) && aligned16(out);
    const int per = wide ? 4 : 1;
    const dim3 grid((conv_dim / per + kThreads - 1) / kThreads, n_seqs,
                    (n_tokens + kConvTokens - 1) / kConvTokens);
    if (wide) {
        if (snaps)
            conv1d_silu_kernel<K, true, 4><<<grid, kThreads, 0, s>>>(
                qkv, w, conv_state, out, n_tokens, conv_dim, slots, pool, err_count, snaps);
        else
            conv1d_silu_kernel<K, false, 4><<<grid, kThreads, 0, s>>>(
                qkv, w, conv_state, out, n_tokens, conv_dim, slots, pool, err_count, nullptr);
    } else {
        if (snaps)
            conv1d_silu_kernel<K, true, 1><<<grid, kThreads, 0, s>>>(
                qkv, w, conv_state, out, n_tokens, conv_dim, slots, pool, err_count, snaps);
        else
            conv1d_silu_kernel<K, false, 1><<<grid, kThreads, 0, s>>>(
                qkv, w, conv_state, out, n_tokens, conv_dim, slots, pool, err_count, nullptr);
    }
    return launch_status();
}

gdn_status conv_common(const float *qkv, const float *w, float *conv_state, float *out,
                       int n_seqs, int n_tokens, int conv_dim, int conv_kernel,
                       const int32_t *slots, int pool, int32_t *err_count, float *snaps,
                       gdn_stream_t stream) {
    if (!qkv || !w || !conv_state || !out) return GDN_ERR_NULL;
    if (n_seqs < 0 || n_tokens < 0 || conv_dim < 1) return GDN_ERR_SHAPE;
    if (conv_kernel < 2 || conv_kernel > 8) return GDN_ERR_SHAPE;
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    if (n_seqs > 65535 || (n_tokens + kConvTokens - 1) / kConvTokens > 65535)
        return GDN_ERR_UNSUPPORTED;
    const cudaStream_t s = as_cuda(stream);
    switch (conv_kernel) {
        case 2: return launch_conv<2>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
        case 3: return launch_conv<3>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
        case 4: return launch_conv<4>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
        case 5: return launch_conv<5>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
        case 6: return launch_conv<6>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
        case 7: return launch_conv<7>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
        default: return launch_conv<8>(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, slots, pool, err_count, snaps, s);
    }
}


// ---------------------------------------------------------------- snapshot restore
// Rollback after a speculative verification: sequence n (grid row n) copies the
// snapshot taken after its accepted[n]-th position into its state slot and, if given,
// its conv slot. The first `state_parts` CTAs of a row copy the state (16-byte
// vectors, kRestoreVec4 per CTA), the rest the conv history (single floats, whose
// count need not be a multiple of 4). A row whose accepted count or slot is out of
// range copies nothing and is counted once.
constexpr int kRestoreVec4 = kThreads * 8;   // float4 per CTA of the state copy (32 KiB)
constexpr int kRestoreConv = kThreads * 16;  // floats per CTA of the conv copy

__global__ void __launch_bounds__(kThreads) snapshot_restore_kernel(
    float *state, const float *__restrict__ snaps, float *conv_state,
    const float *__restrict__ conv_snaps, const int32_t *__restrict__ accepted, const SeqMap seqs,
    size_t state_floats, size_t conv_floats, int state_parts, const int32_t *__restrict__ slots,
    int pool, int32_t *err_count) {
    const int n = blockIdx.y, part = blockIdx.x;
    const int slot = slots ? slots[n] : n;
    const int m = accepted[n];
    size_t t0;  // the snapshot after position t of sequence n is snapshot t0 + t
    int len;
    if (slot < 0 || slot >= pool || !seqs.range(n, t0, len) || m < 1 || m > len) {
        // uniform over the row
        if (err_count && part == 0 && threadIdx.x == 0) atomicAdd(err_count, 1);
        return;
    }
    const size_t snap = t0 + (m - 1);  // snapshot index
    if (part < state_parts) {
        // all 8 loads of a thread in flight before its stores
        const float4 *src = reinterpret_cast<const float4 *>(snaps + snap * state_floats);
        float4 *dst = reinterpret_cast<float4 *>(state + static_cast<size_t>(slot) * state_floats);
        const size_t n4 = state_floats / 4, i0 = static_cast<size_t>(part) * kRestoreVec4 + threadIdx.x;
        float4 v[kRestoreVec4 / kThreads];
#pragma unroll
        for (int j = 0; j < kRestoreVec4 / kThreads; ++j)
            if (i0 + j * kThreads < n4) v[j] = src[i0 + j * kThreads];
#pragma unroll
        for (int j = 0; j < kRestoreVec4 / kThreads; ++j)
            if (i0 + j * kThreads < n4) dst[i0 + j * kThreads] = v[j];
    } else {
        const float *src = conv_snaps + snap * conv_floats;
        float *dst = conv_state + static_cast<size_t>(slot) * conv_floats;
        const size_t end = min(conv_floats, static_cast<size_t>(part - state_parts + 1) * kRestoreConv);
#pragma unroll 4
        for (size_t i = static_cast<size_t>(part - state_parts) * kRestoreConv + threadIdx.x; i < end;
             i += kThreads)
            dst[i] = src[i];
    }
}

}  // namespace

gdn_status launch_gated_norm_seqs(const float *y, const float *w, const float *z, float *out,
                                  long long rows, int head_dim, float eps, int heads, int n_seqs,
                                  SeqMap seqs, const int32_t *slots, int pool, cudaStream_t s) {
    if (rows == 0) return GDN_OK;
    const unsigned blocks = static_cast<unsigned>((rows + kThreads / 32 - 1) / (kThreads / 32));
    switch (head_dim) {
        case 32: gated_norm_kernel<1><<<blocks, kThreads, 0, s>>>(y, w, z, out, rows, eps, heads, n_seqs, seqs, slots, pool); break;
        case 64: gated_norm_kernel<2><<<blocks, kThreads, 0, s>>>(y, w, z, out, rows, eps, heads, n_seqs, seqs, slots, pool); break;
        case 128: gated_norm_kernel<4><<<blocks, kThreads, 0, s>>>(y, w, z, out, rows, eps, heads, n_seqs, seqs, slots, pool); break;
        default: gated_norm_kernel<8><<<blocks, kThreads, 0, s>>>(y, w, z, out, rows, eps, heads, n_seqs, seqs, slots, pool); break;
    }
    return launch_status();
}

}  // namespace gdn

using namespace gdn;

extern "C" {

const char *gdn_status_str(gdn_status status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_NULL: return "GDN_ERR_NULL";
        case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN";
        case GDN_ERR_LAUNCH: return "GDN_ERR_LAUNCH";
        case GDN_ERR_DEVICE: return "GDN_ERR_DEVICE";
    }
    return "GDN_ERR_UNKNOWN";
}

int gdn_version(void) { return (1 << 16) | 0; }

gdn_status gdn_device_error(gdn_stream_t stream) {
    const cudaStream_t s = as_cuda(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_LAUNCH;
    unsigned flags = read_and_clear_watchdog_recurrence(s) | read_and_clear_watchdog_block(s) |
                     read_and_clear_watchdog_chunked(s) | read_and_clear_watchdog_chunked_ws(s);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_LAUNCH;
    return flags ? GDN_ERR_DEVICE : GDN_OK;
}

gdn_status gdn_selftest_bounded_wait(unsigned arm_mask, unsigned limit_us, float *out,
                                     gdn_stream_t stream) {
    if (!out) return GDN_ERR_NULL;
    if (arm_mask > 15u || limit_us < 1 || limit_us > 2000000u) return GDN_ERR_SHAPE;
    const cudaStream_t s = as_cuda(stream);
    const uint64_t ns = 1000ull * limit_us;
    GDN_TRY(launch_wait_probe_recurrence(arm_mask & 1u, ns, out + 0, s));
    GDN_TRY(launch_wait_probe_block(arm_mask & 2u, ns, out + 1, s));
    GDN_TRY(launch_wait_probe_chunked(arm_mask & 4u, ns, out + 2, s));
    return launch_wait_probe_chunked_ws(arm_mask & 8u, ns, out + 3, s);
}

gdn_status gdn_decay_gate(const float *alpha, const float *dt, const float *a, float *g,
                          int n_heads, int rows, gdn_stream_t stream) {
    if (!alpha || !dt || !a || !g) return GDN_ERR_NULL;
    if (n_heads < 1 || rows < 0) return GDN_ERR_SHAPE;
    if (rows == 0) return GDN_OK;
    const long long total = static_cast<long long>(rows) * n_heads;
    const unsigned blocks = static_cast<unsigned>((total + kThreads - 1) / kThreads);
    decay_gate_kernel<<<blocks, kThreads, 0, as_cuda(stream)>>>(alpha, dt, a, g, n_heads, total);
    return launch_status();
}

gdn_status gdn_beta_sigmoid(const float *b, float *beta, int n, gdn_stream_t stream) {
    if (!b || !beta) return GDN_ERR_NULL;
    if (n < 0) return GDN_ERR_SHAPE;
    if (n == 0) return GDN_OK;
    sigmoid_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, as_cuda(stream)>>>(b, beta, n);
    return launch_status();
}

gdn_status gdn_conv1d_silu(const float *qkv, const float *w, float *conv_state, float *out,
                           int n_seqs, int conv_dim, int conv_kernel, const int32_t *slots,
                           int pool, int32_t *err_count, gdn_stream_t stream) {
    return conv_common(qkv, w, conv_state, out, n_seqs, 1, conv_dim, conv_kernel, slots, pool,
                       err_count, nullptr, stream);
}

gdn_status gdn_conv1d_silu_seq(const float *qkv, const float *w, float *conv_state, float *out,
                               int n_seqs, int n_tokens, int conv_dim, int conv_kernel,
                               const int32_t *slots, int pool, int32_t *err_count,
                               gdn_stream_t stream) {
    return conv_common(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, conv_kernel, slots,
                       pool, err_count, nullptr, stream);
}

gdn_status gdn_conv1d_silu_seq_snapshots(const float *qkv, const float *w, float *conv_state,
                                         float *out, float *snaps, int n_seqs, int n_tokens,
                                         int conv_dim, int conv_kernel, const int32_t *slots,
                                         int pool, int32_t *err_count, gdn_stream_t stream) {
    if (!snaps) return GDN_ERR_NULL;
    return conv_common(qkv, w, conv_state, out, n_seqs, n_tokens, conv_dim, conv_kernel, slots,
                       pool, err_count, snaps, stream);
}

}  // extern "C"

namespace {

gdn_status restore_impl(float *state, const float *snaps, float *conv_state,
                        const float *conv_snaps, const int32_t *accepted, int n_seqs, SeqMap seqs,
                        int n_v_heads, int state_size, int conv_dim, int conv_kernel,
                        const int32_t *slots, int pool, int32_t *err_count, gdn_stream_t stream) {
    if (!state || !snaps || !accepted) return GDN_ERR_NULL;
    const bool conv = conv_state || conv_snaps;
    if (conv && !(conv_state && conv_snaps)) return GDN_ERR_NULL;
    if (n_seqs < 0 || n_v_heads < 1) return GDN_ERR_SHAPE;
    if (seqs.cu == nullptr ? seqs.n_tokens < 1 : (seqs.n_tokens < 0 || seqs.total < 0))
        return GDN_ERR_SHAPE;
    if (state_size < 32 || state_size % 32 != 0 || state_size > 256) return GDN_ERR_SHAPE;
    if (!supported_state_size(state_size)) return GDN_ERR_UNSUPPORTED;  // as the snapshot scan
    if (conv && (conv_dim < 1 || conv_kernel < 2 || conv_kernel > 8)) return GDN_ERR_SHAPE;
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(state) || !aligned16(snaps)) return GDN_ERR_ALIGN;
    if (n_seqs == 0) return GDN_OK;
    if (n_seqs > 65535) return GDN_ERR_UNSUPPORTED;
    const size_t state_floats = static_cast<size_t>(n_v_heads) * state_size * state_size;
    const size_t conv_floats = conv ? static_cast<size_t>(conv_dim) * (conv_kernel - 1) : 0;
    const long long state_parts = static_cast<long long>((state_floats / 4 + kRestoreVec4 - 1) / kRestoreVec4);
    const long long conv_parts = static_cast<long long>((conv_floats + kRestoreConv - 1) / kRestoreConv);
    if (state_parts + conv_parts > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(state_parts + conv_parts), static_cast<unsigned>(n_seqs));
    snapshot_restore_kernel<<<grid, kThreads, 0, as_cuda(stream)>>>(
        state, snaps, conv_state, conv_snaps, accepted, seqs, state_floats, conv_floats,
        static_cast<int>(state_parts), slots, pool, err_count);
    return launch_status();
}

}  // namespace

extern "C" {

gdn_status gdn_snapshot_restore(float *state, const float *snaps, float *conv_state,
                                const float *conv_snaps, const int32_t *accepted, int n_seqs,
                                int n_tokens, int n_v_heads, int state_size, int conv_dim,
                                int conv_kernel, const int32_t *slots, int pool,
                                int32_t *err_count, gdn_stream_t stream) {
    return restore_impl(state, snaps, conv_state, conv_snaps, accepted, n_seqs,
                        uniform_seqs(n_seqs, n_tokens), n_v_heads, state_size, conv_dim,
                        conv_kernel, slots, pool, err_count, stream);
}

gdn_status gdn_snapshot_restore_varlen(float *state, const float *snaps, float *conv_state,
                                       const float *conv_snaps, const int32_t *accepted,
                                       const int32_t *cu_seqlens, int n_seqs, int total_tokens,
                                       int max_tokens, int n_v_heads, int state_size,
                                       int conv_dim, int conv_kernel, const int32_t *slots,
                                       int pool, int32_t *err_count, gdn_stream_t stream) {
    GDN_TRY(check_varlen(cu_seqlens, n_seqs, total_tokens, max_tokens));
    return restore_impl(state, snaps, conv_state, conv_snaps, accepted, n_seqs,
                        SeqMap{cu_seqlens, max_tokens, total_tokens}, n_v_heads, state_size,
                        conv_dim, conv_kernel, slots, pool, err_count, stream);
}

gdn_status gdn_qkv_split_norm(const float *conv_out, float *q, float *k, float *v, int rows,
                              int n_k_heads, int n_v_heads, int state_size, float eps,
                              gdn_stream_t stream) {
    if (!conv_out || !q || !k || !v) return GDN_ERR_NULL;
    if (rows < 0) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    if (!aligned16(conv_out) || !aligned16(q) || !aligned16(k) || !aligned16(v)) return GDN_ERR_ALIGN;
    if (rows == 0) return GDN_OK;
    const cudaStream_t s = as_cuda(stream);
    switch (state_size) {
        case 32: qkv_split_norm_kernel<1><<<rows, kThreads, 0, s>>>(conv_out, q, k, v, n_k_heads, n_v_heads, eps); break;
        case 64: qkv_split_norm_kernel<2><<<rows, kThreads, 0, s>>>(conv_out, q, k, v, n_k_heads, n_v_heads, eps); break;
        case 128: qkv_split_norm_kernel<4><<<rows, kThreads, 0, s>>>(conv_out, q, k, v, n_k_heads, n_v_heads, eps); break;
        default: qkv_split_norm_kernel<8><<<rows, kThreads, 0, s>>>(conv_out, q, k, v, n_k_heads, n_v_heads, eps); break;
    }
    return launch_status();
}

gdn_status gdn_gated_norm(const float *y, const float *w, const float *z, float *out, int rows,
                          int head_dim, float eps, gdn_stream_t stream) {
    if (!y || !w || !z || !out) return GDN_ERR_NULL;
    if (rows < 0 || head_dim < 1) return GDN_ERR_SHAPE;
    if (!supported_state_size(head_dim)) {
        return (head_dim % 32 == 0 && head_dim <= 256) ? GDN_ERR_UNSUPPORTED : GDN_ERR_SHAPE;
    }
    if (!aligned16(y) || !aligned16(w) || !aligned16(z) || !aligned16(out)) return GDN_ERR_ALIGN;
    return launch_gated_norm_seqs(y, w, z, out, rows, head_dim, eps, 1, rows,
                                  uniform_seqs(rows, 1), nullptr, 0, as_cuda(stream));
}

}  // extern "C"
