// gdn_prefill.cu -- the block over n_tokens positions per sequence (prefill): the
// conv scan, the q/k split + L2-norm, the decay gate, beta, the sequential scan of
// the recurrence and the gated RMSNorm, chained on one stream. Intermediates live
// in a workspace the caller provides (the library allocates nothing); the scan
// writes y straight into `out`, which the gated norm then rewrites in place.
//
// Follows the batched (prefill) variants of ssm_gated_delta.cu: decay gate, conv
// scan, q/k norm with the v passthrough, then the recurrence scan, per position.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr size_t kAlignFloats = 64;  // 256-byte sub-buffers

size_t round_up(size_t n) { return (n + kAlignFloats - 1) / kAlignFloats * kAlignFloats; }

struct PrefillLayout {
    size_t conv_out, q, k, v, g, beta, total_floats;
    PrefillLayout(long long n, long long t, int hk, int h, int s) {
        const size_t rows = static_cast<size_t>(n) * static_cast<size_t>(t);
        const size_t conv_dim = static_cast<size_t>(2 * hk + h) * s;
        conv_out = 0;
        q = conv_out + round_up(rows * conv_dim);
        k = q + round_up(rows * hk * s);
        v = k + round_up(rows * hk * s);
        g = v + round_up(rows * h * s);
        beta = g + round_up(rows * h);
        total_floats = beta + round_up(rows * h);
    }
};

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t gdn_block_prefill_workspace_size(int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                                        int state_size) {
    if (n_seqs < 0 || n_tokens < 0 || n_k_heads < 1 || n_v_heads < 1 || state_size < 1) return 0;
    return PrefillLayout(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size).total_floats *
           sizeof(float);
}

}  // extern "C"

namespace {

// The prefill block with either scan: the sequential one (bit for bit the fused
// decode step, position after position) or the chunked tensor-core one.
gdn_status prefill_impl(const float *qkv, const float *conv_w, float *conv_state,
                        const float *alpha, const float *b, const float *dt, const float *a,
                        const float *z, const float *norm_w, float *state, float *out,
                        int n_seqs, int n_tokens, int n_k_heads, int n_v_heads, int state_size,
                        int conv_kernel, float scale, float l2_eps, float norm_eps,
                        const int32_t *slots, int pool, int32_t *err_count, void *workspace,
                        size_t workspace_bytes, gdn_stream_t stream, bool chunked) {
    if (!qkv || !conv_w || !conv_state || !alpha || !b || !dt || !a || !z || !norm_w || !state ||
        !out)
        return GDN_ERR_NULL;
    if (n_seqs < 0 || n_tokens < 0) return GDN_ERR_SHAPE;
    if (conv_kernel < 2 || conv_kernel > 8) return GDN_ERR_SHAPE;
    GDN_TRY(check_heads(n_k_heads, n_v_heads, state_size));
    if (chunked && state_size != 128) return GDN_ERR_UNSUPPORTED;
    GDN_TRY(check_pool(n_seqs, slots, pool));
    if (!aligned16(qkv) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(state) ||
        !aligned16(z) || !aligned16(out) || !aligned16(norm_w))
        return GDN_ERR_ALIGN;
    if (n_seqs == 0 || n_tokens == 0) return GDN_OK;
    const PrefillLayout L(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size);
    if (!workspace) return GDN_ERR_NULL;
    if (workspace_bytes < L.total_floats * sizeof(float)) return GDN_ERR_SHAPE;
    if (!aligned16(workspace)) return GDN_ERR_ALIGN;
    const long long rows = static_cast<long long>(n_seqs) * n_tokens;
    if (rows * n_v_heads > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const int S = state_size, H = n_v_heads, Hk = n_k_heads;
    const int conv_dim = (2 * Hk + H) * S;
    float *ws = static_cast<float *>(workspace);
    float *conv_out = ws + L.conv_out, *q = ws + L.q, *k = ws + L.k, *v = ws + L.v;
    float *g = ws + L.g, *beta = ws + L.beta;

    // A skipped sequence is counted once, by the conv scan; nothing of it is written
    // to conv_state, state or out.
    GDN_TRY(gdn_conv1d_silu_seq(qkv, conv_w, conv_state, conv_out, n_seqs, n_tokens, conv_dim,
                                conv_kernel, slots, pool, err_count, stream));
    GDN_TRY(gdn_qkv_split_norm(conv_out, q, k, v, static_cast<int>(rows), Hk, H, S, l2_eps,
                               stream));
    GDN_TRY(gdn_decay_gate(alpha, dt, a, g, H, static_cast<int>(rows), stream));
    GDN_TRY(gdn_beta_sigmoid(b, beta, static_cast<int>(rows * H), stream));
    if (chunked) {
        GDN_TRY(gdn_recurrence_scan_chunked(state, q, k, v, g, beta, out, n_seqs, n_tokens, Hk, H,
                                            S, scale, slots, pool, nullptr, stream));
    } else {
        GDN_TRY(gdn_recurrence_scan(state, q, k, v, g, beta, out, n_seqs, n_tokens, Hk, H, S,
                                    scale, slots, pool, nullptr, stream));
    }
    return launch_gated_norm(out, norm_w, z, out, rows * H, S, norm_eps,
                             static_cast<long long>(n_tokens) * H, slots, pool, as_cuda(stream));
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
                        n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps,
                        norm_eps, slots, pool, err_count, workspace, workspace_bytes, stream, false);
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
                        n_tokens, n_k_heads, n_v_heads, state_size, conv_kernel, scale, l2_eps,
                        norm_eps, slots, pool, err_count, workspace, workspace_bytes, stream, true);
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
    const size_t need =
        PrefillLayout(n_seqs, n_tokens, n_k_heads, n_v_heads, state_size).total_floats *
        sizeof(float);
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
