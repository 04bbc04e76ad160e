// gdn_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {

inline cudaStream_t as_cuda(gdn_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool supported_state_size(int s) { return s == 32 || s == 64 || s == 128 || s == 256; }

// Status of the most recent launch on this thread.
inline gdn_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

// Checks common to the entry points that take a state pool.
inline gdn_status check_pool(int n_seqs, const int32_t *slots, int pool) {
    if (pool < 1) return GDN_ERR_SHAPE;
    if (slots == nullptr && pool < n_seqs) return GDN_ERR_SHAPE;
    return GDN_OK;
}

inline gdn_status check_heads(int n_k_heads, int n_v_heads, int state_size) {
    if (n_k_heads < 1 || n_v_heads < 1 || n_v_heads % n_k_heads != 0) return GDN_ERR_SHAPE;
    if (state_size < 32 || state_size % 32 != 0 || state_size > 256) return GDN_ERR_SHAPE;
    if (!supported_state_size(state_size)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Gated RMSNorm over `rows` rows of head_dim; with `slots` non-NULL the rows of
// sequence r / rows_per_seq are skipped when its slot is outside [0, pool).
gdn_status launch_gated_norm(const float *y, const float *w, const float *z, float *out,
                             long long rows, int head_dim, float eps, long long rows_per_seq,
                             const int32_t *slots, int pool, cudaStream_t s);

// Per-translation-unit watchdog flags (a bounded wait that gave up sets a bit).
unsigned read_and_clear_watchdog_recurrence(cudaStream_t s);
unsigned read_and_clear_watchdog_block(cudaStream_t s);
unsigned read_and_clear_watchdog_chunked(cudaStream_t s);
unsigned read_and_clear_watchdog_chunked_ws(cudaStream_t s);

}  // namespace gdn

#define GDN_TRY(expr)                              \
    do {                                           \
        const gdn_status gdn_st_ = (expr);         \
        if (gdn_st_ != GDN_OK) return gdn_st_;     \
    } while (0)
