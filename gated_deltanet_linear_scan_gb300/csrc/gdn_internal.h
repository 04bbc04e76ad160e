// gdn_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {

inline cudaStream_t as_cuda(gdn_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Where each sequence's positions lie in the token-major arrays of a call.
// Uniform batch (cu == NULL): every sequence has n_tokens positions, sequence n's
// starting at n * n_tokens. Ragged batch: sequence n owns the packed positions
// cu[n] .. cu[n+1] - 1 of `total`, and n_tokens bounds the length of any one
// sequence (it sizes the grids). A ragged range that is not valid (negative, reversed,
// past `total` or longer than n_tokens) makes its sequence be skipped, as an
// out-of-range slot does.
struct SeqMap {
    const int32_t *cu;
    int n_tokens;
    long long total;

    __device__ __forceinline__ bool range(int n, size_t &t0, int &len) const {
        if (cu == nullptr) {
            t0 = static_cast<size_t>(n) * n_tokens;
            len = n_tokens;
            return true;
        }
        const int a = cu[n], b = cu[n + 1];
        if (a < 0 || b < a || b > total || b - a > n_tokens) return false;
        t0 = static_cast<size_t>(a);
        len = b - a;
        return true;
    }
};

inline SeqMap uniform_seqs(int n_seqs, int n_tokens) {
    return SeqMap{nullptr, n_tokens, static_cast<long long>(n_seqs) * n_tokens};
}

// The last index n in [0, count) with key(n) <= target, or -1 if none, for a key that is
// non-decreasing in n (with any other key the answer is still some index in [-1, count),
// which callers validate). Found by a whole warp, every lane returning it: each pass the
// lanes probe 32 evenly spaced keys of the remaining range, so up to 32 keys take one
// round of loads, 1024 two.
template <typename Key>
__device__ __forceinline__ int warp_last_le(int count, long long target, Key key) {
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = count;  // the answer is the last n in [lo, hi) with key(n) <= target, or lo - 1
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const unsigned hit = __ballot_sync(0xffffffffu, idx < hi && key(idx) <= target);
        if (hit == 0) return lo - 1;
        const int last = 31 - __clz(hit);
        lo += last * step;
        hi = min(hi, lo + step);
    }
    const int idx = lo + lane;
    const unsigned hit = __ballot_sync(0xffffffffu, idx < hi && key(idx) <= target);
    return hit == 0 ? lo - 1 : lo + 31 - __clz(hit);
}

// The sequence of a ragged batch that owns packed position pos (with valid offsets), or
// -1: the last n with cu[n] <= pos. Called by a whole warp.
__device__ __forceinline__ int warp_seq_of_position(const int32_t *cu, int n_seqs, long long pos) {
    return warp_last_le(n_seqs, pos, [&](int n) { return static_cast<long long>(cu[n]); });
}

// The sequence whose block slots contain `slot`, when block b of sequence n takes slot
// cu[n] / per_block + n + b (the slots of consecutive sequences never collide): the last n
// with cu[n] / per_block + n <= slot, or -1. Called by a whole warp.
__device__ __forceinline__ int warp_seq_of_slot(const int32_t *cu, int n_seqs, int per_block,
                                                long long slot) {
    return warp_last_le(n_seqs, slot, [&](int n) {
        return static_cast<long long>(cu[n]) / per_block + n;
    });
}

// Longest-first order of a ragged batch for CTA scheduling: the sequence whose valid
// length is the rank-th largest (ties by index; invalid ranges count as length 0), found
// by the whole CTA (every thread returns it; uses one int of shared memory and two
// __syncthreads). O(n_seqs^2 / threads) work, so callers use it for small batches only.
__device__ __forceinline__ int seq_by_length_rank(const SeqMap &seqs, int n_seqs, int rank,
                                                  int *shared_slot) {
    auto len_of = [&](int m) {
        size_t t0;
        int len;
        return seqs.range(m, t0, len) ? len : 0;
    };
    if (threadIdx.x == 0) *shared_slot = rank;  // stays if no thread matches (cannot happen)
    __syncthreads();
    for (int m = threadIdx.x; m < n_seqs; m += blockDim.x) {
        const int lm = len_of(m);
        int above = 0;
        for (int j = 0; j < n_seqs; ++j) {
            const int lj = len_of(j);
            above += (lj > lm) || (lj == lm && j < m);
        }
        if (above == rank) *shared_slot = m;
    }
    __syncthreads();
    return *shared_slot;
}

// Ragged batches up to this many sequences run their per-sequence CTAs longest first.
constexpr int kLongestFirstMaxSeqs = 256;

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

// Gated RMSNorm over `rows` rows of head_dim, row r being head r % heads of position
// r / heads of the positions `seqs` maps. With `slots` non-NULL, or a ragged batch, the
// rows of a skipped sequence (slot outside [0, pool), range not valid) and of positions
// no sequence owns are left untouched.
gdn_status launch_gated_norm_seqs(const float *y, const float *w, const float *z, float *out,
                                  long long rows, int head_dim, float eps, int heads, int n_seqs,
                                  SeqMap seqs, const int32_t *slots, int pool, cudaStream_t s);

// Checks of a ragged batch's host arguments (cu_seqlens itself is device memory).
gdn_status check_varlen(const int32_t *cu_seqlens, int n_seqs, int total_tokens, int max_tokens);

// The sequential scan (snaps non-NULL: its snapshot form) over the positions `seqs` maps.
gdn_status launch_scan_seqs(float *state, const float *q, const float *k, const float *v,
                            const float *g, const float *beta, float *y, int n_seqs, SeqMap seqs,
                            int n_k_heads, int n_v_heads, int state_size, float scale,
                            const int32_t *slots, int pool, int32_t *err_count, float *snaps,
                            cudaStream_t s);

// The chunked scan over the positions `seqs` maps: the two-phase form in `workspace`
// if it holds every chunk of the call (chunked_seqs_ws_size bytes), else the
// one-kernel form.
size_t chunked_seqs_ws_size(int n_seqs, SeqMap seqs, int n_v_heads);
size_t ragged_chunked_ws_size(int n_seqs, long long total, int n_v_heads);
gdn_status launch_chunked_seqs(float *state, const float *q, const float *k, const float *v,
                               const float *g, const float *beta, float *y, int n_seqs,
                               SeqMap seqs, int n_k_heads, int n_v_heads, float scale,
                               const int32_t *slots, int pool, int32_t *err_count,
                               void *workspace, size_t workspace_bytes, cudaStream_t s);
gdn_status launch_chunked_one_kernel(float *state, const float *q, const float *k,
                                     const float *v, const float *g, const float *beta, float *y,
                                     int n_seqs, SeqMap seqs, int n_k_heads, int n_v_heads,
                                     float scale, const int32_t *slots, int pool,
                                     int32_t *err_count, cudaStream_t s);

// Bounded-wait self-test kernels, one per translation unit with a watchdog flag.
gdn_status launch_wait_probe_recurrence(bool arm, uint64_t limit_ns, float *out, cudaStream_t s);
gdn_status launch_wait_probe_block(bool arm, uint64_t limit_ns, float *out, cudaStream_t s);
gdn_status launch_wait_probe_chunked(bool arm, uint64_t limit_ns, float *out, cudaStream_t s);
gdn_status launch_wait_probe_chunked_ws(bool arm, uint64_t limit_ns, float *out, cudaStream_t s);

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
