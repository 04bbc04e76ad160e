/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta-rule SSM library.
 *
 * The Gated-DeltaNet SSM block of a hybrid LLM, per (sequence, v-head h):
 *   decay gate      g = a[h] * softplus(alpha + dt[h])
 *   conv1d + SiLU   causal depthwise, kernel K, rolling conv_state
 *   q/k L2-norm     x / max(||x||, eps), then GQA: v-head vh reads k-head vh % Hk
 *   recurrence      S <- exp(g) S; pred = S k; delta = (v - pred) beta;
 *                   S <- S + k delta^T; y = scale S^T q  (read after the write)
 *   gated RMSNorm   out = y / sqrt(mean(y^2) + eps) * w * silu(z)
 * silu(x) = x / (1 + exp(-x)) is evaluated with CUDA's fast exponential and division
 * (within 1e-5 relative for |x| <= 20; a signed zero below about -88). The decay,
 * softplus and the sigmoid of beta use the precise expf.
 * Sources: "fm_kernel_ssm.m" (Foundry: Metal host dispatch + shader source),
 * "ssm_gated_delta.cu" (Foundry: CUDA kernels), "gated_delta_net_decode.metal"
 * (mlx-native 0.21.1). Each entry point below names the section it follows.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All array arguments are DEVICE pointers to fp32 (int32 for slot ids),
 *   allocated and owned by the caller. The library allocates and frees nothing.
 * - Every call is asynchronous on `stream` (NULL = legacy default stream). A
 *   return of GDN_OK means the work was validated and enqueued.
 * - Arguments are validated on the host before anything is enqueued; on any
 *   error nothing is enqueued and no memory is touched. (The pages' launchers
 *   return silently on bad arguments; here the failure is a status code.)
 * - Pointers used with 128-bit or bulk (TMA) copies must be 16-byte aligned;
 *   a misaligned one gives GDN_ERR_ALIGN. Buffers from cudaMalloc are.
 * - Shapes: n_v_heads % n_k_heads == 0; state_size (= D_k = D_v = S) in
 *   {32, 64, 128, 256}; conv_kernel K in [2, 8] (the fused block: K = 4).
 *   n_seqs == 0 or n_tokens == 0 is a valid no-op.
 * - Layouts (row-major, innermost last):
 *     state       [pool][H][S][S]  state[((slot*H + h)*S + j)*S + i] == S_h[i][j]
 *                                  (transposed: row j, a v-index, is contiguous over i)
 *     conv_state  [pool][C][K-1]   oldest tap first, holding RAW (pre-conv) inputs
 *     conv_w      [C][K]           conv_w[c][K-1] multiplies the current input
 *     qkv         [N][T][C]        C = 2*Hk*S + H*S packed as [q | k | v]
 *     q, k        [N][T][Hk][S]    k-head space (post-L2-norm for the recurrence)
 *     v, y, z     [N][T][H][S]
 *     g, beta     [N][T][H]        g is the log-decay (<= 0), beta in (0, 1)
 * - Serving pool: sequence n uses state (and conv_state) slot slots[n], or n
 *   when `slots` is NULL. `pool` is the number of slots the buffers hold. Slot
 *   ids within one call must be distinct (duplicates race: undefined result).
 *   A sequence whose id lies outside [0, pool) is skipped -- nothing of it is
 *   read or written -- and, if `err_count` (device int32) is non-NULL, 1 is
 *   added to *err_count per skipped sequence. Untouched slots keep their bits.
 * - Kernels that wait on their own asynchronous copies bound every wait (about
 *   two seconds). A wait that gives up skips the work it guarded and raises a
 *   device-side flag; gdn_device_error() reads and clears it.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; spelled here so the header needs no CUDA include. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL */
    GDN_ERR_SHAPE = 2,       /* a dimension is negative/zero where it may not be, or inconsistent */
    GDN_ERR_UNSUPPORTED = 3, /* valid for the method, but no kernel is built for it */
    GDN_ERR_ALIGN = 4,       /* a pointer that needs 16-byte alignment is not aligned */
    GDN_ERR_LAUNCH = 5,      /* the CUDA launch itself failed (see cudaGetLastError) */
    GDN_ERR_DEVICE = 6       /* a kernel's bounded wait gave up (from gdn_device_error) */
} gdn_status;

/* Name of a status code ("GDN_OK", ...); never NULL. */
const char *gdn_status_str(gdn_status status);

/* ABI version of this library, (major << 16) | minor. */
int gdn_version(void);

/* Synchronises `stream`, then reads and clears the device-side flag raised by
 * bounded waits that gave up. GDN_OK if none did, GDN_ERR_DEVICE otherwise, or
 * GDN_ERR_LAUNCH if the synchronisation itself reported a CUDA error.
 * The flag belongs to the library on the current device, not to a stream: it
 * reports, and clears, give-ups of this library's kernels launched on any stream
 * of the current device since the last call. Synchronise the other streams first
 * if their kernels must be covered. */
gdn_status gdn_device_error(gdn_stream_t stream);

/* Self-test of the failure path above, for a caller's health check or a test suite.
 * Enqueues four one-thread kernels, one on each watchdog flag gdn_device_error() reads;
 * probe i (bit i of arm_mask set) waits, bounded by limit_us microseconds, for bytes
 * that no copy will bring -- the wait runs out, the probe raises its flag and skips its
 * guarded write, as a kernel whose copy never lands does. A probe whose bit is clear
 * waits for a phase that completes at once and writes 1.0f to out[i]. So after the
 * call gdn_device_error() returns GDN_ERR_DEVICE if arm_mask != 0 (then GDN_OK on the
 * next call), out[i] keeps its contents for armed probes, and the context stays usable.
 * Nothing faults, traps or waits without bound. The pages have no counterpart: their
 * launchers return silently and their kernels have no bounded waits.
 * out: device float[4]; arm_mask in [0, 15]; limit_us in [1, 2000000]. */
gdn_status gdn_selftest_bounded_wait(unsigned arm_mask, unsigned limit_us, float *out,
                                     gdn_stream_t stream);

/* Decay gate. fm_kernel_ssm.m, decay-gate section; ssm_gated_delta.cu, glue kernels
 * (fc_ssm_decay_gate, _nx). Per row r and head h the log-decay is a[h] times the
 * softplus of alpha[r][h] + dt[h], softplus taken as the identity above 20:
 *   g[r][h] = a[h] * softplus(alpha[r][h] + dt[h]),  softplus(v) = v > 20 ? v : log1p(exp(v))
 * alpha, g: [rows][n_heads]; dt, a: [n_heads] (a = -exp(A_log), baked by the caller).
 * g may alias alpha. rows == 0 is a no-op. */
gdn_status gdn_decay_gate(const float *alpha, const float *dt, const float *a, float *g,
                          int n_heads, int rows, gdn_stream_t stream);

/* beta = 1 / (1 + exp(-b)) over n elements. ssm_gated_delta.cu, glue kernels
 * (fc_sigmoid). beta may alias b. */
gdn_status gdn_beta_sigmoid(const float *b, float *beta, int n, gdn_stream_t stream);

/* Causal depthwise conv1d + SiLU, one token per sequence. fm_kernel_ssm.m, "Causal
 * depthwise conv1d + SiLU"; ssm_gated_delta.cu, Kernel 2 and the slot variant.
 *   pre = qkv[c] * w[c][K-1] + sum_{t<K-1} hist[c][t] * w[c][t];  out[c] = silu(pre)
 * then hist[c] drops its oldest tap and appends the raw qkv[c].
 * qkv, out: [n_seqs][conv_dim]; w: [conv_dim][K]; conv_state: [pool][conv_dim][K-1]
 * (in place). out must not alias qkv. */
gdn_status gdn_conv1d_silu(const float *qkv, const float *w, float *conv_state, float *out,
                           int n_seqs, int conv_dim, int conv_kernel, const int32_t *slots,
                           int pool, int32_t *err_count, gdn_stream_t stream);

/* The same over n_tokens positions per sequence, history carried in registers;
 * bit-identical to n_tokens single-token calls. fm_kernel_ssm.m, the conv scan
 * (fmssm_conv1d_silu_seq); ssm_gated_delta.cu, "BATCHED (prefill) variants".
 * qkv, out: [n_seqs][n_tokens][conv_dim]. */
gdn_status gdn_conv1d_silu_seq(const float *qkv, const float *w, float *conv_state, float *out,
                               int n_seqs, int n_tokens, int conv_dim, int conv_kernel,
                               const int32_t *slots, int pool, int32_t *err_count,
                               gdn_stream_t stream);

/* Split a conv output row [q | k | v] and L2-normalise q and k per k-head.
 * ssm_gated_delta.cu, glue kernels (fc_ssm_qknorm_gqa_nx): each head vector is divided
 * by the larger of its Euclidean norm and eps; v is copied unchanged. No GQA copy is
 * made: the recurrence maps v-head vh to
 * k-head vh % n_k_heads itself.
 * conv_out: [rows][C]; q, k: [rows][Hk][S]; v: [rows][H][S]. No aliasing. */
gdn_status gdn_qkv_split_norm(const float *conv_out, float *q, float *k, float *v, int rows,
                              int n_k_heads, int n_v_heads, int state_size, float eps,
                              gdn_stream_t stream);

/* Delta-rule recurrence, one token per sequence (decode). fm_kernel_ssm.m,
 * "Delta-rule recurrence -- register-resident"; ssm_gated_delta.cu, Kernel 1 and
 * the slot variant; gated_delta_net_decode.metal, "Mathematical recurrence".
 * state: [pool][H][S][S], updated in place (16-byte aligned); q, k: [n_seqs][Hk][S]
 * (post-norm, 16-byte aligned); v, y: [n_seqs][H][S]; g, beta: [n_seqs][H].
 * scale multiplies the readout: 1/sqrt(S), or 1.0f when q is pre-scaled.
 * Consecutive calls visit the state tiles in alternating directions, so a step starts
 * on the state the previous step wrote last, still in L2; the results do not depend on
 * it (a CUDA graph records the direction of the call it captures). */
gdn_status gdn_recurrence_decode(float *state, const float *q, const float *k, const float *v,
                                 const float *g, const float *beta, float *y, int n_seqs,
                                 int n_k_heads, int n_v_heads, int state_size, float scale,
                                 const int32_t *slots, int pool, int32_t *err_count,
                                 gdn_stream_t stream);

/* Decode with the readout factorised. ssm_gated_delta.cu, "T4: 3-pass -> 2-pass
 * state-access factorization" (fc_ssm_recurrence_slots_2pass): with r the decayed
 * row, y = scale * (r . q + delta * (k . q)), so the readout no longer waits for the
 * rank-1 write. Same arguments and layouts as gdn_recurrence_decode; the state is
 * updated bit for bit as there, y agrees with it up to rounding. */
gdn_status gdn_recurrence_decode_2pass(float *state, const float *q, const float *k,
                                       const float *v, const float *g, const float *beta,
                                       float *y, int n_seqs, int n_k_heads, int n_v_heads,
                                       int state_size, float scale, const int32_t *slots,
                                       int pool, int32_t *err_count, gdn_stream_t stream);

/* Sequential scan over n_tokens positions per sequence, the state kept in
 * registers and written back once. fm_kernel_ssm.m, "The sequential scan";
 * ssm_gated_delta.cu, fc_ssm_recurrence_seq and its warp form; gated_delta_net_decode.metal
 * (per-token pointer advance). Bit-identical to n_tokens decode calls.
 * q, k: [n_seqs][n_tokens][Hk][S]; v, y: [n_seqs][n_tokens][H][S];
 * g, beta: [n_seqs][n_tokens][H]; state as for decode. */
gdn_status gdn_recurrence_scan(float *state, const float *q, const float *k, const float *v,
                               const float *g, const float *beta, float *y, int n_seqs,
                               int n_tokens, int n_k_heads, int n_v_heads, int state_size,
                               float scale, const int32_t *slots, int pool, int32_t *err_count,
                               gdn_stream_t stream);

/* The scan, also writing the state after every position, for speculative
 * decoding: ssm_gated_delta.cu, fc_ssm_recurrence_seq's `snaps` argument. snaps[t]
 * holds the whole recurrent state once position t has been applied, so rolling back
 * to the first M verified positions is a single copy of snaps[M-1].
 * snaps: [n_seqs][n_tokens][H][S][S] (the state layout of one slot per position,
 * sequence n in call order), 16-byte aligned, NULL is an error. Otherwise as
 * gdn_recurrence_scan, whose results it reproduces bit for bit. */
gdn_status gdn_recurrence_scan_snapshots(float *state, const float *q, const float *k,
                                         const float *v, const float *g, const float *beta,
                                         float *y, float *snaps, int n_seqs, int n_tokens,
                                         int n_k_heads, int n_v_heads, int state_size,
                                         float scale, const int32_t *slots, int pool,
                                         int32_t *err_count, gdn_stream_t stream);

/* The multi-token scan in chunks of 32 positions with the state-dependent
 * contractions on the tensor cores (tcgen05: every fp32 operand split into bf16
 * parts hi + lo and each product summed as hi*hi + hi*lo + lo*hi, within about
 * 3 * 2^-16 of the exact product; fp32 accumulation), for long prefill.
 * fm_kernel_ssm.m (the softplus note and the sequential-scan section) refers to
 * a chunked prefill path built on cumulative sums of g within each chunk and
 * keeps the sequential scan as its permanent reference; the chunked algebra
 * itself (an exact regrouping of the recurrence, the WY/UT form) is not given on
 * the pages.
 * Arguments, layouts, ownership and slot semantics exactly as gdn_recurrence_scan
 * (a drop-in replacement); it needs no workspace and allocates nothing. y needs
 * no particular alignment; state, q, k and v are 16-byte aligned (GDN_ERR_ALIGN).
 * Only state_size 128 has this form (else GDN_ERR_UNSUPPORTED). Results agree
 * with the sequential scan to within rounding (the 2e-3-of-RMS bound of a
 * 4096-position scan), not bit for bit. */
gdn_status gdn_recurrence_scan_chunked(float *state, const float *q, const float *k,
                                       const float *v, const float *g, const float *beta,
                                       float *y, int n_seqs, int n_tokens, int n_k_heads,
                                       int n_v_heads, int state_size, float scale,
                                       const int32_t *slots, int pool, int32_t *err_count,
                                       gdn_stream_t stream);

/* Bytes of workspace for gdn_recurrence_scan_chunked_ws to prepare every chunk of
 * the call at once: ceil(n_tokens / 32) * n_seqs * n_v_heads * 36 KiB (W, Ut and M of
 * each chunk, fp32). 0 for invalid sizes or a state_size other than 128. */
size_t gdn_recurrence_scan_chunked_ws_size(int n_seqs, int n_tokens, int n_v_heads,
                                           int state_size);

/* The chunked scan of gdn_recurrence_scan_chunked in two phases: a fully parallel
 * kernel over (chunk, sequence, k-head) forms each chunk's state-independent
 * quantities (Gram products, the forward substitutions of the WY/UT form) in the
 * workspace, then one CTA per (sequence, v-head) advances the state over the
 * chunks on the tensor cores. Same sources on the pages as
 * gdn_recurrence_scan_chunked, and the same bits: both run the same arithmetic in
 * the same order.
 * Arguments, layouts, ownership and slot semantics as gdn_recurrence_scan_chunked,
 * plus workspace: device memory owned by the caller, 16-byte aligned
 * (GDN_ERR_ALIGN), contents on entry irrelevant and garbage afterwards; NULL is
 * GDN_ERR_NULL. A workspace of gdn_recurrence_scan_chunked_ws_size() bytes takes
 * two launches; a smaller one is used in waves of as many chunks as it holds
 * (two launches per wave, same results); less than one chunk's worth
 * (n_seqs * n_v_heads * 36 KiB) is GDN_ERR_SHAPE. Calls that share a workspace
 * must not overlap. */
gdn_status gdn_recurrence_scan_chunked_ws(float *state, const float *q, const float *k,
                                          const float *v, const float *g, const float *beta,
                                          float *y, int n_seqs, int n_tokens, int n_k_heads,
                                          int n_v_heads, int state_size, float scale,
                                          const int32_t *slots, int pool, int32_t *err_count,
                                          void *workspace, size_t workspace_bytes,
                                          gdn_stream_t stream);

/* Snapshots the chunked scan writes for n_tokens positions at interval snap_every
 * (in chunks of 32 positions): floor(n_tokens / (32 * snap_every)); -1 for a
 * negative n_tokens or a snap_every below 1. */
int gdn_chunked_snapshot_count(int n_tokens, int snap_every);

/* gdn_recurrence_scan_chunked_ws, also writing the state at every 32 * snap_every
 * positions, for prefix caching of long prompts: a subsample of what
 * gdn_recurrence_scan_snapshots writes (ssm_gated_delta.cu, fc_ssm_recurrence_seq's
 * `snaps` argument: the whole recurrent state after a position's update).
 * Snapshot j of sequence n is the state once position (j + 1) * 32 * snap_every - 1
 * has been applied, j < gdn_chunked_snapshot_count(n_tokens, snap_every); a call
 * whose n_tokens is a multiple of 32 * snap_every ends on one, equal to the final
 * state. snaps: [n_seqs][n_snaps][H][S][S] (each snapshot laid out as one state
 * slot, sequence n in call order, not by slot), device memory owned by the caller,
 * written, 16-byte aligned (GDN_ERR_ALIGN); NULL when n_snaps > 0 is GDN_ERR_NULL.
 * snap_every below 1 is GDN_ERR_SHAPE. Other arguments, errors, workspace and waves
 * as gdn_recurrence_scan_chunked_ws, whose y and state it reproduces bit for bit;
 * the snapshots are the same fp32 values the scan carries (a continuation from
 * snapshot j gives the bits of the full call's later chunks). */
gdn_status gdn_recurrence_scan_chunked_snapshots(
    float *state, const float *q, const float *k, const float *v, const float *g,
    const float *beta, float *y, float *snaps, int snap_every, int n_seqs, int n_tokens,
    int n_k_heads, int n_v_heads, int state_size, float scale, const int32_t *slots, int pool,
    int32_t *err_count, void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* The two phases of gdn_recurrence_scan_chunked_ws as separate calls, for callers
 * that schedule them themselves (e.g. prepare the next wave of chunks on another
 * stream while the state advances over this one). A chunk range is chunk_begin ..
 * chunk_begin + n_chunks - 1 of the ceil(n_tokens / 32) chunks of every sequence
 * (outside it: GDN_ERR_SHAPE); the workspace holds the range's blocks, n_chunks *
 * n_seqs * n_v_heads * 36 KiB (less: GDN_ERR_SHAPE), 16-byte aligned, the block of
 * chunk chunk_begin + c of (sequence n, v-head vh) at byte offset
 * ((c * n_seqs + n) * n_v_heads + vh) * 36 KiB: W [32][128], Ut [32][128], M [32][32].
 * gdn_chunked_prepare reads q, k, v, g, beta and writes the blocks.
 * gdn_chunked_advance reads the blocks, q, k and g, advances the state over the
 * range and writes y of its positions; it counts skipped sequences (slot semantics
 * as gdn_recurrence_scan) only when chunk_begin == 0, so a sweep over the chunks in
 * order counts each once. Running prepare then advance over consecutive ranges
 * from chunk 0 to the last gives the bits of gdn_recurrence_scan_chunked. Other
 * arguments as gdn_recurrence_scan_chunked_ws. */
gdn_status gdn_chunked_prepare(const float *q, const float *k, const float *v, const float *g,
                               const float *beta, void *workspace, size_t workspace_bytes,
                               int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                               int state_size, int chunk_begin, int n_chunks,
                               gdn_stream_t stream);
gdn_status gdn_chunked_advance(float *state, const float *q, const float *k, const float *g,
                               const void *workspace, size_t workspace_bytes, float *y,
                               int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                               int state_size, float scale, int chunk_begin, int n_chunks,
                               const int32_t *slots, int pool, int32_t *err_count,
                               gdn_stream_t stream);

/* The conv scan, also writing the conv history after every position (ssm_gated_delta.cu,
 * fc_ssm_conv1d_silu_seq's `snaps`): snaps [n_seqs][n_tokens][conv_dim][K-1], the
 * conv_state layout of one slot per position. NULL is an error. Otherwise as
 * gdn_conv1d_silu_seq. */
gdn_status gdn_conv1d_silu_seq_snapshots(const float *qkv, const float *w, float *conv_state,
                                         float *out, float *snaps, int n_seqs, int n_tokens,
                                         int conv_dim, int conv_kernel, const int32_t *slots,
                                         int pool, int32_t *err_count, gdn_stream_t stream);

/* Speculative-decoding rollback for a batch in one launch: the restore the two
 * snapshot scans above exist for (ssm_gated_delta.cu, the `snaps` arguments of
 * fc_ssm_recurrence_seq and fc_ssm_conv1d_silu_seq). Each sequence keeps its own
 * number of verified positions. For sequence n, with M = accepted[n]:
 * state slot slots[n] (n when slots is NULL) <- snaps[n][M-1] (n_v_heads*S*S floats,
 * the layouts of gdn_recurrence_scan_snapshots), and, when conv_state and conv_snaps
 * are both given, its conv slot <- conv_snaps[n][M-1] (conv_dim*(K-1) floats, the
 * layouts of gdn_conv1d_silu_seq_snapshots; both NULL skips the conv history, one NULL
 * is GDN_ERR_NULL). accepted: device int32[n_seqs]; M must lie in [1, n_tokens] (the
 * first verified position is always kept; M = n_tokens leaves the scans' final state).
 * A sequence whose M or slot is out of range is left untouched and counted once in the
 * optional err_count. state_size as the snapshot scan (32, 64, 128 or 256), conv_kernel
 * in [2, 8]. state and snaps 16-byte aligned; copies only, no arithmetic. */
gdn_status gdn_snapshot_restore(float *state, const float *snaps, float *conv_state,
                                const float *conv_snaps, const int32_t *accepted, int n_seqs,
                                int n_tokens, int n_v_heads, int state_size, int conv_dim,
                                int conv_kernel, const int32_t *slots, int pool,
                                int32_t *err_count, gdn_stream_t stream);

/* Gated RMSNorm. fm_kernel_ssm.m, "Gated RMSNorm"; ssm_gated_delta.cu, Kernel 3.
 *   out[r][d] = y[r][d] / sqrt(mean_d(y[r]^2) + eps) * w[d] * silu(z[r][d])
 * y, z, out: [rows][head_dim]; w: [head_dim], the one weight shared by all heads.
 * head_dim in {32, 64, 128, 256}. out may alias y. */
gdn_status gdn_gated_norm(const float *y, const float *w, const float *z, float *out, int rows,
                          int head_dim, float eps, gdn_stream_t stream);

/* The whole block for one decode token per sequence, in one kernel: conv1d+SiLU
 * of the raw qkv row (rolling conv_state), q/k L2-norm, GQA, decay gate, beta =
 * sigmoid(b), recurrence, gated RMSNorm. Each state byte is read and written
 * once. Follows the single-token glue order of ssm_gated_delta.cu ("SSM glue
 * kernels" and Kernels 1-3).
 * qkv: [n_seqs][C] raw; conv_w: [C][4]; conv_state: [pool][C][3] in place;
 * alpha, b: [n_seqs][H] raw gate and beta logits; dt, a: [H]; z: [n_seqs][H][S];
 * norm_w: [S]; state: [pool][H][S][S] in place; out: [n_seqs][H][S].
 * conv_kernel must be 4; n_v_heads / n_k_heads <= 8 (<= 4 at state_size 256, whose head
 * tile is split over two CTAs of a cluster of at most 8); otherwise GDN_ERR_UNSUPPORTED.
 * All pointers 16-byte aligned. With many sequences, consecutive calls visit the
 * (sequence, k-head) groups in alternating directions, so a step starts on the state
 * the previous step wrote last, still in L2; the results do not depend on it. A CUDA
 * graph captures the direction of the call it records: capture two consecutive steps
 * to keep the alternation when replaying. */
gdn_status gdn_block_decode(const float *qkv, const float *conv_w, float *conv_state,
                            const float *alpha, const float *b, const float *dt, const float *a,
                            const float *z, const float *norm_w, float *state, float *out,
                            int n_seqs, int n_k_heads, int n_v_heads, int state_size,
                            int conv_kernel, float scale, float l2_eps, float norm_eps,
                            const int32_t *slots, int pool, int32_t *err_count,
                            gdn_stream_t stream);

/* Bytes of workspace gdn_block_prefill needs for these sizes (0 for invalid ones). */
size_t gdn_block_prefill_workspace_size(int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                                        int state_size);

/* The whole block over n_tokens positions per sequence (prefill), following the
 * batched variants of ssm_gated_delta.cu ("BATCHED (prefill) variants": decay gate,
 * conv scan, q/k norm with the v passthrough, recurrence scan) and the gated
 * RMSNorm: conv1d+SiLU scan (rolling conv_state), q/k L2-norm, decay gate, beta =
 * sigmoid(b), the sequential scan (state in place), gated RMSNorm.
 * qkv: [n_seqs][n_tokens][C] raw; alpha, b: [n_seqs][n_tokens][H]; z, out:
 * [n_seqs][n_tokens][H][S]; the other arguments as for gdn_block_decode (any K in
 * [2, 8]). The result equals n_tokens gdn_block_decode calls up to rounding.
 * workspace: device memory of at least gdn_block_prefill_workspace_size() bytes,
 * 16-byte aligned, owned by the caller; its contents on entry do not matter and
 * are garbage afterwards. Too small: GDN_ERR_SHAPE. Several kernels are enqueued
 * on `stream`; calls that share a workspace must not overlap. */
gdn_status gdn_block_prefill(const float *qkv, const float *conv_w, float *conv_state,
                             const float *alpha, const float *b, const float *dt, const float *a,
                             const float *z, const float *norm_w, float *state, float *out,
                             int n_seqs, int n_tokens, int n_k_heads, int n_v_heads,
                             int state_size, int conv_kernel, float scale, float l2_eps,
                             float norm_eps, const int32_t *slots, int pool, int32_t *err_count,
                             void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* The prefill block over draft positions for speculative decoding: gdn_block_prefill
 * (same arguments, workspace and results, bit for bit) that also keeps, for every
 * position t, the recurrent state after t in snaps [n_seqs][n_tokens][H][S][S] (as
 * gdn_recurrence_scan_snapshots) and the conv history after t in conv_snaps
 * [n_seqs][n_tokens][C][K-1] (as gdn_conv1d_silu_seq_snapshots), C = (2 Hk + H) S.
 * ssm_gated_delta.cu, the `snaps` arguments of fc_ssm_recurrence_seq and
 * fc_ssm_conv1d_silu_seq. After verification, gdn_snapshot_restore rolls each
 * sequence back to its accepted count. snaps 16-byte aligned; NULL snaps or
 * conv_snaps is GDN_ERR_NULL; n_tokens above 65535 is GDN_ERR_UNSUPPORTED. */
gdn_status gdn_block_prefill_snapshots(const float *qkv, const float *conv_w,
                                       float *conv_state, const float *alpha, const float *b,
                                       const float *dt, const float *a, const float *z,
                                       const float *norm_w, float *state, float *out,
                                       float *snaps, float *conv_snaps, int n_seqs,
                                       int n_tokens, int n_k_heads, int n_v_heads,
                                       int state_size, int conv_kernel, float scale,
                                       float l2_eps, float norm_eps, const int32_t *slots,
                                       int pool, int32_t *err_count, void *workspace,
                                       size_t workspace_bytes, gdn_stream_t stream);

/* gdn_block_prefill with the chunked tensor-core scan in place of the sequential
 * one: the production path for long prefill. Same arguments, layouts, workspace and
 * error behaviour; state_size must be 128 (else GDN_ERR_UNSUPPORTED). Results agree
 * with gdn_block_prefill to within rounding (the 2e-3-of-RMS long-scan bound), not
 * bit for bit. With the minimum workspace the scan is gdn_recurrence_scan_chunked;
 * workspace bytes beyond gdn_block_prefill_workspace_size() rounded up to 16 serve
 * gdn_recurrence_scan_chunked_ws (in waves if they hold fewer chunks than the call
 * has; used once they hold one chunk of every sequence and v-head), which gives the
 * same bits faster. gdn_block_prefill_chunked_workspace_size() is the size with room
 * for every chunk at once. */
size_t gdn_block_prefill_chunked_workspace_size(int n_seqs, int n_tokens, int n_k_heads,
                                                int n_v_heads, int state_size);

gdn_status gdn_block_prefill_chunked(const float *qkv, const float *conv_w, float *conv_state,
                                     const float *alpha, const float *b, const float *dt,
                                     const float *a, const float *z, const float *norm_w,
                                     float *state, float *out, int n_seqs, int n_tokens,
                                     int n_k_heads, int n_v_heads, int state_size,
                                     int conv_kernel, float scale, float l2_eps, float norm_eps,
                                     const int32_t *slots, int pool, int32_t *err_count,
                                     void *workspace, size_t workspace_bytes,
                                     gdn_stream_t stream);

/* ---------------------------------------------------------------- ragged batches
 * A prefill batch of sequences of different lengths, packed token-major: every
 * [N][T][...] array of the uniform calls becomes [total_tokens][...], and sequence n
 * owns positions cu_seqlens[n] .. cu_seqlens[n+1] - 1 of it. ssm_gated_delta.cu,
 * "BATCHED (prefill) variants", runs one sequence of n positions per launch; these
 * calls run a whole batch of mixed lengths in the launches of one uniform call, and
 * each sequence gets the bits a call of its own would give it (same kernels, same
 * order of operations).
 * - cu_seqlens: DEVICE int32[n_seqs + 1], owned by the caller. It stays on the device
 *   (the host never reads it), so its entries are checked by the kernels: a sequence
 *   whose range is not valid (cu_seqlens[n] < 0, cu_seqlens[n+1] < cu_seqlens[n],
 *   cu_seqlens[n+1] > total_tokens, or a length above max_tokens) is skipped as an
 *   out-of-range slot is -- its state, conv_state and out rows are not written -- and
 *   counted once in err_count. Ranges of different sequences must not overlap
 *   (overlapping ranges race: undefined results, but every access stays inside the
 *   arrays). Rows of out, and snapshots, at positions no sequence owns are not
 *   written. A sequence of length 0 is a no-op.
 * - total_tokens: rows of the packed arrays; max_tokens: an upper bound on any one
 *   sequence's length (it sizes the grids; host int).
 * - Snapshots (the _snapshots form) are packed the same way: the state after position
 *   t of sequence n is snaps[cu_seqlens[n] + t], [total_tokens][H][S][S]; the conv
 *   history likewise, [total_tokens][C][K-1].
 * - Everything else (slots, pool, err_count, layouts of state and conv_state, scale,
 *   eps, alignment, workspace ownership, no allocation) as for the uniform calls. */

/* The sequential scan over a ragged batch: q, k [total][Hk][S]; v, y [total][H][S];
 * g, beta [total][H]. Otherwise as gdn_recurrence_scan. */
gdn_status gdn_recurrence_scan_varlen(float *state, const float *q, const float *k,
                                      const float *v, const float *g, const float *beta,
                                      float *y, const int32_t *cu_seqlens, int n_seqs,
                                      int total_tokens, int max_tokens, int n_k_heads,
                                      int n_v_heads, int state_size, float scale,
                                      const int32_t *slots, int pool, int32_t *err_count,
                                      gdn_stream_t stream);

/* Bytes of workspace for gdn_recurrence_scan_chunked_varlen to take its two-phase form:
 * (total_tokens / 32 + n_seqs) * n_v_heads * 36 KiB -- chunk c of sequence n takes the
 * block row cu_seqlens[n] / 32 + n + c, whatever the lengths. 0 for invalid sizes or a
 * state_size other than 128. */
size_t gdn_recurrence_scan_chunked_varlen_ws_size(int n_seqs, int total_tokens, int n_v_heads,
                                                  int state_size);

/* The chunked tensor-core scan (state_size 128) over a ragged batch; layouts as
 * gdn_recurrence_scan_varlen. With a workspace of at least
 * gdn_recurrence_scan_chunked_varlen_ws_size() bytes (16-byte aligned, contents
 * irrelevant, garbage afterwards) it runs the two-phase form of
 * gdn_recurrence_scan_chunked_ws in one wave; with a smaller one or NULL, the one-kernel
 * form of gdn_recurrence_scan_chunked. Both give the same bits. */
gdn_status gdn_recurrence_scan_chunked_varlen(float *state, const float *q, const float *k,
                                              const float *v, const float *g, const float *beta,
                                              float *y, const int32_t *cu_seqlens, int n_seqs,
                                              int total_tokens, int max_tokens, int n_k_heads,
                                              int n_v_heads, int state_size, float scale,
                                              const int32_t *slots, int pool,
                                              int32_t *err_count, void *workspace,
                                              size_t workspace_bytes, gdn_stream_t stream);

/* gdn_recurrence_scan_chunked_snapshots over a ragged batch (prefix caching of a batch
 * of prompts of different lengths): the two-phase scan of
 * gdn_recurrence_scan_chunked_varlen, also writing each sequence's state after its
 * positions (j + 1) * 32 * snap_every - 1, j < floor(len / (32 * snap_every)) (len its
 * own length; a sequence that ends on an interval gets its final state as its last
 * snapshot). The snapshots go to a caller-managed pool, as the state goes to state
 * slots: snaps holds snap_pool slots of n_v_heads * S * S floats (the layout of one
 * state slot), 16-byte aligned; sequence n's snapshot j goes to slot snap_base[n] + j
 * (snap_base: int32 device array of n_seqs entries). A sequence whose range does not
 * lie in [0, snap_pool) (a negative base included) writes none of its snapshots and is
 * counted in err_count; its scan, state and y are still computed. snaps and snap_base
 * may be NULL when max_tokens < 32 * snap_every (no snapshot can fall), else NULL is
 * GDN_ERR_NULL; snap_every below 1 or a negative snap_pool is GDN_ERR_SHAPE. The
 * workspace is required: at least gdn_recurrence_scan_chunked_varlen_ws_size() bytes
 * (less: GDN_ERR_SHAPE; NULL: GDN_ERR_NULL). y and state are the bits of
 * gdn_recurrence_scan_chunked_varlen; other arguments as that call. */
gdn_status gdn_recurrence_scan_chunked_snapshots_varlen(
    float *state, const float *q, const float *k, const float *v, const float *g,
    const float *beta, float *y, float *snaps, const int32_t *snap_base, int snap_pool,
    int snap_every, const int32_t *cu_seqlens, int n_seqs, int total_tokens, int max_tokens,
    int n_k_heads, int n_v_heads, int state_size, float scale, const int32_t *slots, int pool,
    int32_t *err_count, void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Workspace of the ragged prefill blocks: gdn_block_prefill_varlen and _snapshots_varlen
 * need gdn_block_prefill_varlen_workspace_size() bytes (the intermediates of
 * total_tokens positions); gdn_block_prefill_chunked_varlen takes its two-phase chunked
 * scan when given gdn_block_prefill_chunked_varlen_workspace_size() bytes, else (at
 * least the former) the one-kernel form, with the same bits. */
size_t gdn_block_prefill_varlen_workspace_size(int n_seqs, int total_tokens, int n_k_heads,
                                               int n_v_heads, int state_size);
size_t gdn_block_prefill_chunked_varlen_workspace_size(int n_seqs, int total_tokens,
                                                       int n_k_heads, int n_v_heads,
                                                       int state_size);

/* gdn_block_prefill over a ragged batch: qkv [total][C]; alpha, b [total][H]; z, out
 * [total][H][S]; any K in [2, 8]. Each sequence's out, state and conv_state are the
 * bits of gdn_block_prefill on that sequence alone. */
gdn_status gdn_block_prefill_varlen(const float *qkv, const float *conv_w, float *conv_state,
                                    const float *alpha, const float *b, const float *dt,
                                    const float *a, const float *z, const float *norm_w,
                                    float *state, float *out, const int32_t *cu_seqlens,
                                    int n_seqs, int total_tokens, int max_tokens, int n_k_heads,
                                    int n_v_heads, int state_size, int conv_kernel, float scale,
                                    float l2_eps, float norm_eps, const int32_t *slots, int pool,
                                    int32_t *err_count, void *workspace, size_t workspace_bytes,
                                    gdn_stream_t stream);

/* gdn_block_prefill_chunked over a ragged batch (state_size 128); each sequence gets the
 * bits of gdn_block_prefill_chunked on that sequence alone. */
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
                                            gdn_stream_t stream);

/* gdn_block_prefill_snapshots over a ragged batch: snaps [total][H][S][S], conv_snaps
 * [total][C][K-1] packed as the positions are; max_tokens above 65535 is
 * GDN_ERR_UNSUPPORTED. gdn_snapshot_restore_varlen rolls each sequence back. */
gdn_status gdn_block_prefill_snapshots_varlen(
    const float *qkv, const float *conv_w, float *conv_state, const float *alpha, const float *b,
    const float *dt, const float *a, const float *z, const float *norm_w, float *state, float *out,
    float *snaps, float *conv_snaps, const int32_t *cu_seqlens, int n_seqs, int total_tokens,
    int max_tokens, int n_k_heads, int n_v_heads, int state_size, int conv_kernel, float scale,
    float l2_eps, float norm_eps, const int32_t *slots, int pool, int32_t *err_count,
    void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* gdn_snapshot_restore for snapshots of a ragged batch: sequence n with M = accepted[n]
 * in [1, its length] gets snaps[cu_seqlens[n] + M - 1] (and conv_snaps likewise). A
 * sequence whose M, slot or range is not valid is left untouched and counted once. */
gdn_status gdn_snapshot_restore_varlen(float *state, const float *snaps, float *conv_state,
                                       const float *conv_snaps, const int32_t *accepted,
                                       const int32_t *cu_seqlens, int n_seqs, int total_tokens,
                                       int max_tokens, int n_v_heads, int state_size,
                                       int conv_dim, int conv_kernel, const int32_t *slots,
                                       int pool, int32_t *err_count, gdn_stream_t stream);

/* Bytes of the fixed device scratch gdn_block_prefill_noalloc works in. */
#define GDN_PREFILL_NOALLOC_SCRATCH_BYTES (32u << 20)

/* gdn_block_prefill without a caller workspace, for callers that cannot allocate
 * device memory: e.g. a plugin that only receives an engine's input and output
 * buffers, or a serving loop that must not allocate mid-step (an allocation can
 * synchronise the whole device). The pages have no counterpart; this is a
 * library convenience.
 * The workspace is a fixed GDN_PREFILL_NOALLOC_SCRATCH_BYTES array in device
 * memory that every GPU loading this library holds until the process exits.
 * Sizes whose gdn_block_prefill_workspace_size() exceeds it return
 * GDN_ERR_UNSUPPORTED before anything is enqueued. The first call on a device
 * looks up the array's device address on the current device (the stream must
 * belong to it); make that first call before any stream capture. All calls share
 * the array, which keeps the last call's contents (nothing in it needs to start
 * at zero): calls that overlap on the GPU, on any stream, race. Allocates
 * nothing. Arguments and results otherwise as gdn_block_prefill. */
gdn_status gdn_block_prefill_noalloc(const float *qkv, const float *conv_w, float *conv_state,
                                     const float *alpha, const float *b, const float *dt,
                                     const float *a, const float *z, const float *norm_w,
                                     float *state, float *out, int n_seqs, int n_tokens,
                                     int n_k_heads, int n_v_heads, int state_size,
                                     int conv_kernel, float scale, float l2_eps, float norm_eps,
                                     const int32_t *slots, int pool, int32_t *err_count,
                                     gdn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H */
