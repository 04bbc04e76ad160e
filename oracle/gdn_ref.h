/*
 * gdn_ref.h -- CPU oracle for the gated delta-rule (Gated-DeltaNet) SSM block.
 *
 * TEST INFRASTRUCTURE ONLY. This is the slow, obviously-correct reference the
 * CUDA library is checked against. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * One source, two precisions: the build compiles it once with
 * gdn_real = float (the precision the pages' kernels and CPU reference use)
 * and once with -DGDN_REF_DOUBLE, gdn_real = double (the "exact" reference the GPU error is
 * measured against). Every array argument is of that real type, host memory,
 * caller-owned. Compiled with -ffp-contract=off so no multiply-add is fused and
 * every sum runs in index order 0..n-1.
 *
 * Layouts (all row-major, innermost last):
 *   state       [pool][H][S][S]   state[((slot*H + h)*S + j)*S + i] == S_h[i][j]
 *   conv_state  [pool][C][K-1]    oldest tap first, holding RAW inputs
 *   conv weight [C][K]            w[c][K-1] multiplies the current input
 *   qkv / conv_out [N][T][C]      C = 2*Hk*S + H*S, packed [q | k | v]
 *   q, k        [N][T][Hk][S]     k-head space (post L2-norm for the recurrence)
 *   v, y, z     [N][T][H][S]
 *   g, beta     [N][T][H]
 *
 * Sequence n uses pool slot slots[n] (or n when slots is NULL). A sequence whose
 * slot lies outside [0, pool) is skipped (nothing of it is written) and counted
 * in the return value.
 */
#ifndef GDN_REF_H
#define GDN_REF_H

#include <stdint.h>

#if defined(GDN_REF_DOUBLE)
typedef double gdn_real;
#else
typedef float gdn_real;
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* 1 if built with float, 2 if built with double. */
int gdn_ref_precision(void);

/* softplus(v) = v > 20 ? v : log1p(exp(v)); silu(x) = x / (1 + exp(-x)). */
gdn_real gdn_ref_softplus(gdn_real v);
gdn_real gdn_ref_silu(gdn_real x);

/* g[r][h] = a[h] * softplus(alpha[r][h] + dt[h]) for r < rows, h < n_heads. */
void gdn_ref_decay_gate(const gdn_real *alpha, const gdn_real *dt, const gdn_real *a,
                        gdn_real *g, int n_heads, int rows);

/* beta[i] = 1 / (1 + exp(-b[i])). */
void gdn_ref_sigmoid(const gdn_real *b, gdn_real *beta, int n);

/* Causal depthwise conv1d + SiLU over n_tokens positions of each sequence,
 * rolling conv_state. With apply_silu == 0 the pre-activation is written
 * instead (used by the impulse-response pin). Returns the skipped count. */
int gdn_ref_conv1d_silu_seq(const gdn_real *qkv, const gdn_real *w, gdn_real *conv_state,
                            gdn_real *out, int n_seqs, int n_tokens, int conv_dim,
                            int conv_kernel, const int32_t *slots, int pool,
                            int apply_silu);

/* out[r][:] = x[r][:] / max(||x[r][:]||_2, eps) for r < rows (row length dim). */
void gdn_ref_l2norm(const gdn_real *x, gdn_real *out, int rows, int dim, gdn_real eps);

/* Delta-rule recurrence over n_tokens positions per sequence (decode is
 * n_tokens == 1). q, k are post-norm in k-head space; v-head vh reads k-head
 * vh % n_k_heads. State updated in place. Returns the skipped count. */
int gdn_ref_recurrence(gdn_real *state, const gdn_real *q, const gdn_real *k,
                       const gdn_real *v, const gdn_real *g, const gdn_real *beta,
                       gdn_real *y, int n_seqs, int n_tokens, int n_k_heads,
                       int n_v_heads, int state_size, gdn_real scale,
                       const int32_t *slots, int pool);

/* out[r][d] = y[r][d] / sqrt(mean_d(y[r]^2) + eps) * w[d] * silu(z[r][d]). */
void gdn_ref_gated_norm(const gdn_real *y, const gdn_real *w, const gdn_real *z,
                        gdn_real *out, int rows, int head_dim, gdn_real eps);

/* One decode token of the whole block per sequence: conv1d+SiLU over the raw
 * qkv row, q/k L2-norm, decay gate, beta sigmoid, recurrence, gated RMSNorm.
 * Returns the skipped count. */
int gdn_ref_block_decode(const gdn_real *qkv, const gdn_real *conv_w, gdn_real *conv_state,
                         const gdn_real *alpha, const gdn_real *b, const gdn_real *dt,
                         const gdn_real *a, const gdn_real *z, const gdn_real *norm_w,
                         gdn_real *state, gdn_real *out, int n_seqs, int n_k_heads,
                         int n_v_heads, int state_size, int conv_kernel, gdn_real scale,
                         gdn_real l2_eps, gdn_real norm_eps, const int32_t *slots,
                         int pool);

#ifdef __cplusplus
}
#endif
#endif /* GDN_REF_H */
