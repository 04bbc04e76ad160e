/*
 * gdn_ref.c -- CPU oracle for the gated delta-rule SSM block.
 *
 * TEST INFRASTRUCTURE ONLY (see gdn_ref.h). Plain single-threaded C99, written
 * from the equations on the pages, one step per function, sums in index order.
 * Sources, by page and section:
 *   [fm]   fm_kernel_ssm.m (Foundry, Metal host + shader source)
 *   [cu]   ssm_gated_delta.cu (Foundry, CUDA kernels for the K80)
 *   [mlx]  gated_delta_net_decode.metal (mlx-native 0.21.1)
 *
 * Every function here is pinned by a test in tests/test_oracle.py against a
 * closed form, an invariant or an independent dense-matrix formulation.
 */
#include "gdn_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#if defined(GDN_REF_DOUBLE)
#define R_EXP exp
#define R_LOG1P log1p
#define R_SQRT sqrt
#define R_FMAX fmax
#else
#define R_EXP expf
#define R_LOG1P log1pf
#define R_SQRT sqrtf
#define R_FMAX fmaxf
#endif

int gdn_ref_precision(void) { return (int)(sizeof(gdn_real) / sizeof(float)); }

/* Softplus, log(1 + e^v), taken as v itself above 20: both pages guard it there
 * ([fm] decay-gate section, [cu] fc_ssm_decay_gate). Above 20 the dropped term
 * log1p(exp(-v)) is below 2.1e-9. */
gdn_real gdn_ref_softplus(gdn_real v) {
    if (v > (gdn_real)20) return v;
    return R_LOG1P(R_EXP(v));
}

/* SiLU in the divisor form both pages use: [fm] fmssm_silu, [cu] fc_ssm_silu. */
gdn_real gdn_ref_silu(gdn_real x) { return x / ((gdn_real)1 + R_EXP(-x)); }

/* Decay gate, [fm] decay-gate section: g = a * softplus(alpha + dt) per row and head;
 * dt and a are per head, broadcast over rows. a = -exp(A_log) is baked by the
 * caller ([cu] "Glue" section, fc_ssm_decay_gate). */
void gdn_ref_decay_gate(const gdn_real *alpha, const gdn_real *dt, const gdn_real *a,
                        gdn_real *g, int n_heads, int rows) {
    for (int r = 0; r < rows; r++)
        for (int h = 0; h < n_heads; h++) {
            size_t idx = (size_t)r * n_heads + h;
            g[idx] = a[h] * gdn_ref_softplus(alpha[idx] + dt[h]);
        }
}

/* beta = sigmoid(b) = 1 / (1 + e^-b), [cu] fc_sigmoid. */
void gdn_ref_sigmoid(const gdn_real *b, gdn_real *beta, int n) {
    for (int i = 0; i < n; i++) beta[i] = (gdn_real)1 / ((gdn_real)1 + R_EXP(-b[i]));
}

static int slot_of(const int32_t *slots, int n) { return slots ? (int)slots[n] : n; }

/* Causal depthwise conv1d + SiLU, [fm] "Causal depthwise conv1d + SiLU" and
 * [cu] "Kernel 2" plus its batched form. Per channel c the window is the
 * (K-1)-deep history (oldest first) followed by the current input x:
 *     pre = x * w[c][K-1] + sum_{t=0}^{K-2} hist[t] * w[c][t]
 * accumulated newest tap first, then history oldest-first. The history then
 * drops its oldest tap and appends the RAW x (not the convolved value). */
int gdn_ref_conv1d_silu_seq(const gdn_real *qkv, const gdn_real *w, gdn_real *conv_state,
                            gdn_real *out, int n_seqs, int n_tokens, int conv_dim,
                            int conv_kernel, const int32_t *slots, int pool,
                            int apply_silu) {
    const int K = conv_kernel, taps = conv_kernel - 1;
    int skipped = 0;
    for (int n = 0; n < n_seqs; n++) {
        const int slot = slot_of(slots, n);
        if (slot < 0 || slot >= pool) { skipped++; continue; }
        for (int t = 0; t < n_tokens; t++) {
            const gdn_real *x_row = qkv + ((size_t)n * n_tokens + t) * conv_dim;
            gdn_real *o_row = out + ((size_t)n * n_tokens + t) * conv_dim;
            for (int c = 0; c < conv_dim; c++) {
                const gdn_real *wc = w + (size_t)c * K;
                gdn_real *hist = conv_state + ((size_t)slot * conv_dim + c) * taps;
                const gdn_real x = x_row[c];
                gdn_real pre = x * wc[K - 1];
                for (int u = 0; u < taps; u++) pre += hist[u] * wc[u];
                o_row[c] = apply_silu ? gdn_ref_silu(pre) : pre;
                for (int u = 0; u + 1 < taps; u++) hist[u] = hist[u + 1];
                hist[taps - 1] = x;
            }
        }
    }
    return skipped;
}

/* L2-norm of one head vector, [cu] fc_ssm_qknorm_gqa: the vector divided by the
 * larger of its Euclidean norm and eps. Applied to q and k after conv+SiLU, never
 * to v. */
void gdn_ref_l2norm(const gdn_real *x, gdn_real *out, int rows, int dim, gdn_real eps) {
    for (int r = 0; r < rows; r++) {
        const gdn_real *xr = x + (size_t)r * dim;
        gdn_real ss = 0;
        for (int d = 0; d < dim; d++) ss += xr[d] * xr[d];
        const gdn_real nrm = R_FMAX(R_SQRT(ss), eps);
        for (int d = 0; d < dim; d++) out[(size_t)r * dim + d] = xr[d] / nrm;
    }
}

/* The delta-rule recurrence on the transposed state, [fm] "Delta-rule
 * recurrence -- register-resident" and "The sequential scan", [cu] "Kernel 1",
 * [mlx] "Mathematical recurrence". Row j of head vh is S_vh[:, j]; per token:
 *     row   <- exp(g) * row
 *     pred  =  sum_i row[i] * k[i]
 *     delta =  (v[j] - pred) * beta
 *     row   <- row + k * delta
 *     y[j]  =  scale * sum_i row[i] * q[i]      (read after the write)
 * GQA: v-head vh reads k-head vh % n_k_heads ([mlx] "GQA: tiled mapping"; [cu]
 * interleaved tiling vh = r*n_k_heads + kh). The scan is this step repeated with
 * the state carried, so decode and scan share this one code path. */
int gdn_ref_recurrence(gdn_real *state, const gdn_real *q, const gdn_real *k,
                       const gdn_real *v, const gdn_real *g, const gdn_real *beta,
                       gdn_real *y, int n_seqs, int n_tokens, int n_k_heads,
                       int n_v_heads, int state_size, gdn_real scale,
                       const int32_t *slots, int pool) {
    const int S = state_size, H = n_v_heads, Hk = n_k_heads;
    int skipped = 0;
    for (int n = 0; n < n_seqs; n++) {
        const int slot = slot_of(slots, n);
        if (slot < 0 || slot >= pool) { skipped++; continue; }
        for (int t = 0; t < n_tokens; t++) {
            const size_t nt = (size_t)n * n_tokens + t;
            for (int vh = 0; vh < H; vh++) {
                const int kh = vh % Hk;
                const gdn_real *kv = k + (nt * Hk + kh) * S;
                const gdn_real *qv = q + (nt * Hk + kh) * S;
                const gdn_real *vv = v + (nt * H + vh) * S;
                gdn_real *yv = y + (nt * H + vh) * S;
                const gdn_real decay = R_EXP(g[nt * H + vh]);
                const gdn_real b = beta[nt * H + vh];
                for (int j = 0; j < S; j++) {
                    gdn_real *row = state + (((size_t)slot * H + vh) * S + j) * S;
                    for (int i = 0; i < S; i++) row[i] = row[i] * decay;
                    gdn_real pred = 0;
                    for (int i = 0; i < S; i++) pred += row[i] * kv[i];
                    const gdn_real delta = (vv[j] - pred) * b;
                    for (int i = 0; i < S; i++) row[i] = row[i] + kv[i] * delta;
                    gdn_real acc = 0;
                    for (int i = 0; i < S; i++) acc += row[i] * qv[i];
                    yv[j] = scale * acc;
                }
            }
        }
    }
    return skipped;
}

/* Gated RMSNorm, [fm] "Gated RMSNorm" and [cu] "Kernel 3":
 *     out[d] = y[d] * (1 / sqrt(mean(y^2) + eps)) * w[d] * silu(z[d])
 * with one weight vector of length head_dim shared by every head. */
void gdn_ref_gated_norm(const gdn_real *y, const gdn_real *w, const gdn_real *z,
                        gdn_real *out, int rows, int head_dim, gdn_real eps) {
    for (int r = 0; r < rows; r++) {
        const gdn_real *yr = y + (size_t)r * head_dim;
        const gdn_real *zr = z + (size_t)r * head_dim;
        gdn_real ss = 0;
        for (int d = 0; d < head_dim; d++) ss += yr[d] * yr[d];
        const gdn_real inv_rms = (gdn_real)1 / R_SQRT(ss / (gdn_real)head_dim + eps);
        for (int d = 0; d < head_dim; d++)
            out[(size_t)r * head_dim + d] = yr[d] * inv_rms * w[d] * gdn_ref_silu(zr[d]);
    }
}

/* One decode token of the block, in the order of the [cu] single-token glue:
 * conv1d+SiLU over the packed [q | k | v] channels, L2-norm of q and k per
 * k-head (v passes through), decay gate, beta = sigmoid(b), recurrence, gated
 * RMSNorm. Built from the functions above; scratch is heap-allocated here. */
int gdn_ref_block_decode(const gdn_real *qkv, const gdn_real *conv_w, gdn_real *conv_state,
                         const gdn_real *alpha, const gdn_real *b, const gdn_real *dt,
                         const gdn_real *a, const gdn_real *z, const gdn_real *norm_w,
                         gdn_real *state, gdn_real *out, int n_seqs, int n_k_heads,
                         int n_v_heads, int state_size, int conv_kernel, gdn_real scale,
                         gdn_real l2_eps, gdn_real norm_eps, const int32_t *slots,
                         int pool) {
    const int S = state_size, H = n_v_heads, Hk = n_k_heads;
    const int key_dim = Hk * S, conv_dim = 2 * key_dim + H * S;
    gdn_real *conv_out = (gdn_real *)malloc(sizeof(gdn_real) * (size_t)conv_dim);
    gdn_real *qn = (gdn_real *)malloc(sizeof(gdn_real) * (size_t)key_dim);
    gdn_real *kn = (gdn_real *)malloc(sizeof(gdn_real) * (size_t)key_dim);
    gdn_real *g = (gdn_real *)malloc(sizeof(gdn_real) * (size_t)H);
    gdn_real *bt = (gdn_real *)malloc(sizeof(gdn_real) * (size_t)H);
    gdn_real *y = (gdn_real *)malloc(sizeof(gdn_real) * (size_t)H * S);
    int skipped = 0;
    for (int n = 0; n < n_seqs; n++) {
        const int slot = slot_of(slots, n);
        if (slot < 0 || slot >= pool) { skipped++; continue; }
        const int32_t one_slot = slot;
        gdn_ref_conv1d_silu_seq(qkv + (size_t)n * conv_dim, conv_w, conv_state, conv_out, 1, 1,
                                conv_dim, conv_kernel, &one_slot, pool, 1);
        gdn_ref_l2norm(conv_out, qn, Hk, S, l2_eps);
        gdn_ref_l2norm(conv_out + key_dim, kn, Hk, S, l2_eps);
        gdn_ref_decay_gate(alpha + (size_t)n * H, dt, a, g, H, 1);
        gdn_ref_sigmoid(b + (size_t)n * H, bt, H);
        gdn_ref_recurrence(state, qn, kn, conv_out + 2 * key_dim, g, bt, y, 1, 1, Hk, H, S,
                           scale, &one_slot, pool);
        gdn_ref_gated_norm(y, norm_w, z + (size_t)n * H * S, out + (size_t)n * H * S, H, S,
                           norm_eps);
    }
    free(conv_out); free(qn); free(kn); free(g); free(bt); free(y);
    return skipped;
}
