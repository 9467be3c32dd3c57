/*
 * gdn_oracle.h -- CPU oracle of the Gated DeltaNet (GDN) layer core forward.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The CUDA library and its
 * Python binding never include, link or call it, and it shares no code with
 * them.
 *
 * Every quantity is computed in double precision from float inputs that
 * already hold the activation-dtype-rounded values. The functions follow the
 * definitions step by step:
 *
 *  - "GDN Elementwise Fusion" (Megatron Core developer guide), option table:
 *    the pre-GDR steps (causal convolution, SiLU, Q/K L2 normalisation, head
 *    expansion, beta and decay preparation) and the post-GDR step (output
 *    RMSNorm then SiLU gating). Section "Execution and numerical behavior":
 *    the RMSNorm result is materialised in the activation dtype before the
 *    FP32 gating multiply.
 *  - "perf(gated_delta_net): fold q/k L2-norm into the gated_delta_rule
 *    kernel" (Megatron-LM PR #5396), section "Why": L2 norm with eps = 1e-6,
 *    per head over the last dimension.
 *  - "fused q/k/v short conv" (flash-linear-attention PR #972), sections
 *    "Summary" and "Why": depthwise (per-channel) causal short convolution of
 *    the q/k/v projections; concatenating channels leaves the math unchanged.
 *  - The gated delta rule of the GDN core:
 *        S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *        o_t = S_t q_t,  beta = sigmoid(b),  g = -exp(A_log) softplus(a + dt_bias).
 *
 * Parity status: every function here is pinned by the CPU tests (closed
 * forms, brute force on tiny inputs, invariants); see tests/test_oracle_*.py.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* activation dtype codes (rounding of the RMSNorm output); GDN_ORACLE_F64
 * leaves it unrounded (the real-valued forward that the backward differentiates) */
enum { GDN_ORACLE_F32 = 0, GDN_ORACLE_BF16 = 1, GDN_ORACLE_F16 = 2, GDN_ORACLE_F64 = 3 };

/* Round x to the nearest value of the activation dtype, ties to even. */
double gdn_oracle_round_act(double x, int act);

/* y[t][c] = silu( sum_{i=0..width-1} w[c][i] * x[t-(width-1)+i][c] ), where x is
 * zero before the start of the sequence holding t.  seq_start[0..n_seq] are
 * token offsets; x row t is at x + t*x_stride; y is [ntok][nch] dense. */
void gdn_oracle_conv_silu(int n_seq, const int64_t *seq_start, int nch, int width,
                          const float *x, int64_t x_stride, const float *w,
                          double *y);

/* The same with the raw inputs of the width-1 tokens before each sequence
 * start given: prefix rows [n_seq][width-1][prefix_stride] (oldest first)
 * stand in for the zeros. prefix NULL: as gdn_oracle_conv_silu. */
void gdn_oracle_conv_silu_prefix(int n_seq, const int64_t *seq_start, int nch, int width,
                                 const float *x, int64_t x_stride, const float *w,
                                 const float *prefix, int64_t prefix_stride, double *y);

/* In place, per row and per head: x <- x / sqrt(sum x^2 + eps). x is
 * [nrows][nheads*d]. */
void gdn_oracle_l2norm(int64_t nrows, int nheads, int d, double eps, double *x);

/* beta = sigmoid(b), g = -exp(A_log[h]) * softplus(a + dt_bias[h]);
 * a, b, beta, g are [ntok][H]. */
void gdn_oracle_beta_decay(int64_t ntok, int H, const float *a, const float *b,
                           const float *A_log, const float *dt_bias,
                           double *beta, double *g);

/* Token-by-token gated delta rule for one (sequence, v head).
 * q,k: [T][dk] rows at the given strides; v: [T][dv]; beta, g: T values at
 * stride bg_stride.  h0: initial state stored transposed, h0[i*dv+j] = S[j][i]
 * (dk x dv), or NULL for zeros.  o: [T][dv] at o_stride (o_t = scale*S_t q_t).
 * hT: final state, same layout as h0 (may be NULL). */
void gdn_oracle_delta_rule(int T, int dk, int dv,
                           const double *q, int64_t q_stride,
                           const double *k, int64_t k_stride,
                           const double *v, int64_t v_stride,
                           const double *beta, const double *g, int64_t bg_stride,
                           double scale, const double *h0,
                           double *o, int64_t o_stride, double *hT);

/* The same map computed chunk by chunk (chunk length C) in the WY/UT form;
 * same arguments and results as gdn_oracle_delta_rule. */
void gdn_oracle_delta_rule_chunked(int T, int dk, int dv, int C,
                                   const double *q, int64_t q_stride,
                                   const double *k, int64_t k_stride,
                                   const double *v, int64_t v_stride,
                                   const double *beta, const double *g, int64_t bg_stride,
                                   double scale, const double *h0,
                                   double *o, int64_t o_stride, double *hT);

/* y = round_act(norm_w * o / sqrt(mean(o^2) + eps)) * silu(gate), per row of
 * dv values; o, gate, y rows at the given strides. The product is not
 * rounded (the caller compares it with a tolerance). */
void gdn_oracle_gated_rmsnorm(int64_t nrows, int dv,
                              const double *o, int64_t o_stride,
                              const float *gate, int64_t gate_stride,
                              const float *norm_w, double eps, int act,
                              double *y, int64_t y_stride);

/* Whole core forward for v heads [head_begin, head_end). All inputs are float
 * arrays over the flattened token axis (ntok = seq_start[n_seq]):
 *   q_raw, k_raw [ntok][Hk*dk], v_raw [ntok][Hv*dv], a, b [ntok][Hv],
 *   gate [ntok][Hv*dv], conv_w [2*Hk*dk+Hv*dv][width] (q|k|v order),
 *   A_log, dt_bias [Hv], norm_w [dv], initial_state [n_seq][Hv][dk][dv] or NULL.
 * Outputs (double): out [ntok][Hv][dv], final_state [n_seq][Hv][dk][dv] or NULL.
 * V head h reads q/k head h / (Hv/Hk). Returns 0, or -1 on bad arguments or
 * allocation failure. */
typedef struct {
    int n_seq;
    const int64_t *seq_start; /* [n_seq+1] */
    int Hk, Hv, dk, dv, conv_width;
    int act;
    double l2_eps, norm_eps, scale;
    const float *q_raw, *k_raw, *v_raw, *a, *b, *gate, *conv_w;
    const float *A_log, *dt_bias, *norm_w, *initial_state;
    double *out, *final_state;
    int chunked;    /* 0: token loop; >0: chunked variant with this chunk length */
    /* NULL, or the raw inputs of the width-1 tokens before each sequence start,
     * [n_seq][width-1][2*Hk*dk+Hv*dv] (q|k|v channels, oldest first): the conv
     * reads them instead of zeros (a sequence continued from an earlier part) */
    const float *conv_prefix;
} gdn_oracle_problem;

int gdn_oracle_forward(const gdn_oracle_problem *p, int head_begin, int head_end);

/* One decode step: a single new token for each of n_seq sequences, given each
 * sequence's conv cache and state (the forward of one more token of those
 * sequences; the decode entry of the GPU library has no counterpart on the
 * pages beyond the forward it must agree with).
 *   q_raw, k_raw [n_seq][Hk*dk], v_raw [n_seq][Hv*dv], a, b [n_seq][Hv],
 *   gate [n_seq][Hv*dv], conv_w, A_log, dt_bias, norm_w as in the forward;
 *   conv_state [n_seq][ch][width-1]: the raw inputs of the sequence's last
 *   width-1 tokens per channel, oldest first (ch = 2*Hk*dk + Hv*dv, q|k|v
 *   order; zeros where the sequence is shorter);
 *   state [n_seq][Hv][dk][dv]: S^T as in the forward, in double precision
 *   (so that a chain of steps carries the state as the forward does).
 * Outputs (double): out [n_seq][Hv][dv]; conv_state_out and state_out in the
 * layouts of conv_state and state, advanced by the token. Returns 0, or -1. */
typedef struct {
    int n_seq, Hk, Hv, dk, dv, conv_width, act;
    double l2_eps, norm_eps, scale;
    const float *q_raw, *k_raw, *v_raw, *a, *b, *gate, *conv_w;
    const float *A_log, *dt_bias, *norm_w, *conv_state;
    const double *state;
    double *out, *conv_state_out, *state_out;
} gdn_oracle_decode_problem;
int gdn_oracle_decode(const gdn_oracle_decode_problem *p);

/* Backward of the whole core (gdn_oracle_bwd.c): the gradients of
 *   L = sum(grad_out * out) + sum(grad_final * final_state)
 * with respect to every input of gdn_oracle_forward, the RMSNorm rounding taken
 * as the identity. Inputs as in the forward plus grad_out [ntok][Hv][dv] and
 * grad_final [n_seq][Hv][dk][dv] (or NULL for zeros). Outputs (double, each
 * written in full for the heads of the call):
 *   dq_raw, dk_raw [ntok][Hk*dk], dv_raw [ntok][Hv*dv], da, db [ntok][Hv],
 *   dgate [ntok][Hv*dv], dconv_w [ch][width], dA_log, ddt_bias [Hv],
 *   dnorm_w [Hv][dv] (each v head's share; the gradient is their sum),
 *   dinitial_state [n_seq][Hv][dk][dv] or NULL.
 * gdn_oracle_backward(p, b, e) covers q/k heads [b, e) and their v heads. */
typedef struct {
    int n_seq;
    const int64_t *seq_start;
    int Hk, Hv, dk, dv, conv_width;
    double l2_eps, norm_eps, scale;
    const float *q_raw, *k_raw, *v_raw, *a, *b, *gate, *conv_w;
    const float *A_log, *dt_bias, *norm_w, *initial_state;
    const float *grad_out, *grad_final;
    double *dq_raw, *dk_raw, *dv_raw, *da, *db, *dgate, *dconv_w;
    double *dA_log, *ddt_bias, *dnorm_w, *dinitial_state;
} gdn_oracle_bwd_problem;
int gdn_oracle_backward(const gdn_oracle_bwd_problem *p, int hk_begin, int hk_end);

#ifdef __cplusplus
}
#endif
#endif
