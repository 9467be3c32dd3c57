/*
 * gdn_oracle.c -- CPU oracle of the Gated DeltaNet (GDN) layer core forward.
 *
 * TEST INFRASTRUCTURE ONLY: see gdn_oracle.h for the sources each function
 * follows and for who may call it. Plain loops, double precision, no
 * blocking or reordering beyond what each definition states.
 */
#include "gdn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static double silu(double x) { return x / (1.0 + exp(-x)); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus(x) = log(1 + e^x), written so that e^x never overflows */
static double softplus(double x) {
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

/* Round to a binary format with p significand bits (implicit bit included),
 * minimum normal exponent emin and largest finite value maxv; ties to even
 * (nearbyint in the default rounding mode). */
static double round_format(double x, int p, int emin, double maxv) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);              /* |x| in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E < emin) E = emin;    /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, E - (p - 1));
    double r = nearbyint(x / quantum) * quantum;
    if (fabs(r) > maxv) r = copysign(INFINITY, x);
    return r;
}

double gdn_oracle_round_act(double x, int act) {
    switch (act) {
    case GDN_ORACLE_BF16:
        return round_format(x, 8, -126, ldexp(255.0, 120));   /* (2-2^-7)*2^127 */
    case GDN_ORACLE_F16:
        return round_format(x, 11, -14, 65504.0);
    case GDN_ORACLE_F64:
        return x;
    default:
        return round_format(x, 24, -126, ldexp(16777215.0, 104)); /* FLT_MAX */
    }
}

void gdn_oracle_conv_silu_prefix(int n_seq, const int64_t *seq_start, int nch, int width,
                                 const float *x, int64_t x_stride, const float *w,
                                 const float *prefix, int64_t prefix_stride, double *y) {
    for (int n = 0; n < n_seq; ++n) {
        for (int64_t t = seq_start[n]; t < seq_start[n + 1]; ++t) {
            for (int c = 0; c < nch; ++c) {
                double acc = 0.0;
                for (int i = 0; i < width; ++i) {
                    int64_t tau = t - (width - 1) + i;   /* tap width-1 is the current token */
                    double xv;
                    if (tau >= seq_start[n]) {
                        xv = (double)x[tau * x_stride + c];
                    } else if (prefix) {                 /* the raw tokens before the start */
                        int64_t r = tau - (seq_start[n] - (width - 1));   /* 0 = oldest */
                        xv = (double)prefix[((int64_t)n * (width - 1) + r) * prefix_stride + c];
                    } else {
                        continue;                        /* zero before the sequence start */
                    }
                    acc += (double)w[(int64_t)c * width + i] * xv;
                }
                y[t * nch + c] = silu(acc);
            }
        }
    }
}

void gdn_oracle_conv_silu(int n_seq, const int64_t *seq_start, int nch, int width,
                          const float *x, int64_t x_stride, const float *w,
                          double *y) {
    gdn_oracle_conv_silu_prefix(n_seq, seq_start, nch, width, x, x_stride, w, NULL, 0, y);
}

void gdn_oracle_l2norm(int64_t nrows, int nheads, int d, double eps, double *x) {
    for (int64_t r = 0; r < nrows; ++r) {
        for (int h = 0; h < nheads; ++h) {
            double *row = x + (r * nheads + h) * d;
            double ss = 0.0;
            for (int i = 0; i < d; ++i) ss += row[i] * row[i];
            double inv = 1.0 / sqrt(ss + eps);
            for (int i = 0; i < d; ++i) row[i] *= inv;
        }
    }
}

static void beta_decay_one(double a, double b, double A_log, double dt_bias,
                           double *beta, double *g) {
    *beta = sigmoid(b);
    *g = -exp(A_log) * softplus(a + dt_bias);
}

void gdn_oracle_beta_decay(int64_t ntok, int H, const float *a, const float *b,
                           const float *A_log, const float *dt_bias,
                           double *beta, double *g) {
    for (int64_t t = 0; t < ntok; ++t)
        for (int h = 0; h < H; ++h)
            beta_decay_one(a[t * H + h], b[t * H + h], A_log[h], dt_bias[h],
                           &beta[t * H + h], &g[t * H + h]);
}

void gdn_oracle_delta_rule(int T, int dk, int dv,
                           const double *q, int64_t q_stride,
                           const double *k, int64_t k_stride,
                           const double *v, int64_t v_stride,
                           const double *beta, const double *g, int64_t bg_stride,
                           double scale, const double *h0,
                           double *o, int64_t o_stride, double *hT) {
    /* S is dv x dk: S[j][i] at S[j*dk + i] */
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *Sk = (double *)malloc((size_t)dv * sizeof(double));
    if (h0)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(int64_t)j * dk + i] = h0[(int64_t)i * dv + j];
    for (int t = 0; t < T; ++t) {
        const double *qt = q + t * q_stride, *kt = k + t * k_stride, *vt = v + t * v_stride;
        double bt = beta[t * bg_stride];
        double decay = exp(g[t * bg_stride]);
        /* S_{t-1} (I - b k k^T) = S_{t-1} - b (S_{t-1} k) k^T */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += S[(int64_t)j * dk + i] * kt[i];
            Sk[j] = acc;
        }
        for (int j = 0; j < dv; ++j)
            for (int i = 0; i < dk; ++i) {
                double *s = &S[(int64_t)j * dk + i];
                *s = decay * (*s - bt * Sk[j] * kt[i]) + bt * vt[j] * kt[i];
            }
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += S[(int64_t)j * dk + i] * qt[i];
            o[t * o_stride + j] = scale * acc;
        }
    }
    if (hT)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) hT[(int64_t)i * dv + j] = S[(int64_t)j * dk + i];
    free(S);
    free(Sk);
}

/*
 * Chunked form. Within a chunk of L tokens with gam_i = sum_{u<=i} g_u:
 *   A[i][j] = beta_i exp(gam_i - gam_j) (k_i . k_j) for j < i (zero otherwise)
 *   Tm = (I + A)^{-1}                                  (forward substitution)
 *   W  = Tm diag(beta exp(gam)) K,   U = Tm diag(beta) V
 *   Vn = U - W H                     (H = S^T of the chunk's start, dk x dv)
 *   o_i = scale ( exp(gam_i) q_i^T H + sum_{j<=i} exp(gam_i - gam_j)(q_i . k_j) Vn_j )
 *   H  <- exp(gam_L) H + sum_j exp(gam_L - gam_j) k_j Vn_j^T
 * exp() is only ever taken of a difference gam_i - gam_j with j <= i, or of
 * gam_i itself, so no factor exceeds 1.
 */
void gdn_oracle_delta_rule_chunked(int T, int dk, int dv, int C,
                                   const double *q, int64_t q_stride,
                                   const double *k, int64_t k_stride,
                                   const double *v, int64_t v_stride,
                                   const double *beta, const double *g, int64_t bg_stride,
                                   double scale, const double *h0,
                                   double *o, int64_t o_stride, double *hT) {
    double *H = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *gam = (double *)malloc((size_t)C * sizeof(double));
    double *A = (double *)malloc((size_t)C * C * sizeof(double));
    double *Tm = (double *)malloc((size_t)C * C * sizeof(double));
    double *W = (double *)malloc((size_t)C * dk * sizeof(double));
    double *U = (double *)malloc((size_t)C * dv * sizeof(double));
    double *Vn = (double *)malloc((size_t)C * dv * sizeof(double));
    if (h0) memcpy(H, h0, (size_t)dk * dv * sizeof(double));
    for (int c0 = 0; c0 < T; c0 += C) {
        int L = (T - c0) < C ? (T - c0) : C;
        const double *Q = q + (int64_t)c0 * q_stride, *K = k + (int64_t)c0 * k_stride;
        const double *V = v + (int64_t)c0 * v_stride;
        double acc = 0.0;
        for (int i = 0; i < L; ++i) {
            acc += g[(int64_t)(c0 + i) * bg_stride];
            gam[i] = acc;
        }
        /* A, strictly lower triangular */
        for (int i = 0; i < L; ++i)
            for (int j = 0; j < L; ++j) {
                double val = 0.0;
                if (j < i) {
                    double kk = 0.0;
                    for (int d = 0; d < dk; ++d) kk += K[i * k_stride + d] * K[j * k_stride + d];
                    val = beta[(int64_t)(c0 + i) * bg_stride] * exp(gam[i] - gam[j]) * kk;
                }
                A[i * C + j] = val;
            }
        /* Tm = (I + A)^{-1}: row i of (I + A) Tm = I gives
         * Tm[i][:] = e_i - sum_{j<i} A[i][j] Tm[j][:] */
        for (int i = 0; i < L; ++i)
            for (int c = 0; c < L; ++c) {
                double val = (i == c) ? 1.0 : 0.0;
                for (int j = 0; j < i; ++j) val -= A[i * C + j] * Tm[j * C + c];
                Tm[i * C + c] = val;
            }
        /* W = Tm diag(beta e^gam) K ; U = Tm diag(beta) V */
        for (int i = 0; i < L; ++i) {
            for (int d = 0; d < dk; ++d) {
                double s = 0.0;
                for (int j = 0; j < L; ++j)
                    s += Tm[i * C + j] * beta[(int64_t)(c0 + j) * bg_stride] * exp(gam[j]) *
                         K[j * k_stride + d];
                W[(int64_t)i * dk + d] = s;
            }
            for (int e = 0; e < dv; ++e) {
                double s = 0.0;
                for (int j = 0; j < L; ++j)
                    s += Tm[i * C + j] * beta[(int64_t)(c0 + j) * bg_stride] * V[j * v_stride + e];
                U[(int64_t)i * dv + e] = s;
            }
        }
        /* Vn = U - W H */
        for (int i = 0; i < L; ++i)
            for (int e = 0; e < dv; ++e) {
                double s = U[(int64_t)i * dv + e];
                for (int d = 0; d < dk; ++d) s -= W[(int64_t)i * dk + d] * H[(int64_t)d * dv + e];
                Vn[(int64_t)i * dv + e] = s;
            }
        /* outputs: inter-chunk part through H, intra-chunk part through Vn */
        for (int i = 0; i < L; ++i) {
            double qk[256 + 1];
            double *qkp = (L <= 256) ? qk : (double *)malloc((size_t)L * sizeof(double));
            for (int j = 0; j <= i; ++j) {
                double s = 0.0;
                for (int d = 0; d < dk; ++d) s += Q[i * q_stride + d] * K[j * k_stride + d];
                qkp[j] = s * exp(gam[i] - gam[j]);
            }
            double eg = exp(gam[i]);
            for (int e = 0; e < dv; ++e) {
                double s = 0.0;
                for (int d = 0; d < dk; ++d) s += Q[i * q_stride + d] * H[(int64_t)d * dv + e];
                s *= eg;
                for (int j = 0; j <= i; ++j) s += qkp[j] * Vn[(int64_t)j * dv + e];
                o[(int64_t)(c0 + i) * o_stride + e] = scale * s;
            }
            if (qkp != qk) free(qkp);
        }
        /* state hand-off to the next chunk */
        double eL = exp(gam[L - 1]);
        for (int d = 0; d < dk; ++d)
            for (int e = 0; e < dv; ++e) {
                double s = eL * H[(int64_t)d * dv + e];
                for (int j = 0; j < L; ++j)
                    s += exp(gam[L - 1] - gam[j]) * K[j * k_stride + d] * Vn[(int64_t)j * dv + e];
                H[(int64_t)d * dv + e] = s;
            }
    }
    if (hT) memcpy(hT, H, (size_t)dk * dv * sizeof(double));
    free(H); free(gam); free(A); free(Tm); free(W); free(U); free(Vn);
}

void gdn_oracle_gated_rmsnorm(int64_t nrows, int dv,
                              const double *o, int64_t o_stride,
                              const float *gate, int64_t gate_stride,
                              const float *norm_w, double eps, int act,
                              double *y, int64_t y_stride) {
    for (int64_t r = 0; r < nrows; ++r) {
        const double *orow = o + r * o_stride;
        double ms = 0.0;
        for (int j = 0; j < dv; ++j) ms += orow[j] * orow[j];
        ms /= dv;
        double inv = 1.0 / sqrt(ms + eps);
        for (int j = 0; j < dv; ++j) {
            double rn = gdn_oracle_round_act((double)norm_w[j] * orow[j] * inv, act);
            y[r * y_stride + j] = rn * silu((double)gate[r * gate_stride + j]);
        }
    }
}

int gdn_oracle_forward(const gdn_oracle_problem *p, int head_begin, int head_end) {
    if (!p || p->n_seq < 0 || p->Hk <= 0 || p->Hv <= 0 || p->Hv % p->Hk != 0 ||
        p->dk <= 0 || p->dv <= 0 || p->conv_width <= 0 || head_begin < 0 ||
        head_end > p->Hv || head_begin > head_end)
        return -1;
    const int64_t *s = p->seq_start;
    const int64_t ntok = s[p->n_seq];
    const int G = p->Hv / p->Hk;
    const int dk = p->dk, dv = p->dv, W = p->conv_width;
    const int64_t ch_qk = (int64_t)p->Hk * dk, ch_v = (int64_t)p->Hv * dv;
    double *qh = (double *)malloc((size_t)(ntok > 0 ? ntok : 1) * dk * sizeof(double));
    double *kh = (double *)malloc((size_t)(ntok > 0 ? ntok : 1) * dk * sizeof(double));
    double *vh = (double *)malloc((size_t)(ntok > 0 ? ntok : 1) * dv * sizeof(double));
    double *ob = (double *)malloc((size_t)(ntok > 0 ? ntok : 1) * dv * sizeof(double));
    double *beta = (double *)malloc((size_t)(ntok > 0 ? ntok : 1) * sizeof(double));
    double *g = (double *)malloc((size_t)(ntok > 0 ? ntok : 1) * sizeof(double));
    double *h0 = (double *)malloc((size_t)dk * dv * sizeof(double));
    double *hT = (double *)malloc((size_t)dk * dv * sizeof(double));
    int rc = 0;
    if (!qh || !kh || !vh || !ob || !beta || !g || !h0 || !hT) { rc = -1; goto done; }
    for (int h = head_begin; h < head_end; ++h) {
        const int hk = h / G;   /* GQA: v head h reads q/k head h / G */
        /* conv_prefix rows hold all channels, q|k|v */
        const float *pre = p->conv_prefix;
        const int64_t ch = 2 * ch_qk + ch_v;
        gdn_oracle_conv_silu_prefix(p->n_seq, s, dk, W, p->q_raw + (int64_t)hk * dk, ch_qk,
                                    p->conv_w + (int64_t)hk * dk * W,
                                    pre ? pre + (int64_t)hk * dk : NULL, ch, qh);
        gdn_oracle_conv_silu_prefix(p->n_seq, s, dk, W, p->k_raw + (int64_t)hk * dk, ch_qk,
                                    p->conv_w + (ch_qk + (int64_t)hk * dk) * W,
                                    pre ? pre + ch_qk + (int64_t)hk * dk : NULL, ch, kh);
        gdn_oracle_conv_silu_prefix(p->n_seq, s, dv, W, p->v_raw + (int64_t)h * dv, ch_v,
                                    p->conv_w + (2 * ch_qk + (int64_t)h * dv) * W,
                                    pre ? pre + 2 * ch_qk + (int64_t)h * dv : NULL, ch, vh);
        gdn_oracle_l2norm(ntok, 1, dk, p->l2_eps, qh);
        gdn_oracle_l2norm(ntok, 1, dk, p->l2_eps, kh);
        for (int64_t t = 0; t < ntok; ++t)
            beta_decay_one(p->a[t * p->Hv + h], p->b[t * p->Hv + h], p->A_log[h],
                           p->dt_bias[h], &beta[t], &g[t]);
        for (int n = 0; n < p->n_seq; ++n) {
            const int64_t t0 = s[n];
            const int T = (int)(s[n + 1] - s[n]);
            const double *h0p = NULL;
            if (p->initial_state) {
                const float *src = p->initial_state + ((int64_t)n * p->Hv + h) * dk * dv;
                for (int64_t i = 0; i < (int64_t)dk * dv; ++i) h0[i] = src[i];
                h0p = h0;
            }
            if (p->chunked > 0)
                gdn_oracle_delta_rule_chunked(T, dk, dv, p->chunked, qh + t0 * dk, dk,
                                              kh + t0 * dk, dk, vh + t0 * dv, dv,
                                              beta + t0, g + t0, 1, p->scale, h0p,
                                              ob + t0 * dv, dv, hT);
            else
                gdn_oracle_delta_rule(T, dk, dv, qh + t0 * dk, dk, kh + t0 * dk, dk,
                                      vh + t0 * dv, dv, beta + t0, g + t0, 1, p->scale,
                                      h0p, ob + t0 * dv, dv, hT);
            if (p->final_state)
                memcpy(p->final_state + ((int64_t)n * p->Hv + h) * dk * dv, hT,
                       (size_t)dk * dv * sizeof(double));
        }
        gdn_oracle_gated_rmsnorm(ntok, dv, ob, dv, p->gate + (int64_t)h * dv, ch_v,
                                 p->norm_w, p->norm_eps, p->act,
                                 p->out + (int64_t)h * dv, ch_v);
    }
done:
    free(qh); free(kh); free(vh); free(ob); free(beta); free(g); free(h0); free(hT);
    return rc;
}

/* One decode step per sequence: the window of the last W-1 raw inputs (from
 * the conv cache) and the new token gives the token's conv outputs (the conv
 * definition applied to a W-row sequence, last row kept); then the same
 * L2 norm, beta / decay, one step of the token-by-token rule from the carried
 * state, and the gated RMSNorm as in the forward. */
int gdn_oracle_decode(const gdn_oracle_decode_problem *p) {
    if (!p || p->n_seq < 0 || p->Hk <= 0 || p->Hv <= 0 || p->Hv % p->Hk != 0 || p->dk <= 0 ||
        p->dv <= 0 || p->conv_width < 2)
        return -1;
    const int W = p->conv_width, dk = p->dk, dv = p->dv, G = p->Hv / p->Hk;
    const int ch_qk = p->Hk * dk, ch_v = p->Hv * dv, ch = 2 * ch_qk + ch_v;
    float *win = (float *)malloc(sizeof(float) * (size_t)W * ch);
    double *y = (double *)malloc(sizeof(double) * (size_t)W * ch);
    double *o = (double *)malloc(sizeof(double) * (size_t)dv);
    double *h0 = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *hT = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    int rc = 0;
    if (!win || !y || !o || !h0 || !hT) { rc = -1; goto done; }
    const int64_t s[2] = {0, W};
    for (int n = 0; n < p->n_seq; ++n) {
        /* window rows 0..W-2: cached raw inputs (oldest first); row W-1: the token */
        const float *cs = p->conv_state + (int64_t)n * ch * (W - 1);
        for (int r = 0; r < W - 1; ++r)
            for (int c = 0; c < ch; ++c) win[(int64_t)r * ch + c] = cs[(int64_t)c * (W - 1) + r];
        float *last = win + (int64_t)(W - 1) * ch;
        for (int c = 0; c < ch_qk; ++c) {
            last[c] = p->q_raw[(int64_t)n * ch_qk + c];
            last[ch_qk + c] = p->k_raw[(int64_t)n * ch_qk + c];
        }
        for (int c = 0; c < ch_v; ++c) last[2 * ch_qk + c] = p->v_raw[(int64_t)n * ch_v + c];
        gdn_oracle_conv_silu(1, s, ch, W, win, ch, p->conv_w, y);
        double *yq = y + (int64_t)(W - 1) * ch, *yk = yq + ch_qk, *yv = yq + 2 * ch_qk;
        gdn_oracle_l2norm(1, p->Hk, dk, p->l2_eps, yq);
        gdn_oracle_l2norm(1, p->Hk, dk, p->l2_eps, yk);
        /* the cache advanced by this token */
        double *cso = p->conv_state_out + (int64_t)n * ch * (W - 1);
        for (int r = 0; r < W - 1; ++r)
            for (int c = 0; c < ch; ++c) cso[(int64_t)c * (W - 1) + r] = win[(int64_t)(r + 1) * ch + c];
        for (int h = 0; h < p->Hv; ++h) {
            const int hk = h / G;
            double beta, g;
            beta_decay_one(p->a[(int64_t)n * p->Hv + h], p->b[(int64_t)n * p->Hv + h], p->A_log[h],
                           p->dt_bias[h], &beta, &g);
            memcpy(h0, p->state + ((int64_t)n * p->Hv + h) * dk * dv, (size_t)dk * dv * sizeof(double));
            gdn_oracle_delta_rule(1, dk, dv, yq + (int64_t)hk * dk, dk, yk + (int64_t)hk * dk, dk,
                                  yv + (int64_t)h * dv, dv, &beta, &g, 1, p->scale, h0, o, dv, hT);
            memcpy(p->state_out + ((int64_t)n * p->Hv + h) * dk * dv, hT, (size_t)dk * dv * sizeof(double));
            gdn_oracle_gated_rmsnorm(1, dv, o, dv, p->gate + (int64_t)n * ch_v + (int64_t)h * dv, ch_v,
                                     p->norm_w, p->norm_eps, p->act,
                                     p->out + ((int64_t)n * p->Hv + h) * dv, dv);
        }
    }
done:
    free(win); free(y); free(o); free(h0); free(hT);
    return rc;
}
