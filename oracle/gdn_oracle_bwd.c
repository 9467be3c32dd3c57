/*
 * gdn_oracle_bwd.c -- CPU oracle of the backward of the GDN layer core.
 *
 * TEST INFRASTRUCTURE ONLY (see gdn_oracle.h for who may call it). The pages
 * define the forward only. The backward here is the exact derivative (reverse
 * mode, chain rule, double precision) of the forward's real-valued function;
 * the rounding of the RMSNorm result to the activation dtype is taken as the
 * identity. It follows the forward's steps in reverse:
 *
 *   gated RMSNorm  y = w * o * rstd * silu(gate),  rstd = (mean(o^2) + eps)^-1/2
 *   delta rule     S' = e^g S_{t-1},  u = S' k,  r = beta (v - u),
 *                  S_t = S' + r k^T,  o_t = scale S_t q_t
 *                  (the token form of S_t = e^g S_{t-1}(I - beta k k^T) + beta v k^T)
 *   beta / decay   beta = sigmoid(b),  g = -exp(A_log) softplus(a + dt_bias)
 *   L2 norm        x_n = x (sum x^2 + eps)^-1/2 per head
 *   conv + SiLU    y_t = silu(z_t),  z_t = sum_i w_i x_{t-W+1+i}  (zero before the start)
 *   GQA            v head h reads q/k head h / (Hv/Hk), so a q/k head collects
 *                  the gradients of its v heads.
 *
 * States are recomputed from checkpoints every kCkpt tokens of the exact
 * forward recurrence (a memory strategy only: the values are those of the
 * token loop). Pinned by finite differences of gdn_oracle_forward in
 * tests/test_oracle_backward.py.
 */
#include "gdn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { kCkpt = 64 };

static double sig(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu_b(double x) { return x * sig(x); }
/* d/dz silu(z) = sigma(z) (1 + z (1 - sigma(z))) */
static double dsilu(double z) {
    double s = sig(z);
    return s * (1.0 + z * (1.0 - s));
}
static double softplus_b(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

/* z[t][c] = sum_i w[c][i] x[t-W+1+i][c] (zero before the sequence start) */
static void conv_pre(int n_seq, const int64_t *s, int nch, int W, const float *x, int64_t xs,
                     const float *w, double *z) {
    for (int n = 0; n < n_seq; ++n)
        for (int64_t t = s[n]; t < s[n + 1]; ++t)
            for (int c = 0; c < nch; ++c) {
                double acc = 0.0;
                for (int i = 0; i < W; ++i) {
                    int64_t tau = t - (W - 1) + i;
                    if (tau < s[n]) continue;
                    acc += (double)w[(int64_t)c * W + i] * (double)x[tau * xs + c];
                }
                z[t * nch + c] = acc;
            }
}

/* Reverse of conv_pre for dz [ntok][nch]: dx (row stride dxs) and dw [nch][W]
 * receive dz's contributions (both overwritten). */
static void conv_bwd(int n_seq, const int64_t *s, int nch, int W, const float *x, int64_t xs,
                     const float *w, const double *dz, double *dx, int64_t dxs, double *dw) {
    for (int64_t t = 0; t < s[n_seq]; ++t)
        for (int c = 0; c < nch; ++c) dx[t * dxs + c] = 0.0;
    for (int c = 0; c < nch; ++c)
        for (int i = 0; i < W; ++i) dw[(int64_t)c * W + i] = 0.0;
    for (int n = 0; n < n_seq; ++n)
        for (int64_t t = s[n]; t < s[n + 1]; ++t)
            for (int c = 0; c < nch; ++c) {
                double g = dz[t * nch + c];
                for (int i = 0; i < W; ++i) {
                    int64_t tau = t - (W - 1) + i;
                    if (tau < s[n]) continue;
                    dx[tau * dxs + c] += (double)w[(int64_t)c * W + i] * g;
                    dw[(int64_t)c * W + i] += g * (double)x[tau * xs + c];
                }
            }
}

/* One step of the delta rule on S (dv x dk, S[j*dk+i]) in place. */
static void step(int dk, int dv, double *S, const double *k, const double *v, double beta, double g,
                 double *u) {
    double e = exp(g);
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += e * S[(int64_t)j * dk + i] * k[i];
        u[j] = acc;
    }
    for (int j = 0; j < dv; ++j) {
        double r = beta * (v[j] - u[j]);
        for (int i = 0; i < dk; ++i) {
            double *s = &S[(int64_t)j * dk + i];
            *s = e * *s + r * k[i];
        }
    }
}

/*
 * Reverse pass of the delta rule for one (sequence, v head) of T tokens.
 * q, k [T][dk], v [T][dv], beta, g [T] (dense rows); h0 [dk][dv] (S^T) or NULL.
 * do_ [T][dv]: gradient of o; dhT [dk][dv] (S^T layout) or NULL.
 * Outputs (overwritten): dq, dk_ [T][dk], dv_ [T][dv], dbeta, dg [T], dh0 [dk][dv].
 */
static int delta_rule_bwd(int T, int dk, int dv, const double *q, const double *k, const double *v,
                          const double *beta, const double *g, double scale, const double *h0,
                          const double *do_, const double *dhT, double *dq, double *dk_,
                          double *dv_, double *dbeta, double *dg, double *dh0) {
    const int64_t SZ = (int64_t)dk * dv;
    const int nck = (T + kCkpt - 1) / kCkpt;
    /* ck[c]: S before token c*kCkpt; blk[m]: S after token c*kCkpt+m (m < kCkpt) */
    double *ck = (double *)malloc(sizeof(double) * (size_t)(nck > 0 ? nck : 1) * SZ);
    double *blk = (double *)malloc(sizeof(double) * (size_t)kCkpt * SZ);
    double *S = (double *)calloc((size_t)SZ, sizeof(double));
    double *dS = (double *)calloc((size_t)SZ, sizeof(double));
    double *Sp = (double *)malloc(sizeof(double) * (size_t)SZ);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    double *dr = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!ck || !blk || !S || !dS || !Sp || !u || !dr) {
        free(ck); free(blk); free(S); free(dS); free(Sp); free(u); free(dr);
        return -1;
    }
    if (h0)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[(int64_t)j * dk + i] = h0[(int64_t)i * dv + j];
    for (int t = 0; t < T; ++t) {
        if (t % kCkpt == 0) memcpy(ck + (int64_t)(t / kCkpt) * SZ, S, sizeof(double) * (size_t)SZ);
        step(dk, dv, S, k + (int64_t)t * dk, v + (int64_t)t * dv, beta[t], g[t], u);
    }
    if (dhT)
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) dS[(int64_t)j * dk + i] = dhT[(int64_t)i * dv + j];
    for (int c = nck - 1; c >= 0; --c) {
        const int t0 = c * kCkpt, t1 = (t0 + kCkpt < T) ? t0 + kCkpt : T;
        memcpy(S, ck + (int64_t)c * SZ, sizeof(double) * (size_t)SZ);
        for (int t = t0; t < t1; ++t) {
            step(dk, dv, S, k + (int64_t)t * dk, v + (int64_t)t * dv, beta[t], g[t], u);
            memcpy(blk + (int64_t)(t - t0) * SZ, S, sizeof(double) * (size_t)SZ);
        }
        for (int t = t1 - 1; t >= t0; --t) {
            const double *St = blk + (int64_t)(t - t0) * SZ;
            const double *Sprev = (t > t0) ? blk + (int64_t)(t - t0 - 1) * SZ : ck + (int64_t)c * SZ;
            const double *qt = q + (int64_t)t * dk, *kt = k + (int64_t)t * dk, *vt = v + (int64_t)t * dv;
            const double *dot = do_ + (int64_t)t * dv;
            const double e = exp(g[t]), bt = beta[t];
            /* o_t = scale S_t q_t */
            for (int j = 0; j < dv; ++j)
                for (int i = 0; i < dk; ++i) dS[(int64_t)j * dk + i] += scale * dot[j] * qt[i];
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += St[(int64_t)j * dk + i] * dot[j];
                dq[(int64_t)t * dk + i] = scale * acc;
            }
            /* S' = e^g S_{t-1}, u = S' k, r = beta (v - u) */
            for (int64_t x = 0; x < SZ; ++x) Sp[x] = e * Sprev[x];
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += Sp[(int64_t)j * dk + i] * kt[i];
                u[j] = acc;
            }
            /* S_t = S' + r k^T */
            double db = 0.0;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += dS[(int64_t)j * dk + i] * kt[i];
                dr[j] = acc;
                db += acc * (vt[j] - u[j]);
                dv_[(int64_t)t * dv + j] = bt * acc;
            }
            dbeta[t] = db;
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += dS[(int64_t)j * dk + i] * bt * (vt[j] - u[j]);
                dk_[(int64_t)t * dk + i] = acc;
            }
            /* through u: du = -beta dr; dS' = dS + du k^T; dk += S'^T du */
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += Sp[(int64_t)j * dk + i] * (-bt * dr[j]);
                dk_[(int64_t)t * dk + i] += acc;
            }
            for (int j = 0; j < dv; ++j)
                for (int i = 0; i < dk; ++i) dS[(int64_t)j * dk + i] += -bt * dr[j] * kt[i];
            /* S' = e^g S_{t-1}: dg = <dS', S'>, dS_{t-1} = e^g dS' */
            double gg = 0.0;
            for (int64_t x = 0; x < SZ; ++x) gg += dS[x] * Sp[x];
            dg[t] = gg;
            for (int64_t x = 0; x < SZ; ++x) dS[x] *= e;
        }
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) dh0[(int64_t)i * dv + j] = dS[(int64_t)j * dk + i];
    free(ck); free(blk); free(S); free(dS); free(Sp); free(u); free(dr);
    return 0;
}

/*
 * Whole core backward for the q/k heads [hk_begin, hk_end) and their v heads.
 * Each call owns the outputs of its heads (q/k channels of its q/k heads, v
 * channels and a, b, gate columns of its v heads, their conv_w rows, A_log /
 * dt_bias entries, initial-state slices and dnorm_w rows), so calls over
 * disjoint head ranges may run concurrently.
 */
int gdn_oracle_backward(const gdn_oracle_bwd_problem *p, int hk_begin, int hk_end) {
    if (!p || p->n_seq < 0 || p->Hk <= 0 || p->Hv <= 0 || p->Hv % p->Hk != 0 || p->dk <= 0 ||
        p->dv <= 0 || p->conv_width <= 0 || hk_begin < 0 || hk_end > p->Hk || hk_begin > hk_end)
        return -1;
    const int64_t *s = p->seq_start;
    const int64_t ntok = s[p->n_seq], nt1 = ntok > 0 ? ntok : 1;
    const int G = p->Hv / p->Hk, dk = p->dk, dv = p->dv, W = p->conv_width;
    const int64_t ch_qk = (int64_t)p->Hk * dk, ch_v = (int64_t)p->Hv * dv;
    const int64_t SZ = (int64_t)dk * dv;
    double *zq = (double *)malloc(sizeof(double) * (size_t)nt1 * dk);
    double *zk = (double *)malloc(sizeof(double) * (size_t)nt1 * dk);
    double *qn = (double *)malloc(sizeof(double) * (size_t)nt1 * dk);
    double *kn = (double *)malloc(sizeof(double) * (size_t)nt1 * dk);
    double *rq = (double *)malloc(sizeof(double) * (size_t)nt1);
    double *rk = (double *)malloc(sizeof(double) * (size_t)nt1);
    double *dqn = (double *)calloc((size_t)nt1 * dk, sizeof(double));
    double *dkn = (double *)calloc((size_t)nt1 * dk, sizeof(double));
    double *zv = (double *)malloc(sizeof(double) * (size_t)nt1 * dv);
    double *vv = (double *)malloc(sizeof(double) * (size_t)nt1 * dv);
    double *o = (double *)malloc(sizeof(double) * (size_t)nt1 * dv);
    double *dO = (double *)malloc(sizeof(double) * (size_t)nt1 * dv);
    double *dvv = (double *)malloc(sizeof(double) * (size_t)nt1 * dv);
    double *beta = (double *)malloc(sizeof(double) * (size_t)nt1);
    double *g = (double *)malloc(sizeof(double) * (size_t)nt1);
    double *dbeta = (double *)malloc(sizeof(double) * (size_t)nt1);
    double *dg = (double *)malloc(sizeof(double) * (size_t)nt1);
    double *dqh = (double *)malloc(sizeof(double) * (size_t)nt1 * dk);
    double *dkh = (double *)malloc(sizeof(double) * (size_t)nt1 * dk);
    double *dz = (double *)malloc(sizeof(double) * (size_t)nt1 * (dk > dv ? dk : dv));
    double *h0 = (double *)malloc(sizeof(double) * (size_t)SZ);
    double *dhT = (double *)malloc(sizeof(double) * (size_t)SZ);
    double *dh0 = (double *)malloc(sizeof(double) * (size_t)SZ);
    double *hT = (double *)malloc(sizeof(double) * (size_t)SZ);
    int rc = 0;
    if (!zq || !zk || !qn || !kn || !rq || !rk || !dqn || !dkn || !zv || !vv || !o || !dO || !dvv ||
        !beta || !g || !dbeta || !dg || !dqh || !dkh || !dz || !h0 || !dhT || !dh0 || !hT) {
        rc = -1;
        goto done;
    }
    for (int hk = hk_begin; hk < hk_end; ++hk) {
        /* forward of the q / k head: z = conv, y = silu(z), x_n = y rho */
        conv_pre(p->n_seq, s, dk, W, p->q_raw + (int64_t)hk * dk, ch_qk, p->conv_w + (int64_t)hk * dk * W, zq);
        conv_pre(p->n_seq, s, dk, W, p->k_raw + (int64_t)hk * dk, ch_qk,
                 p->conv_w + (ch_qk + (int64_t)hk * dk) * W, zk);
        for (int64_t t = 0; t < ntok; ++t) {
            double sq = 0.0, sk = 0.0;
            for (int i = 0; i < dk; ++i) {
                double a = silu_b(zq[t * dk + i]), b = silu_b(zk[t * dk + i]);
                qn[t * dk + i] = a;
                kn[t * dk + i] = b;
                sq += a * a;
                sk += b * b;
            }
            rq[t] = 1.0 / sqrt(sq + p->l2_eps);
            rk[t] = 1.0 / sqrt(sk + p->l2_eps);
            for (int i = 0; i < dk; ++i) {
                qn[t * dk + i] *= rq[t];
                kn[t * dk + i] *= rk[t];
            }
        }
        memset(dqn, 0, sizeof(double) * (size_t)nt1 * dk);
        memset(dkn, 0, sizeof(double) * (size_t)nt1 * dk);
        for (int h = hk * G; h < (hk + 1) * G; ++h) {
            const int64_t vc0 = 2 * ch_qk + (int64_t)h * dv;   /* first conv_w row of v head h */
            conv_pre(p->n_seq, s, dv, W, p->v_raw + (int64_t)h * dv, ch_v, p->conv_w + vc0 * W, zv);
            for (int64_t x = 0; x < ntok * dv; ++x) vv[x] = silu_b(zv[x]);
            const double eA = exp((double)p->A_log[h]);
            for (int64_t t = 0; t < ntok; ++t) {
                beta[t] = sig((double)p->b[t * p->Hv + h]);
                g[t] = -eA * softplus_b((double)p->a[t * p->Hv + h] + (double)p->dt_bias[h]);
            }
            /* forward outputs o of every sequence (the token loop) */
            for (int n = 0; n < p->n_seq; ++n) {
                const int64_t t0 = s[n];
                const double *h0p = NULL;
                if (p->initial_state) {
                    const float *src = p->initial_state + ((int64_t)n * p->Hv + h) * SZ;
                    for (int64_t x = 0; x < SZ; ++x) h0[x] = src[x];
                    h0p = h0;
                }
                gdn_oracle_delta_rule((int)(s[n + 1] - t0), dk, dv, qn + t0 * dk, dk, kn + t0 * dk, dk,
                                      vv + t0 * dv, dv, beta + t0, g + t0, 1, p->scale, h0p,
                                      o + t0 * dv, dv, hT);
            }
            /* gated RMSNorm backward, per token */
            double *dnw = p->dnorm_w + (int64_t)h * dv;
            for (int j = 0; j < dv; ++j) dnw[j] = 0.0;
            for (int64_t t = 0; t < ntok; ++t) {
                const double *ot = o + t * dv;
                double ms = 0.0;
                for (int j = 0; j < dv; ++j) ms += ot[j] * ot[j];
                const double rstd = 1.0 / sqrt(ms / dv + p->norm_eps);
                double dnn = 0.0;
                for (int j = 0; j < dv; ++j) {
                    const double gt = (double)p->gate[t * ch_v + (int64_t)h * dv + j];
                    const double dy = (double)p->grad_out[(t * p->Hv + h) * dv + j];
                    const double nj = ot[j] * rstd, wj = (double)p->norm_w[j];
                    p->dgate[t * ch_v + (int64_t)h * dv + j] = dy * wj * nj * dsilu(gt);
                    const double dr = dy * silu_b(gt);
                    dnw[j] += dr * nj;
                    dO[t * dv + j] = dr * wj;          /* d(normalised o), for now */
                    dnn += dr * wj * nj;
                }
                for (int j = 0; j < dv; ++j) dO[t * dv + j] = rstd * (dO[t * dv + j] - ot[j] * rstd * dnn / dv);
            }
            /* delta rule backward, per sequence */
            for (int n = 0; n < p->n_seq; ++n) {
                const int64_t t0 = s[n];
                const int T = (int)(s[n + 1] - t0);
                const double *h0p = NULL, *dhp = NULL;
                if (p->initial_state) {
                    const float *src = p->initial_state + ((int64_t)n * p->Hv + h) * SZ;
                    for (int64_t x = 0; x < SZ; ++x) h0[x] = src[x];
                    h0p = h0;
                }
                if (p->grad_final) {
                    const float *src = p->grad_final + ((int64_t)n * p->Hv + h) * SZ;
                    for (int64_t x = 0; x < SZ; ++x) dhT[x] = src[x];
                    dhp = dhT;
                }
                if (delta_rule_bwd(T, dk, dv, qn + t0 * dk, kn + t0 * dk, vv + t0 * dv, beta + t0, g + t0,
                                   p->scale, h0p, dO + t0 * dv, dhp, dqh + t0 * dk, dkh + t0 * dk,
                                   dvv + t0 * dv, dbeta + t0, dg + t0, dh0) != 0) {
                    rc = -1;
                    goto done;
                }
                if (p->dinitial_state)
                    memcpy(p->dinitial_state + ((int64_t)n * p->Hv + h) * SZ, dh0, sizeof(double) * (size_t)SZ);
            }
            for (int64_t x = 0; x < ntok * dk; ++x) {
                dqn[x] += dqh[x];
                dkn[x] += dkh[x];
            }
            /* beta = sigmoid(b); g = -e^A softplus(a + dt_bias) */
            double dA = 0.0, ddt = 0.0;
            for (int64_t t = 0; t < ntok; ++t) {
                const double x = (double)p->a[t * p->Hv + h] + (double)p->dt_bias[h];
                p->db[t * p->Hv + h] = dbeta[t] * beta[t] * (1.0 - beta[t]);
                const double dx = dg[t] * (-eA) * sig(x);
                p->da[t * p->Hv + h] = dx;
                ddt += dx;
                dA += dg[t] * g[t];
            }
            p->dA_log[h] = dA;
            p->ddt_bias[h] = ddt;
            /* v = silu(conv(v_raw)) */
            for (int64_t x = 0; x < ntok * dv; ++x) dz[x] = dvv[x] * dsilu(zv[x]);
            conv_bwd(p->n_seq, s, dv, W, p->v_raw + (int64_t)h * dv, ch_v, p->conv_w + vc0 * W, dz,
                     p->dv_raw + (int64_t)h * dv, ch_v, p->dconv_w + vc0 * W);
        }
        /* L2 norm, SiLU and conv of the q / k head */
        for (int pass = 0; pass < 2; ++pass) {
            const double *xn = pass ? kn : qn, *dxn = pass ? dkn : dqn, *z = pass ? zk : zq;
            const double *rho = pass ? rk : rq;
            for (int64_t t = 0; t < ntok; ++t) {
                double dot = 0.0;
                for (int i = 0; i < dk; ++i) dot += xn[t * dk + i] * dxn[t * dk + i];
                for (int i = 0; i < dk; ++i)
                    dz[t * dk + i] = rho[t] * (dxn[t * dk + i] - xn[t * dk + i] * dot) * dsilu(z[t * dk + i]);
            }
            const int64_t c0 = (pass ? ch_qk : 0) + (int64_t)hk * dk;
            conv_bwd(p->n_seq, s, dk, W, (pass ? p->k_raw : p->q_raw) + (int64_t)hk * dk, ch_qk,
                     p->conv_w + c0 * W, dz, (pass ? p->dk_raw : p->dq_raw) + (int64_t)hk * dk, ch_qk,
                     p->dconv_w + c0 * W);
        }
    }
done:
    free(zq); free(zk); free(qn); free(kn); free(rq); free(rk); free(dqn); free(dkn); free(zv); free(vv);
    free(o); free(dO); free(dvv); free(beta); free(g); free(dbeta); free(dg); free(dqh); free(dkh);
    free(dz); free(h0); free(dhT); free(dh0); free(hT);
    return rc;
}
