// gdn_chunk_simt.cu -- chunked gated delta rule on CUDA cores in fp32.
//
// Precision-first kernel (fp32 FFMA throughout): it serves fp32 activations,
// where the tensor cores' tf32 mantissa is too short for a 1e-4 relative
// error bound. One CTA owns one (sequence, v head, dv tile of NV columns) and
// walks the sequence chunk by chunk (64 tokens) with its slice of the state,
// H = S^T [dk][NV], resident in shared memory in fp32.
//
// Per chunk, with gam_i the in-chunk cumulative decay (inclusive):
//   A   = strict_lower( beta_i exp(gam_i - gam_j) k_i.k_j )
//   P   = lower( exp(gam_i - gam_j) q_i.k_j )
//   Tm  = (I + A)^{-1}                       (blocked forward substitution)
//   R   = diag(beta) (V - diag(exp(gam)) K H)
//   Vn  = Tm R                               (new values, "u" of the delta rule)
//   O   = diag(exp(gam)) Q H + P Vn
//   H  <- exp(gam_L) H + (diag(exp(gam_L - gam)) K)^T Vn
// Only exp of differences gam_i - gam_j (j <= i) or of gam itself is ever
// formed, so no factor exceeds 1. Tokens past the end of a short chunk get
// beta = 0 and zero rows, which makes them contribute nothing.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int DS = 32;              // dk slice staged in shared memory
constexpr int LDA = kChunk + 1;     // padded row length of 64x64 tiles
constexpr int LDS = DS + 1;

template <int NV>
size_t simt_smem_floats(int dk) {
    return (size_t)dk * NV + 3 * kChunk * LDA + 2 * kChunk * LDS + 3 * kChunk * NV + 4 * kChunk;
}

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) chunk_simt_kernel(const Problem p, int ntiles) {
    using S = typename Inter<T>::S;   // storage of q, k, v, o
    using GT = typename Inter<T>::G;  // in-chunk cumulative decay
    constexpr int NB = NV / 16;     // output columns per thread
    extern __shared__ float sm[];
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv;
    const int G = Hv / d.Hk;
    int bid = blockIdx.x;
    const int tile = bid % ntiles;
    bid /= ntiles;
    const int j = bid % Hv;
    const int n = bid / Hv;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    const int64_t seq0 = p.cu ? (int64_t)p.cu[n] : (int64_t)n * d.T;
    const int64_t seq1 = p.cu ? (int64_t)p.cu[n + 1] : seq0 + d.T;
    const int hk = j / G;
    const int v0 = tile * NV;

    float *Hs = sm;                          // [dk][NV]
    float *As = Hs + (size_t)dk * NV;        // [64][LDA]
    float *Ts = As + kChunk * LDA;           // [64][LDA]
    float *Ps = Ts + kChunk * LDA;           // [64][LDA]
    float *Ks = Ps + kChunk * LDA;           // [64][LDS]
    float *Qs = Ks + kChunk * LDS;           // [64][LDS]
    float *Vs = Qs + kChunk * LDS;           // [64][NV]   V tile, then R
    float *Vn = Vs + kChunk * NV;            // [64][NV]
    float *Xs = Vn + kChunk * NV;            // [64][NV]   scratch of the solve
    float *bet = Xs + kChunk * NV;           // [64]
    GT *gam = (GT *)(bet + 2 * kChunk);      // [64] (8-byte aligned)

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const S *kq = (const S *)p.k + (int64_t)hk * p.ntok * dk;
    const S *qq = (const S *)p.q + (int64_t)hk * p.ntok * dk;
    const S *vv = (const S *)p.v + (int64_t)j * p.ntok * dv;
    const GT *gw = (const GT *)p.gamma + (int64_t)j * p.ntok;
    const float *bw = p.beta + (int64_t)j * p.ntok;
    S *o = (S *)p.o;
    // q/k: fp32, or fp16 hi + lo planes for 2-byte activations
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    auto load_qk = [&](const S *base, int64_t idx) -> float {
        if (sizeof(S) == 4) return to_f<S>(base[idx]);
        return to_f<S>(base[idx]) + to_f<S>(base[idx + plane]);
    };

    // state slice
    const size_t sbase = ((size_t)n * Hv + j) * dk * dv;
    for (int idx = tid; idx < dk * NV; idx += kThreads) {
        const int r = idx / NV, c = idx - r * NV;
        Hs[idx] = p.h0 ? p.h0[sbase + (size_t)r * dv + v0 + c] : 0.f;
    }

    for (int64_t tok0 = seq0; tok0 < seq1; tok0 += kChunk) {
        const int L = (seq1 - tok0) < kChunk ? (int)(seq1 - tok0) : kChunk;
        __syncthreads();
        // ---- decay, beta, V tile
        if (tid < kChunk) {
            const int i = tid < L ? tid : L - 1;
            gam[tid] = gw[tok0 + i];
            bet[tid] = tid < L ? bw[tok0 + i] : 0.f;
        }
        for (int idx = tid; idx < kChunk * NV; idx += kThreads) {
            const int i = idx / NV, c = idx - i * NV;
            Vs[idx] = i < L ? to_f<S>(vv[(tok0 + i) * dv + v0 + c]) : 0.f;
        }
        // ---- K K^T, Q K^T, K H, Q H over dk slices
        float kk[4][4], qk[4][4], kh[4][NB], qh[4][NB];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
#pragma unroll
            for (int b = 0; b < 4; ++b) kk[a][b] = qk[a][b] = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b) kh[a][b] = qh[a][b] = 0.f;
        }
        for (int d0 = 0; d0 < dk; d0 += DS) {
            __syncthreads();
            for (int idx = tid; idx < kChunk * DS; idx += kThreads) {
                const int i = idx / DS, c = idx - i * DS;
                const bool ok = i < L && d0 + c < dk;
                Ks[i * LDS + c] = ok ? load_qk(kq, (tok0 + i) * dk + d0 + c) : 0.f;
                Qs[i * LDS + c] = ok ? load_qk(qq, (tok0 + i) * dk + d0 + c) : 0.f;
            }
            __syncthreads();
            const int dn = min(DS, dk - d0);
            for (int c = 0; c < dn; ++c) {
                float ki[4], qi[4], kj[4], hv[NB];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    ki[a] = Ks[(ty + 16 * a) * LDS + c];
                    qi[a] = Qs[(ty + 16 * a) * LDS + c];
                    kj[a] = Ks[(tx + 16 * a) * LDS + c];
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) hv[b] = Hs[(d0 + c) * NV + tx + 16 * b];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        kk[a][b] = fmaf(ki[a], kj[b], kk[a][b]);
                        qk[a][b] = fmaf(qi[a], kj[b], qk[a][b]);
                    }
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        kh[a][b] = fmaf(ki[a], hv[b], kh[a][b]);
                        qh[a][b] = fmaf(qi[a], hv[b], qh[a][b]);
                    }
                }
            }
        }
        // ---- decay masks
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = ty + 16 * a;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int jj = tx + 16 * b;
                const float dec = jj <= i ? expf((float)(gam[i] - gam[jj])) : 0.f;
                As[i * LDA + jj] = jj < i ? bet[i] * dec * kk[a][b] : 0.f;
                Ps[i * LDA + jj] = dec * qk[a][b];
                Ts[i * LDA + jj] = 0.f;
            }
        }
        // R = beta (V - e^gam K H) ; keep e^gam Q H in registers
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = ty + 16 * a;
            const float eg = expf((float)gam[i]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const int c = tx + 16 * b;
                Vs[i * NV + c] = bet[i] * (Vs[i * NV + c] - eg * kh[a][b]);
                qh[a][b] *= eg;
            }
        }
        __syncthreads();
        // ---- Tm = (I + A)^{-1}: 16x16 diagonal blocks by forward substitution
        if (tid < kChunk) {
            const int blk = tid >> 4, c = tid & 15, o0 = blk * 16;
            for (int r = c; r < 16; ++r) {
                float val = (r == c) ? 1.f : 0.f;
                for (int m = c; m < r; ++m)
                    val -= As[(o0 + r) * LDA + o0 + m] * Ts[(o0 + m) * LDA + o0 + c];
                Ts[(o0 + r) * LDA + o0 + c] = val;
            }
        }
        __syncthreads();
        // off-diagonal blocks, one block diagonal at a time:
        // T[bi][bj] = -T[bi][bi] * sum_{m=bj}^{bi-1} A[bi][m] T[m][bj]
        for (int dd = 1; dd < 4; ++dd) {
            const int npairs = 4 - dd;
            for (int e = tid; e < npairs * 256; e += kThreads) {
                const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
                const int bj = pr, bi = pr + dd;
                float x = 0.f;
                for (int m = bj * 16; m < bi * 16; ++m)
                    x += As[(bi * 16 + r) * LDA + m] * Ts[m * LDA + bj * 16 + c];
                Xs[pr * 256 + r * 16 + c] = x;
            }
            __syncthreads();
            for (int e = tid; e < npairs * 256; e += kThreads) {
                const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
                const int bj = pr, bi = pr + dd;
                float t = 0.f;
                for (int m = 0; m < 16; ++m)
                    t += Ts[(bi * 16 + r) * LDA + bi * 16 + m] * Xs[pr * 256 + m * 16 + c];
                Ts[(bi * 16 + r) * LDA + bj * 16 + c] = -t;
            }
            __syncthreads();
        }
        // ---- Vn = Tm R
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = ty + 16 * a;
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = 0.f;
            for (int m = 0; m <= i; ++m) {
                const float t = Ts[i * LDA + m];
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[b] = fmaf(t, Vs[m * NV + tx + 16 * b], acc[b]);
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) Vn[i * NV + tx + 16 * b] = acc[b];
        }
        __syncthreads();
        // ---- O = e^gam Q H + P Vn
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = ty + 16 * a;
            for (int m = 0; m <= i; ++m) {
                const float pv = Ps[i * LDA + m];
#pragma unroll
                for (int b = 0; b < NB; ++b) qh[a][b] = fmaf(pv, Vn[m * NV + tx + 16 * b], qh[a][b]);
            }
            if (i < L) {
                S *orow = o + ((tok0 + i) * Hv + j) * (int64_t)dv + v0;
#pragma unroll
                for (int b = 0; b < NB; ++b) orow[tx + 16 * b] = from_f<S>(qh[a][b] * d.scale);
            }
        }
        // ---- H <- e^{gam_L} H + (e^{gam_L - gam} K)^T Vn, over dk slices
        const float eL = expf((float)gam[kChunk - 1]);
        for (int d0 = 0; d0 < dk; d0 += DS) {
            __syncthreads();
            for (int idx = tid; idx < kChunk * DS; idx += kThreads) {
                const int i = idx / DS, c = idx - i * DS;
                const bool ok = i < L && d0 + c < dk;
                Ks[i * LDS + c] = ok ? load_qk(kq, (tok0 + i) * dk + d0 + c) *
                                           expf((float)(gam[kChunk - 1] - gam[i])) : 0.f;
            }
            __syncthreads();
            const int dn = min(DS, dk - d0);
            for (int r = ty; r < dn; r += 16) {
                float acc[NB];
#pragma unroll
                for (int b = 0; b < NB; ++b) acc[b] = 0.f;
                for (int i = 0; i < kChunk; ++i) {
                    const float kv = Ks[i * LDS + r];
#pragma unroll
                    for (int b = 0; b < NB; ++b) acc[b] = fmaf(kv, Vn[i * NV + tx + 16 * b], acc[b]);
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float *h = &Hs[(d0 + r) * NV + tx + 16 * b];
                    *h = fmaf(eL, *h, acc[b]);
                }
            }
        }
    }
    __syncthreads();
    if (p.hT) {
        for (int idx = tid; idx < dk * NV; idx += kThreads) {
            const int r = idx / NV, c = idx - r * NV;
            p.hT[sbase + (size_t)r * dv + v0 + c] = Hs[idx];
        }
    }
}

template <typename T, int NV>
cudaError_t launch_nv(const Problem &p, cudaStream_t s) {
    const int ntiles = p.d.dv / NV;
    const size_t bytes = simt_smem_floats<NV>(p.d.dk) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<T, NV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)p.d.N * p.d.Hv * ntiles;
    if (blocks == 0) return cudaSuccess;
    chunk_simt_kernel<T, NV><<<(unsigned)blocks, kThreads, bytes, s>>>(p, ntiles);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const Problem &p, cudaStream_t s) {
    const int dk = p.d.dk, dv = p.d.dv;
    if (dv >= 64 && dk <= 256) return launch_nv<T, 64>(p, s);
    if (dv >= 32) return launch_nv<T, 32>(p, s);
    return launch_nv<T, 16>(p, s);
}

}  // namespace

cudaError_t launch_chunk_simt(const Problem &p, cudaStream_t s) {
    switch (p.d.dtype) {
    case GDN_F32: return launch_t<float>(p, s);
    case GDN_BF16: return launch_t<__nv_bfloat16>(p, s);
    default: return launch_t<__half>(p, s);
    }
}

}  // namespace gdn
