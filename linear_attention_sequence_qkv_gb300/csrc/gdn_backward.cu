// gdn_backward.cu -- backward of the GDN layer core on CUDA cores in fp32.
//
// The pages define the forward (the gated delta rule S_t = e^{g_t} S_{t-1}
// (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t, with the
// "GDN Elementwise Fusion" pre- and post-GDR steps); this file computes the
// gradient of sum(grad_out * out) + sum(grad_final * final_state) with respect
// to every input, the RMSNorm rounding taken as the identity. The forward's
// prologue runs first (gdn_api.cu) and leaves q, k, v, beta and the in-chunk
// cumulative decay gam in the workspace.
//
// Chunk form (H = S^T, dk x dv; L the chunk's last valid token, E_ij =
// e^{gam_i - gam_j}, Kd = diag(e^{gam_L - gam}) K, Ak = strict_lower(E . K K^T),
// A = diag(beta) Ak, T = (I + A)^{-1}, Pm = lower(E . Q K^T)):
//   R0 = diag(beta)(V - diag(e^gam) K H0),  Vn = T R0,
//   O  = scale (diag(e^gam) Q H0 + Pm Vn),  H1 = e^{gam_L} H0 + Kd^T Vn.
// Reverse, with dO' = scale dO and dH1 the gradient of the chunk's end state:
//   dVn = Pm^T dO' + Kd dH1,  dR0 = T^T dVn,  dV = beta dR0,
//   dH0 = e^{gam_L} dH1 + Q^T diag(e^gam) dO' - K^T diag(beta e^gam) dR0,
//   dA  = -dR0 Vn^T (strictly lower),  dPm = dO' Vn^T (lower),
//   dQ  = diag(e^gam) dO' H0^T + (dPm . E) K,
//   dK  = (dPm . E)^T Q + F K + F^T K - diag(beta e^gam) dR0 H0^T + diag(e^{gam_L - gam}) Vn dH1^T,
//         F = dA . beta_i E (strictly lower),
//   dbeta_i = dR0_i . V_i - e^{gam_i} K_i . (dR0 H0^T)_i + sum_j dA_ij Ak_ij,
//   dgam_i from every e^{...} factor, and dg = reverse cumulative sum of dgam.
//
// Kernels, in launch order. Serial over the chunks of a sequence (one CTA per
// (sequence, v head, dv tile)): states (H0 of every chunk and Vn) and chain_bwd
// (dH1 of every chunk and dR0, chunks in reverse). Everything else runs over all
// chunks or tokens in parallel: mats (T, Pm, Ak), out (O), rms_bwd (gated
// RMSNorm: dgate, dO'), dterms (Pm^T dO' and Q^T diag(e^gam) dO', the parts of
// the reverse step that do not depend on dH), chunk_grad (dq, dk per v head,
// dbeta, dg), prologue_bwd (L2 norm, SiLU, beta / decay), conv_bwd (input
// gradients and per-block weight sums) and sum_kernel (fixed-order sums of the
// partials: dnorm_w, dconv_w, ddt_bias, dA_log). Every sum has a fixed order,
// so results are run-to-run identical.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int DS = 32;              // dk slice staged in shared memory
constexpr int LDA = kChunk + 1;     // padded row length of 64x64 tiles
constexpr int LDS = DS + 1;
constexpr int kC2 = kChunk * kChunk;

__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float dsilu(float z) {
    const float s = sigm(z);
    return s * (1.0f + z * (1.0f - s));
}

// q / k of the forward's workspace: fp32, or fp16 hi + lo planes
template <typename S>
__device__ __forceinline__ float load_qk(const S *base, int64_t idx, int64_t plane) {
    if (sizeof(S) == 4) return to_f<S>(base[idx]);
    return to_f<S>(base[idx]) + to_f<S>(base[idx + plane]);
}

// flattened token t -> (batch row b, position tau) of the strided inputs
__device__ __forceinline__ void tok_pos(const gdn_desc &d, int64_t t, int64_t &b, int64_t &tau) {
    b = d.T > 0 ? t / d.T : 0;
    tau = t - b * d.T;
}

// sequence [s0, s1) holding flattened token t
__device__ __forceinline__ void seq_of(const gdn_desc &d, const int32_t *cu, int64_t t, int64_t &s0,
                                       int64_t &s1) {
    if (cu == nullptr) {
        s0 = (t / d.T) * d.T;
        s1 = s0 + d.T;
        return;
    }
    int lo = 0, hi = d.N;   // cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    s0 = cu[lo];
    s1 = cu[lo + 1];
}

// ------------------------------------------------------------ gated RMSNorm
// One warp per (token, v head) row, NE columns per lane. Forward:
// y = w * o * rstd * silu(gate). Reads o (fp32, [Hv][ntok][dv], from out_kernel),
// writes dgate, dO' = scale * dL/do over o, and the warp's partial sums of dnorm_w.
template <typename T, typename GTy, typename WT, int NE>
__global__ void __launch_bounds__(kThreads) rms_bwd_kernel(const BwdProblem bp, int64_t rows, int64_t nwarps) {
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dv = d.dv, Hv = d.Hv;
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    float accw[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) accw[e] = 0.f;
    for (int64_t r = w; r < rows; r += nwarps) {
        const int64_t t = r / Hv;
        const int h = (int)(r - t * Hv);
        int64_t b, tau;
        tok_pos(d, t, b, tau);
        float *orow = bp.dO + ((int64_t)h * p.ntok + t) * dv;   // o in, dO' out (same row)
        const GTy *grow = (const GTy *)p.gate + b * d.gate_stride_b + tau * d.gate_stride_t + (int64_t)h * dv;
        const T *dyrow = (const T *)bp.grad_out + r * dv;
        float o[NE], dn[NE], nn[NE];
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int c = lane + 32 * e;
            o[e] = c < dv ? orow[c] : 0.f;
            ss = fmaf(o[e], o[e], ss);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float rstd = 1.0f / sqrtf(ss / dv + d.norm_eps);
        float dot = 0.f;
        GTy *dgrow = (GTy *)bp.dgate + r * dv;
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int c = lane + 32 * e;
            nn[e] = o[e] * rstd;
            dn[e] = 0.f;
            if (c < dv) {
                const float g = to_f<GTy>(grow[c]), dy = to_f<T>(dyrow[c]), wc = to_f<WT>(((const WT *)p.norm_w)[c]);
                const float sg = sigm(g);
                dgrow[c] = from_f<GTy>(dy * wc * nn[e] * (sg * (1.0f + g * (1.0f - sg))));
                const float dr = dy * g * sg;
                accw[e] = fmaf(dr, nn[e], accw[e]);
                dn[e] = dr * wc;
                dot = fmaf(dn[e], nn[e], dot);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        float *drow = orow;
        const float k = d.scale * rstd, m = dot / dv;
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int c = lane + 32 * e;
            if (c < dv) drow[c] = k * (dn[e] - nn[e] * m);
        }
    }
    if (w < nwarps) {
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int c = lane + 32 * e;
            if (c < dv) bp.pnorm[w * dv + c] = accw[e];
        }
    }
}

constexpr int LDK = 68;             // row of a 64-column slice (float4-aligned rows)
constexpr int DK = 64;              // dk slice of the 4x4-tiled kernels

// acc[x][y] += a[x] * b[y]
__device__ __forceinline__ void fma4x4(float (&acc)[4][4], const float (&a)[4], const float4 b) {
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        acc[x][0] = fmaf(a[x], b.x, acc[x][0]);
        acc[x][1] = fmaf(a[x], b.y, acc[x][1]);
        acc[x][2] = fmaf(a[x], b.z, acc[x][2]);
        acc[x][3] = fmaf(a[x], b.w, acc[x][3]);
    }
}
__device__ __forceinline__ void fma4x4(float (&acc)[4][4], const float4 a, const float4 b) {
    const float av[4] = {a.x, a.y, a.z, a.w};
    fma4x4(acc, av, b);
}
__device__ __forceinline__ void zero4x4(float (&acc)[4][4]) {
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
}
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

// ------------------------------------------------------------ chunk matrices
// One CTA per (chunk slot, v head): K K^T and Q K^T over dk slices, the decay
// masks, and T = (I + A)^{-1} by forward substitution on 16 x 16 diagonal blocks
// then block diagonals. Writes [T, Pm, Ak] of the chunk.
size_t mats_smem_bytes() { return sizeof(float) * (2 * kChunk * LDA + 2 * kChunk * LDS + 3 * 256); }

template <typename T>
__global__ void __launch_bounds__(kThreads) mats_kernel(const BwdProblem bp) {
    using S = typename Inter<T>::S;
    using GT = typename Inter<T>::G;
    __shared__ GT gam[kChunk];
    __shared__ float bet[kChunk];
    extern __shared__ float sm[];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dk = d.dk, Hv = d.Hv;
    const int j = blockIdx.y;
    const int64_t slot = blockIdx.x;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    ChunkLoc loc;
    if (!locate_chunk(slot, p.cu, p.chunk_off, d.N, d.T, loc)) return;
    const int64_t tok0 = loc.tok0;
    const int L = loc.len;
    const int hk = j / (Hv / d.Hk);
    float *As = sm;                           // [64][LDA]
    float *Ts = As + kChunk * LDA;            // [64][LDA]
    float *Ks = Ts + kChunk * LDA;            // [64][LDS]
    float *Qs = Ks + kChunk * LDS;            // [64][LDS]
    float *Xs = Qs + kChunk * LDS;            // [3][16][16]
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const S *kq = (const S *)p.k + (int64_t)hk * p.ntok * dk;
    const S *qq = (const S *)p.q + (int64_t)hk * p.ntok * dk;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    float *mats = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2;
    if (tid < kChunk) {
        const int i = tid < L ? tid : L - 1;
        gam[tid] = ((const GT *)p.gamma)[(int64_t)j * p.ntok + tok0 + i];
        bet[tid] = tid < L ? p.beta[(int64_t)j * p.ntok + tok0 + i] : 0.f;
    }
    float kk[4][4], qk[4][4];
    zero4x4(kk);
    zero4x4(qk);
    for (int d0 = 0; d0 < dk; d0 += DS) {
        __syncthreads();
        for (int idx = tid; idx < kChunk * DS; idx += kThreads) {
            const int i = idx / DS, c = idx - i * DS;
            const bool ok = i < L && d0 + c < dk;
            Ks[i * LDS + c] = ok ? load_qk(kq, (tok0 + i) * dk + d0 + c, plane) : 0.f;
            Qs[i * LDS + c] = ok ? load_qk(qq, (tok0 + i) * dk + d0 + c, plane) : 0.f;
        }
        __syncthreads();
        const int dn = min(DS, dk - d0);
        for (int c = 0; c < dn; ++c) {
            float ki[4], qi[4], kj[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                ki[a] = Ks[(ty + 16 * a) * LDS + c];
                qi[a] = Qs[(ty + 16 * a) * LDS + c];
                kj[a] = Ks[(tx + 16 * a) * LDS + c];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    kk[a][b] = fmaf(ki[a], kj[b], kk[a][b]);
                    qk[a][b] = fmaf(qi[a], kj[b], qk[a][b]);
                }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = ty + 16 * a;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int m = tx + 16 * b;
            const float dec = m <= i ? expf((float)(gam[i] - gam[m])) : 0.f;
            const float ak = m < i ? dec * kk[a][b] : 0.f;
            mats[kC2 + i * kChunk + m] = dec * qk[a][b];
            mats[2 * kC2 + i * kChunk + m] = ak;
            As[i * LDA + m] = bet[i] * ak;
            Ts[i * LDA + m] = 0.f;
        }
    }
    __syncthreads();
    // diagonal 16 x 16 blocks: column c of block b by forward substitution
    if (tid < kChunk) {
        const int o0 = (tid >> 4) * 16, c = tid & 15;
        for (int r = c; r < 16; ++r) {
            float val = (r == c) ? 1.f : 0.f;
            for (int m = c; m < r; ++m) val -= As[(o0 + r) * LDA + o0 + m] * Ts[(o0 + m) * LDA + o0 + c];
            Ts[(o0 + r) * LDA + o0 + c] = val;
        }
    }
    __syncthreads();
    // block (bi, bj), bi > bj, one block diagonal at a time:
    // T[bi][bj] = -T[bi][bi] sum_{m in blocks bj .. bi-1} A[bi][m] T[m][bj]
    for (int dd = 1; dd < 4; ++dd) {
        const int npairs = 4 - dd;
        for (int e = tid; e < npairs * 256; e += kThreads) {
            const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int bj = pr, bi = pr + dd;
            float x = 0.f;
            for (int m = bj * 16; m < bi * 16; ++m) x += As[(bi * 16 + r) * LDA + m] * Ts[m * LDA + bj * 16 + c];
            Xs[pr * 256 + r * 16 + c] = x;
        }
        __syncthreads();
        for (int e = tid; e < npairs * 256; e += kThreads) {
            const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int bj = pr, bi = pr + dd;
            float t = 0.f;
            for (int m = 0; m < 16; ++m) t += Ts[(bi * 16 + r) * LDA + bi * 16 + m] * Xs[pr * 256 + m * 16 + c];
            Ts[(bi * 16 + r) * LDA + bj * 16 + c] = -t;
        }
        __syncthreads();
    }
    for (int idx = tid; idx < kC2; idx += kThreads) mats[idx] = Ts[(idx / kChunk) * LDA + (idx % kChunk)];
}

// ------------------------------------------------------------ outputs
// One CTA per (chunk slot, v head): O = scale (diag(e^gam) Q H0 + Pm Vn) in fp32,
// [Hv][ntok][dv] (the RMSNorm backward's input), 64 dv columns at a time.
size_t out_smem_bytes() { return sizeof(float) * (kChunk * LDA + kChunk * LDK + 2 * kChunk * 64); }

template <typename T>
__global__ void __launch_bounds__(kThreads) out_kernel(const BwdProblem bp) {
    using S = typename Inter<T>::S;
    using GT = typename Inter<T>::G;
    __shared__ GT gam[kChunk];
    extern __shared__ float sm[];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv;
    const int j = blockIdx.y;
    const int64_t slot = blockIdx.x;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    ChunkLoc loc;
    if (!locate_chunk(slot, p.cu, p.chunk_off, d.N, d.T, loc)) return;
    const int64_t tok0 = loc.tok0;
    const int L = loc.len;
    const int hk = j / (Hv / d.Hk);
    float *Ps = sm;                            // [64][LDA]
    float *Qs = Ps + kChunk * LDA;             // [64][LDK]
    float *Hs = Qs + kChunk * LDK;             // [64][64] rows of H0, 64 columns
    float *Vs = Hs + kChunk * 64;              // [64][64] Vn
    const int tid = threadIdx.x, ci = tid & 15, ti = tid >> 4;
    const S *qq = (const S *)p.q + (int64_t)hk * p.ntok * dk;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const float *mats = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2;
    const float *H0 = bp.h0 + ((size_t)slot * Hv + j) * dk * dv;
    if (tid < kChunk) {
        const int i = tid < L ? tid : L - 1;
        gam[tid] = ((const GT *)p.gamma)[(int64_t)j * p.ntok + tok0 + i];
    }
#pragma unroll 8
    for (int idx = tid; idx < kC2; idx += kThreads) Ps[(idx / kChunk) * LDA + (idx % kChunk)] = mats[kC2 + idx];
    float acc[4][4], a[4];
    for (int c0 = 0; c0 < dv; c0 += 64) {
        zero4x4(acc);
        for (int d0 = 0; d0 < dk; d0 += DK) {
            __syncthreads();
#pragma unroll 8
            for (int idx = tid; idx < kChunk * DK; idx += kThreads) {
                const int i = idx / DK, c = idx - i * DK;
                Qs[i * LDK + c] = (i < L && d0 + c < dk) ? load_qk(qq, (tok0 + i) * dk + d0 + c, plane) : 0.f;
                Hs[idx] = (d0 + i < dk && c0 + c < dv) ? H0[(size_t)(d0 + i) * dv + c0 + c] : 0.f;
            }
            __syncthreads();
            const int dn = min(DK, dk - d0);
            for (int c = 0; c < dn; ++c) {
#pragma unroll
                for (int x = 0; x < 4; ++x) a[x] = Qs[(ti + 16 * x) * LDK + c];
                fma4x4(acc, a, ld4(Hs + c * 64 + 4 * ci));
            }
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float eg = expf((float)gam[ti + 16 * x]);
#pragma unroll
            for (int y = 0; y < 4; ++y) acc[x][y] *= eg;
        }
        __syncthreads();
#pragma unroll 8
        for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
            const int i = idx >> 6, c = idx & 63;
            Vs[idx] = (i < L && c0 + c < dv) ? bp.vn[((size_t)j * p.ntok + tok0 + i) * dv + c0 + c] : 0.f;
        }
        __syncthreads();
        for (int m = 0; m < kChunk; ++m) {
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = Ps[(ti + 16 * x) * LDA + m];
            fma4x4(acc, a, ld4(Vs + m * 64 + 4 * ci));
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = ti + 16 * x;
            if (i < L && c0 + 4 * ci < dv)
                st4(bp.dO + ((size_t)j * p.ntok + tok0 + i) * dv + c0 + 4 * ci, d.scale * acc[x][0],
                    d.scale * acc[x][1], d.scale * acc[x][2], d.scale * acc[x][3]);
        }
    }
}

// ------------------------------------------------------------ dO' terms
// One CTA per (chunk slot, v head): the parts of the reverse step that do not
// depend on the carried gradient, W = Pm^T dO' ([Hv][ntok][dv]) and
// U = Q^T diag(e^gam) dO' ([slot][Hv][dk][dv]).
size_t dterms_smem_bytes() { return sizeof(float) * (kChunk * LDA + kChunk * 64 + kChunk * LDK); }

template <typename T>
__global__ void __launch_bounds__(kThreads) dterms_kernel(const BwdProblem bp) {
    using S = typename Inter<T>::S;
    using GT = typename Inter<T>::G;
    __shared__ GT gam[kChunk];
    extern __shared__ float sm[];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv;
    const int j = blockIdx.y;
    const int64_t slot = blockIdx.x;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    ChunkLoc loc;
    if (!locate_chunk(slot, p.cu, p.chunk_off, d.N, d.T, loc)) return;
    const int64_t tok0 = loc.tok0;
    const int L = loc.len;
    const int hk = j / (Hv / d.Hk);
    float *Ps = sm;                            // [64][LDA]
    float *Os = Ps + kChunk * LDA;             // [64][64] dO' tile
    float *Qs = Os + kChunk * 64;              // [64][LDK] e^gam Q slice
    const int tid = threadIdx.x, ci = tid & 15, ti = tid >> 4;
    const S *qq = (const S *)p.q + (int64_t)hk * p.ntok * dk;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const float *mats = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2;
    float *U = bp.uq + ((size_t)slot * Hv + j) * dk * dv;
    if (tid < kChunk) {
        const int i = tid < L ? tid : L - 1;
        gam[tid] = ((const GT *)p.gamma)[(int64_t)j * p.ntok + tok0 + i];
    }
#pragma unroll 8
    for (int idx = tid; idx < kC2; idx += kThreads) Ps[(idx / kChunk) * LDA + (idx % kChunk)] = mats[kC2 + idx];
    float acc[4][4], a[4];
    for (int c0 = 0; c0 < dv; c0 += 64) {
        __syncthreads();
#pragma unroll 8
        for (int idx = tid; idx < kChunk * 64; idx += kThreads) {
            const int i = idx >> 6, c = idx & 63;
            Os[idx] = (i < L && c0 + c < dv) ? bp.dO[((size_t)j * p.ntok + tok0 + i) * dv + c0 + c] : 0.f;
        }
        __syncthreads();
        // W = Pm^T dO'
        zero4x4(acc);
        for (int m = 0; m < kChunk; ++m) {
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = Ps[m * LDA + ti + 16 * x];
            fma4x4(acc, a, ld4(Os + m * 64 + 4 * ci));
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = ti + 16 * x;
            if (i < L && c0 + 4 * ci < dv)
                st4(bp.wv + ((size_t)j * p.ntok + tok0 + i) * dv + c0 + 4 * ci, acc[x][0], acc[x][1], acc[x][2],
                    acc[x][3]);
        }
        // U = (e^gam Q)^T dO' over dk slices
        for (int d0 = 0; d0 < dk; d0 += DK) {
            __syncthreads();
#pragma unroll 8
            for (int idx = tid; idx < kChunk * DK; idx += kThreads) {
                const int i = idx / DK, c = idx - i * DK;
                Qs[i * LDK + c] = (i < L && d0 + c < dk)
                                      ? load_qk(qq, (tok0 + i) * dk + d0 + c, plane) * expf((float)gam[i])
                                      : 0.f;
            }
            __syncthreads();
            zero4x4(acc);
            for (int i = 0; i < kChunk; ++i) {
                fma4x4(acc, ld4(Qs + i * LDK + 4 * ti), ld4(Os + i * 64 + 4 * ci));
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int r = d0 + 4 * ti + x;
                if (r < dk && c0 + 4 * ci < dv)
                    st4(U + (size_t)r * dv + c0 + 4 * ci, acc[x][0], acc[x][1], acc[x][2], acc[x][3]);
            }
        }
    }
}

// ------------------------------------------------------------ serial kernels
// One CTA of 4 * NV threads per (sequence, v head, dv tile of NV columns).
// Each chunk step loads the chunk's K block once (64 x dk, fp32 in shared
// memory, every load of a thread in flight together) and folds the per-row
// decay factors into the accumulators or the other operand. Thread (ti, ci)
// owns rows ti + 16x of token tiles, rows 64s + 4ti + x of the state, and
// columns 4ci + y, x, y < 4.
template <int NV>
size_t serial_smem_bytes(int dk) {
    return sizeof(double) * kChunk +
           sizeof(float) * (2 * kChunk + (size_t)dk * NV + kChunk * LDA + (size_t)kChunk * (dk + 4) + 2 * kChunk * NV);
}

// Kc[i][d] = k of token i (rows i < L, zeros after), fp32, row length dk + 4
template <typename S, int NT>
__device__ __forceinline__ void load_k_block(float *Kc, const S *kq, int64_t tok0, int L, int dk, int64_t plane,
                                             int tid) {
    const int ldk = dk + 4;
    if (sizeof(S) == 2) {
        const int groups = kChunk * dk / 8;            // 8 halves = 16 bytes per plane
#pragma unroll 8
        for (int g = tid; g < groups; g += NT) {
            const int i = g / (dk / 8), c = (g - i * (dk / 8)) * 8;
            float v[8];
            if (i < L) {
                const int64_t e = (tok0 + i) * dk + c;
                const uint4 hi = *reinterpret_cast<const uint4 *>(kq + e);
                const uint4 lo = *reinterpret_cast<const uint4 *>(kq + e + plane);
                float h[8], l[8];
                unpack16<S>(hi, h);
                unpack16<S>(lo, l);
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = h[u] + l[u];
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = 0.f;
            }
            st4(Kc + i * ldk + c, v[0], v[1], v[2], v[3]);
            st4(Kc + i * ldk + c + 4, v[4], v[5], v[6], v[7]);
        }
    } else {
        const int groups = kChunk * dk / 4;
#pragma unroll 8
        for (int g = tid; g < groups; g += NT) {
            const int i = g / (dk / 4), c = (g - i * (dk / 4)) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < L) v = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(kq) + (tok0 + i) * dk + c);
            *reinterpret_cast<float4 *>(Kc + i * ldk + c) = v;
        }
    }
}

// Forward recompute: per chunk store H0, Vn = T diag(beta)(V - diag(e^gam) K H0)
// (to the workspace), then H <- e^{gam_L} H + K^T (diag(e^{gam_L - gam}) Vn).
template <typename T, int NV>
__global__ void __launch_bounds__(256) states_kernel(const BwdProblem bp, int ntiles) {
    using S = typename Inter<T>::S;
    using GT = typename Inter<T>::G;
    constexpr int NQ = NV / 4, NT = 4 * NV;
    extern __shared__ float sm[];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv, ldk = dk + 4;
    int bid = blockIdx.x;
    const int tile = bid % ntiles;
    bid /= ntiles;
    const int j = bid % Hv;
    const int n = bid / Hv;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    const int64_t seq0 = p.cu ? (int64_t)p.cu[n] : (int64_t)n * d.T;
    const int64_t seq1 = p.cu ? (int64_t)p.cu[n + 1] : seq0 + d.T;
    const int64_t slot0 = p.cu ? (int64_t)p.chunk_off[n] : (int64_t)n * ((d.T + kChunk - 1) / kChunk);
    const int nch = (int)((seq1 - seq0 + kChunk - 1) / kChunk);
    const int hk = j / (Hv / d.Hk);
    const int v0 = tile * NV;
    GT *gam = (GT *)sm;                        // [64]
    float *bet = (float *)(gam + kChunk);      // [64]
    float *dec = bet + kChunk;                 // [64] e^{gam_L - gam}
    float *Hs = dec + kChunk;                  // [dk][NV]
    float *Ts = Hs + (size_t)dk * NV;          // [64][LDA]
    float *Kc = Ts + kChunk * LDA;             // [64][dk + 4]
    float *Vs = Kc + (size_t)kChunk * ldk;     // [64][NV]  V, then R0
    float *Vn = Vs + kChunk * NV;              // [64][NV]  e^{gam_L - gam} Vn
    const int tid = threadIdx.x, ci = tid % NQ, ti = tid / NQ;
    const S *kq = (const S *)p.k + (int64_t)hk * p.ntok * dk;
    const S *vv = (const S *)p.v + (int64_t)j * p.ntok * dv;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const GT *gw = (const GT *)p.gamma + (int64_t)j * p.ntok;
    const float *bw = p.beta + (int64_t)j * p.ntok;
    const size_t sbase = ((size_t)n * Hv + j) * dk * dv;
    for (int idx = tid; idx < dk * NV; idx += NT) {
        const int r = idx / NV, c = idx - r * NV;
        Hs[idx] = p.h0 ? p.h0[sbase + (size_t)r * dv + v0 + c] : 0.f;
    }
    float acc[4][4], a[4];
    for (int cc = 0; cc < nch; ++cc) {
        const int64_t tok0 = seq0 + (int64_t)cc * kChunk, slot = slot0 + cc;
        const int L = (seq1 - tok0) < kChunk ? (int)(seq1 - tok0) : kChunk;
        __syncthreads();
        float *dst = bp.h0 + ((size_t)slot * Hv + j) * dk * dv + v0;
        for (int idx = tid; idx < dk * NQ; idx += NT) {
            const int r = idx / NQ, q = idx - r * NQ;
            *reinterpret_cast<float4 *>(dst + (size_t)r * dv + 4 * q) = ld4(Hs + r * NV + 4 * q);
        }
        load_k_block<S, NT>(Kc, kq, tok0, L, dk, plane, tid);
        const float *mats = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2;
#pragma unroll 4
        for (int q = tid; q < kC2 / 4; q += NT) {
            const float4 t4 = ld4(mats + 4 * q);
            const int i = q / (kChunk / 4), m = (q - i * (kChunk / 4)) * 4;
            Ts[i * LDA + m] = t4.x;
            Ts[i * LDA + m + 1] = t4.y;
            Ts[i * LDA + m + 2] = t4.z;
            Ts[i * LDA + m + 3] = t4.w;
        }
        if (tid < kChunk) {
            const int i = tid < L ? tid : L - 1;
            gam[tid] = gw[tok0 + i];
            bet[tid] = tid < L ? bw[tok0 + i] : 0.f;
        }
#pragma unroll 4
        for (int idx = tid; idx < kChunk * NV; idx += NT) {
            const int i = idx / NV, c = idx - i * NV;
            Vs[idx] = i < L ? to_f<S>(vv[(tok0 + i) * dv + v0 + c]) : 0.f;
        }
        __syncthreads();
        if (tid < kChunk) dec[tid] = expf((float)(gam[kChunk - 1] - gam[tid]));
        // ---- K H
        zero4x4(acc);
        for (int c = 0; c < dk; ++c) {
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = Kc[(ti + 16 * x) * ldk + c];
            fma4x4(acc, a, ld4(Hs + c * NV + 4 * ci));
        }
        // ---- R0 = beta (V - e^gam K H)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = ti + 16 * x;
            const float eg = expf((float)gam[i]);
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                float *v = &Vs[i * NV + 4 * ci + y];
                *v = bet[i] * (*v - eg * acc[x][y]);
            }
        }
        __syncthreads();
        // ---- Vn = T R0 (stored; kept scaled by e^{gam_L - gam} for the state step)
        zero4x4(acc);
        for (int m = 0; m < kChunk; ++m) {
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = Ts[(ti + 16 * x) * LDA + m];
            fma4x4(acc, a, ld4(Vs + m * NV + 4 * ci));
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = ti + 16 * x;
            const float s = dec[i];
            st4(Vn + i * NV + 4 * ci, s * acc[x][0], s * acc[x][1], s * acc[x][2], s * acc[x][3]);
            if (i < L)
                st4(bp.vn + ((size_t)j * p.ntok + tok0 + i) * dv + v0 + 4 * ci, acc[x][0], acc[x][1], acc[x][2],
                    acc[x][3]);
        }
        __syncthreads();
        // ---- H <- e^{gam_L} H + K^T (e^{gam_L - gam} Vn)
        const float eL = expf((float)gam[kChunk - 1]);
        for (int r0 = 0; r0 < dk; r0 += 64) {
            zero4x4(acc);
            if (r0 + 4 * ti < dk) {
                for (int i = 0; i < kChunk; ++i) fma4x4(acc, ld4(Kc + i * ldk + r0 + 4 * ti), ld4(Vn + i * NV + 4 * ci));
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    float *h = Hs + (r0 + 4 * ti + x) * NV + 4 * ci;
                    st4(h, fmaf(eL, h[0], acc[x][0]), fmaf(eL, h[1], acc[x][1]), fmaf(eL, h[2], acc[x][2]),
                        fmaf(eL, h[3], acc[x][3]));
                }
            }
        }
    }
}

// Reverse chain: chunks in reverse, carrying dH [dk][NV]; per chunk store dH1,
// dR0 = T^T (W + diag(e^{gam_L - gam}) K dH1) (to the workspace), then
// dH <- e^{gam_L} dH + U - K^T (diag(beta e^gam) dR0).
template <typename T, int NV>
__global__ void __launch_bounds__(256) chain_bwd_kernel(const BwdProblem bp, int ntiles) {
    using S = typename Inter<T>::S;
    using GT = typename Inter<T>::G;
    constexpr int NQ = NV / 4, NT = 4 * NV;
    extern __shared__ float sm[];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv, ldk = dk + 4;
    int bid = blockIdx.x;
    const int tile = bid % ntiles;
    bid /= ntiles;
    const int j = bid % Hv;
    const int n = bid / Hv;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    const int64_t seq0 = p.cu ? (int64_t)p.cu[n] : (int64_t)n * d.T;
    const int64_t seq1 = p.cu ? (int64_t)p.cu[n + 1] : seq0 + d.T;
    const int64_t slot0 = p.cu ? (int64_t)p.chunk_off[n] : (int64_t)n * ((d.T + kChunk - 1) / kChunk);
    const int nch = (int)((seq1 - seq0 + kChunk - 1) / kChunk);
    const int hk = j / (Hv / d.Hk);
    const int v0 = tile * NV;
    GT *gam = (GT *)sm;                        // [64]
    float *bet = (float *)(gam + kChunk);      // [64]
    float *dec = bet + kChunk;                 // [64] e^{gam_L - gam}
    float *dHs = dec + kChunk;                 // [dk][NV]
    float *Ts = dHs + (size_t)dk * NV;         // [64][LDA]
    float *Kc = Ts + kChunk * LDA;             // [64][dk + 4]
    float *dVs = Kc + (size_t)kChunk * ldk;    // [64][NV]  W, then dVn
    float *dRs = dVs + kChunk * NV;            // [64][NV]  beta e^gam dR0
    const int tid = threadIdx.x, ci = tid % NQ, ti = tid / NQ;
    const S *kq = (const S *)p.k + (int64_t)hk * p.ntok * dk;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const GT *gw = (const GT *)p.gamma + (int64_t)j * p.ntok;
    const float *bw = p.beta + (int64_t)j * p.ntok;
    const size_t sbase = ((size_t)n * Hv + j) * dk * dv;
    for (int idx = tid; idx < dk * NV; idx += NT) {
        const int r = idx / NV, c = idx - r * NV;
        dHs[idx] = bp.grad_final ? bp.grad_final[sbase + (size_t)r * dv + v0 + c] : 0.f;
    }
    float acc[4][4], a[4];
    for (int cc = nch - 1; cc >= 0; --cc) {
        const int64_t tok0 = seq0 + (int64_t)cc * kChunk, slot = slot0 + cc;
        const int L = (seq1 - tok0) < kChunk ? (int)(seq1 - tok0) : kChunk;
        __syncthreads();
        float *dst = bp.dh1 + ((size_t)slot * Hv + j) * dk * dv + v0;
        for (int idx = tid; idx < dk * NQ; idx += NT) {
            const int r = idx / NQ, q = idx - r * NQ;
            *reinterpret_cast<float4 *>(dst + (size_t)r * dv + 4 * q) = ld4(dHs + r * NV + 4 * q);
        }
        load_k_block<S, NT>(Kc, kq, tok0, L, dk, plane, tid);
        const float *mats = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2;
#pragma unroll 4
        for (int q = tid; q < kC2 / 4; q += NT) {
            const float4 t4 = ld4(mats + 4 * q);
            const int i = q / (kChunk / 4), m = (q - i * (kChunk / 4)) * 4;
            Ts[i * LDA + m] = t4.x;
            Ts[i * LDA + m + 1] = t4.y;
            Ts[i * LDA + m + 2] = t4.z;
            Ts[i * LDA + m + 3] = t4.w;
        }
        if (tid < kChunk) {
            const int i = tid < L ? tid : L - 1;
            gam[tid] = gw[tok0 + i];
            bet[tid] = tid < L ? bw[tok0 + i] : 0.f;
        }
#pragma unroll 4
        for (int q = tid; q < kChunk * NQ; q += NT) {
            const int i = q / NQ, c = (q - i * NQ) * 4;
            const float4 w4 = i < L ? ld4(bp.wv + ((size_t)j * p.ntok + tok0 + i) * dv + v0 + c)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(dVs + i * NV + c) = w4;
        }
        __syncthreads();
        if (tid < kChunk) dec[tid] = expf((float)(gam[kChunk - 1] - gam[tid]));
        __syncthreads();
        // ---- dVn = W + diag(e^{gam_L - gam}) K dH1
        zero4x4(acc);
        for (int c = 0; c < dk; ++c) {
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = Kc[(ti + 16 * x) * ldk + c];
            fma4x4(acc, a, ld4(dHs + c * NV + 4 * ci));
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const float s = dec[ti + 16 * x];
            float *v = dVs + (ti + 16 * x) * NV + 4 * ci;
            st4(v, fmaf(s, acc[x][0], v[0]), fmaf(s, acc[x][1], v[1]), fmaf(s, acc[x][2], v[2]),
                fmaf(s, acc[x][3], v[3]));
        }
        __syncthreads();
        // ---- dR0 = T^T dVn (stored), kept scaled by beta e^gam for the state step
        zero4x4(acc);
        for (int m = 0; m < kChunk; ++m) {
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = Ts[m * LDA + ti + 16 * x];
            fma4x4(acc, a, ld4(dVs + m * NV + 4 * ci));
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = ti + 16 * x;
            const float s = bet[i] * expf((float)gam[i]);
            st4(dRs + i * NV + 4 * ci, s * acc[x][0], s * acc[x][1], s * acc[x][2], s * acc[x][3]);
            if (i < L)
                st4(bp.dR + ((size_t)j * p.ntok + tok0 + i) * dv + v0 + 4 * ci, acc[x][0], acc[x][1], acc[x][2],
                    acc[x][3]);
        }
        __syncthreads();
        // ---- dH0 = e^{gam_L} dH1 + U - K^T (beta e^gam dR0)
        const float eL = expf((float)gam[kChunk - 1]);
        const float *U = bp.uq + ((size_t)slot * Hv + j) * dk * dv + v0;
        for (int r0 = 0; r0 < dk; r0 += 64) {
            if (r0 + 4 * ti < dk) {
                float4 u[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) u[x] = ld4(U + (size_t)(r0 + 4 * ti + x) * dv + 4 * ci);
                zero4x4(acc);
                for (int i = 0; i < kChunk; ++i) fma4x4(acc, ld4(Kc + i * ldk + r0 + 4 * ti), ld4(dRs + i * NV + 4 * ci));
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    float *h = dHs + (r0 + 4 * ti + x) * NV + 4 * ci;
                    st4(h, fmaf(eL, h[0], u[x].x - acc[x][0]), fmaf(eL, h[1], u[x].y - acc[x][1]),
                        fmaf(eL, h[2], u[x].z - acc[x][2]), fmaf(eL, h[3], u[x].w - acc[x][3]));
                }
            }
        }
    }
    __syncthreads();
    if (bp.dinit) {
        for (int idx = tid; idx < dk * NV; idx += NT) {
            const int r = idx / NV, c = idx - r * NV;
            bp.dinit[sbase + (size_t)r * dv + v0 + c] = dHs[idx];
        }
    }
}

// ------------------------------------------------------------ per-chunk gradients
// One CTA per (chunk slot, v head); thread (ti, ci) owns rows 4 ti + x and
// columns 4 ci + y of every 64 x 64 block. Phase A sums dPm = dO' Vn^T and
// dA = -dR0 Vn^T over dv; phase B, per 64-wide dk slice, forms X1 = dO' H0^T,
// X2 = dR0 H0^T and X3 = Vn dH1^T over dv and the q / k gradients of the
// slice; phase C finishes dbeta and dg. dv is staged 16 columns at a time,
// transposed (row index contiguous) so that every operand is a float4.
constexpr int kTileV = 16;

size_t grad_smem_bytes() { return sizeof(float) * (4 * kChunk * LDK + 5 * kTileV * LDK); }

template <typename T, bool XPRE>   // XPRE: X1, X2, X3 and <H0, dH1> come from chunk_x (tensor cores)
__global__ void __launch_bounds__(kThreads, 2) chunk_grad_kernel(const BwdProblem bp) {
    using S = typename Inter<T>::S;
    using GT = typename Inter<T>::G;
    __shared__ GT gam[kChunk];
    __shared__ float bet[kChunk], eg[kChunk], ed[kChunk], dbet[kChunk], dgm[kChunk], red[64];
    extern __shared__ float sm[];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv;
    const int j = blockIdx.y;
    const int64_t slot = blockIdx.x;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    ChunkLoc loc;
    if (!locate_chunk(slot, p.cu, p.chunk_off, d.N, d.T, loc)) return;
    const int64_t tok0 = loc.tok0;
    const int L = loc.len;
    const int hk = j / (Hv / d.Hk);

    float *Ps = sm;                            // [64][LDK] Pm, then Pg = dPm . E
    float *As = Ps + kChunk * LDK;             // [64][LDK] Ak, then F = dA . beta_i E
    float *Ks = As + kChunk * LDK;             // [64][LDK] k slice (token rows)
    float *Qs = Ks + kChunk * LDK;             // [64][LDK] q slice
    float *tO = Qs + kChunk * LDK;             // [16][LDK] dO'^T tile (column c: 64 token rows)
    float *tR = tO + kTileV * LDK;             // [16][LDK] dR0^T
    float *tV = tR + kTileV * LDK;             // [16][LDK] Vn^T
    float *th = tV + kTileV * LDK;             // [16][LDK] H0^T slice (column c: 64 dk rows)
    float *tdh = th + kTileV * LDK;            // [16][LDK] dH1^T slice
    float *Gs = tO;                            // [64][LDK] after phase A (aliases the tiles)

    const int tid = threadIdx.x, ci = tid & 15, ti = tid >> 4;
    const S *kq = (const S *)p.k + (int64_t)hk * p.ntok * dk;
    const S *qq = (const S *)p.q + (int64_t)hk * p.ntok * dk;
    const S *vv = (const S *)p.v + (int64_t)j * p.ntok * dv;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const float *mats = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2;
    const float *H0 = bp.h0 + ((size_t)slot * Hv + j) * dk * dv;
    const float *dH1 = bp.dh1 + ((size_t)slot * Hv + j) * dk * dv;
    const float *dOg = bp.dO + ((size_t)j * p.ntok + tok0) * dv;
    const float *dRg = bp.dR + ((size_t)j * p.ntok + tok0) * dv;
    const float *Vng = bp.vn + ((size_t)j * p.ntok + tok0) * dv;

    if (tid < kChunk) {
        const int i = tid < L ? tid : L - 1;
        gam[tid] = ((const GT *)p.gamma)[(int64_t)j * p.ntok + tok0 + i];
        bet[tid] = tid < L ? p.beta[(int64_t)j * p.ntok + tok0 + i] : 0.f;
    }
    for (int idx = tid; idx < kC2; idx += kThreads) {
        const int i = idx >> 6, m = idx & 63;
        Ps[i * LDK + m] = mats[kC2 + idx];
        As[i * LDK + m] = mats[2 * kC2 + idx];
    }
    __syncthreads();
    if (tid < kChunk) {
        eg[tid] = expf((float)gam[tid]);
        ed[tid] = expf((float)(gam[kChunk - 1] - gam[tid]));
    }
    // transposed tiles of token rows: dst[c][i] = src[i][c0 + c] (rows i < L)
    auto load_rows_t = [&](float *dst, const float *src, int c0) {
#pragma unroll 4
        for (int idx = tid; idx < kChunk * kTileV; idx += kThreads) {
            const int i = idx / kTileV, c = idx - i * kTileV;
            dst[c * LDK + i] = (i < L && c0 + c < dv) ? src[(int64_t)i * dv + c0 + c] : 0.f;
        }
    };

    // ---- phase A
    float dP[4][4], dA[4][4];
    zero4x4(dP);
    zero4x4(dA);
    float pb[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < dv; c0 += kTileV) {
        __syncthreads();
        load_rows_t(tO, dOg, c0);
        load_rows_t(tR, dRg, c0);
        load_rows_t(tV, Vng, c0);
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < kTileV; ++c) {
            const float4 vm = ld4(tV + c * LDK + 4 * ci);
            fma4x4(dP, ld4(tO + c * LDK + 4 * ti), vm);
            fma4x4(dA, ld4(tR + c * LDK + 4 * ti), vm);
        }
        // dbeta's dR0 . V: row 4 ti + x, columns ci (16 lanes per row)
        if (c0 + ci < dv) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int i = 4 * ti + x;
                if (i < L) pb[x] = fmaf(tR[ci * LDK + i], to_f<S>(vv[(tok0 + i) * dv + c0 + ci]), pb[x]);
            }
        }
    }
    // G = dPm . Pm + dA . beta_i Ak; Pg = dPm . E; F = dA . beta_i E (dA = -dR0 Vn^T)
    float rowG[4], rowA[4], pg[4][4], fg[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int i = 4 * ti + x;
        rowG[x] = rowA[x] = 0.f;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int m = 4 * ci + y;
            const float dAv = -dA[x][y];
            const float e = m <= i ? expf((float)(gam[i] - gam[m])) : 0.f;
            const float pm = Ps[i * LDK + m], ak = As[i * LDK + m];
            const float g = (m <= i ? dP[x][y] * pm : 0.f) + (m < i ? dAv * bet[i] * ak : 0.f);
            rowG[x] += g;
            if (m < i) rowA[x] = fmaf(dAv, ak, rowA[x]);
            pg[x][y] = m <= i ? dP[x][y] * e : 0.f;
            fg[x][y] = m < i ? dAv * bet[i] * e : 0.f;
            dP[x][y] = g;   // G, kept for the column sums
        }
    }
    __syncthreads();   // every thread has read Pm, Ak and the tiles
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int i = 4 * ti + x;
        st4(Ps + i * LDK + 4 * ci, pg[x][0], pg[x][1], pg[x][2], pg[x][3]);
        st4(As + i * LDK + 4 * ci, fg[x][0], fg[x][1], fg[x][2], fg[x][3]);
        st4(Gs + i * LDK + 4 * ci, dP[x][0], dP[x][1], dP[x][2], dP[x][3]);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            rowG[x] += __shfl_xor_sync(0xffffffffu, rowG[x], off);
            rowA[x] += __shfl_xor_sync(0xffffffffu, rowA[x], off);
            pb[x] += __shfl_xor_sync(0xffffffffu, pb[x], off);
        }
    }
    if (ci == 0) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            dgm[4 * ti + x] = rowG[x];
            dbet[4 * ti + x] = pb[x] + rowA[x];
        }
    }
    __syncthreads();
    if (tid < kChunk) {
        float col = 0.f;
        for (int i = 0; i < kChunk; ++i) col += Gs[i * LDK + tid];
        dgm[tid] -= col;
    }
    // ---- phase B
    float rg[4] = {0.f, 0.f, 0.f, 0.f}, rb[4] = {0.f, 0.f, 0.f, 0.f}, kap = 0.f, hd = 0.f;
    float *dqo = bp.dq + ((size_t)j * p.ntok + tok0) * dk;
    float *dko = bp.dk + ((size_t)j * p.ntok + tok0) * dk;
    const float *Xb = bp.xbuf + ((size_t)slot * Hv + j) * 3 * 64 * dk;
    for (int d0 = 0; d0 < dk; d0 += DK) {
        float X1[4][4], X2[4][4], X3[4][4];
        zero4x4(X1);
        zero4x4(X2);
        zero4x4(X3);
        if (XPRE && d0 + 4 * ci < dk) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const size_t r = (size_t)(4 * ti + x) * dk + d0 + 4 * ci;
                const float4 a = ld4(Xb + r), b = ld4(Xb + 64 * (size_t)dk + r), c = ld4(Xb + 128 * (size_t)dk + r);
                X1[x][0] = a.x; X1[x][1] = a.y; X1[x][2] = a.z; X1[x][3] = a.w;
                X2[x][0] = b.x; X2[x][1] = b.y; X2[x][2] = b.z; X2[x][3] = b.w;
                X3[x][0] = c.x; X3[x][1] = c.y; X3[x][2] = c.z; X3[x][3] = c.w;
            }
        }
        for (int c0 = 0; c0 < (XPRE ? 0 : dv); c0 += kTileV) {
            __syncthreads();
            load_rows_t(tO, dOg, c0);
            load_rows_t(tR, dRg, c0);
            load_rows_t(tV, Vng, c0);
#pragma unroll 4
            for (int idx = tid; idx < DK * kTileV; idx += kThreads) {
                const int r = idx / kTileV, c = idx - r * kTileV;
                const bool ok = d0 + r < dk && c0 + c < dv;
                th[c * LDK + r] = ok ? H0[(int64_t)(d0 + r) * dv + c0 + c] : 0.f;
                tdh[c * LDK + r] = ok ? dH1[(int64_t)(d0 + r) * dv + c0 + c] : 0.f;
            }
            __syncthreads();
#pragma unroll 4
            for (int c = 0; c < kTileV; ++c) {
                const float4 h = ld4(th + c * LDK + 4 * ci), dh = ld4(tdh + c * LDK + 4 * ci);
                fma4x4(X1, ld4(tO + c * LDK + 4 * ti), h);
                fma4x4(X2, ld4(tR + c * LDK + 4 * ti), h);
                fma4x4(X3, ld4(tV + c * LDK + 4 * ti), dh);
            }
            for (int idx = tid; idx < DK * kTileV; idx += kThreads) hd = fmaf(th[idx % kTileV * LDK + idx / kTileV],
                                                                             tdh[idx % kTileV * LDK + idx / kTileV], hd);
        }
        __syncthreads();
#pragma unroll 4
        for (int idx = tid; idx < kChunk * DK; idx += kThreads) {
            const int i = idx / DK, c = idx - i * DK;
            const bool ok = i < L && d0 + c < dk;
            Ks[i * LDK + c] = ok ? load_qk(kq, (tok0 + i) * dk + d0 + c, plane) : 0.f;
            Qs[i * LDK + c] = ok ? load_qk(qq, (tok0 + i) * dk + d0 + c, plane) : 0.f;
        }
        __syncthreads();
        // dQ = e^gam X1 + Pg K;  dK = Pg^T Q + F K + F^T K - beta e^gam X2 + e^{gam_L - gam} X3
        float gq[4][4], gk[4][4], a[4], b[4];
        zero4x4(gq);
        zero4x4(gk);
        for (int m = 0; m < kChunk; ++m) {
            const float4 km = ld4(Ks + m * LDK + 4 * ci), qm = ld4(Qs + m * LDK + 4 * ci);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                a[x] = Ps[(4 * ti + x) * LDK + m];
                b[x] = As[(4 * ti + x) * LDK + m];
            }
            fma4x4(gq, a, km);
            fma4x4(gk, b, km);
            fma4x4(gk, ld4(Ps + m * LDK + 4 * ti), qm);
            fma4x4(gk, ld4(As + m * LDK + 4 * ti), km);
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            const int i = 4 * ti + x;
            const float be = bet[i] * eg[i];
            float oq[4], ok[4];
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const int dd = 4 * ci + y;
                const float qv = Qs[i * LDK + dd], kv = Ks[i * LDK + dd];
                oq[y] = fmaf(eg[i], X1[x][y], gq[x][y]);
                ok[y] = gk[x][y] - be * X2[x][y] + ed[i] * X3[x][y];
                rg[x] += qv * eg[i] * X1[x][y] - kv * be * X2[x][y] - kv * ed[i] * X3[x][y];
                kap = fmaf(kv * ed[i], X3[x][y], kap);
                rb[x] = fmaf(-eg[i] * kv, X2[x][y], rb[x]);
            }
            if (i < L && d0 + 4 * ci < dk) {
                st4(dqo + (int64_t)i * dk + d0 + 4 * ci, oq[0], oq[1], oq[2], oq[3]);
                st4(dko + (int64_t)i * dk + d0 + 4 * ci, ok[0], ok[1], ok[2], ok[3]);
            }
        }
    }
    // ---- phase C: dbeta, dgam, then dg = reverse cumulative sum of dgam
#pragma unroll
    for (int x = 0; x < 4; ++x) {
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) {
            rg[x] += __shfl_xor_sync(0xffffffffu, rg[x], off);
            rb[x] += __shfl_xor_sync(0xffffffffu, rb[x], off);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        kap += __shfl_xor_sync(0xffffffffu, kap, off);
        hd += __shfl_xor_sync(0xffffffffu, hd, off);
    }
    __syncthreads();
    if ((tid & 31) == 0) {
        red[tid >> 5] = kap;
        red[32 + (tid >> 5)] = hd;
    }
    if (ci == 0) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            dgm[4 * ti + x] += rg[x];
            dbet[4 * ti + x] += rb[x];
        }
    }
    __syncthreads();
    if (tid == 0) {
        float ks = 0.f, hs_ = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) {
            ks += red[w];
            hs_ += red[32 + w];
        }
        if (XPRE) hs_ = bp.hdbuf[(size_t)slot * Hv + j];
        dgm[L - 1] += ks + expf((float)gam[kChunk - 1]) * hs_;
        float acc = 0.f;
        float *dbo = bp.dbeta + (size_t)j * p.ntok + tok0;
        float *dgo = bp.dgam + (size_t)j * p.ntok + tok0;
        for (int i = L - 1; i >= 0; --i) {
            acc += dgm[i];
            dgo[i] = acc;
            dbo[i] = dbet[i];
        }
    }
}

// 4 adjacent act-dtype values as fp32 and back (8- or 16-byte accesses)
template <typename T> __device__ __forceinline__ float4 ld4_act(const T *p) {
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const float4 *>(p);
    } else {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const T *h = reinterpret_cast<const T *>(&u);
        return make_float4(to_f<T>(h[0]), to_f<T>(h[1]), to_f<T>(h[2]), to_f<T>(h[3]));
    }
}
template <typename T> __device__ __forceinline__ void st4_act(T *p, float4 v) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4 *>(p) = v;
    } else {
        uint2 u;
        T *h = reinterpret_cast<T *>(&u);
        h[0] = from_f<T>(v.x); h[1] = from_f<T>(v.y); h[2] = from_f<T>(v.z); h[3] = from_f<T>(v.w);
        *reinterpret_cast<uint2 *>(p) = u;
    }
}
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {
    return make_float4(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y), fmaf(a.z, b.z, c.z), fmaf(a.w, b.w, c.w));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// ------------------------------------------------------------ prologue backward
// One 1-D grid of 256-thread CTAs in three ranges. Each item recomputes the conv
// pre-activation z of its channels and writes dz = dL/dz ([ntok][ch]):
//   * q/k: a group of dk / CPL lanes per (token, q or k head), CPL adjacent
//     channels per lane; the L2-norm backward's two sums over the head are
//     shuffle reductions within the group;
//   * v: one thread per 4 adjacent channels of a token;
//   * beta / decay: one thread per (token, v head): db, da and the per-token
//     terms of ddt_bias and dA_log.
constexpr int kProThreads = 256;

template <typename T, int N> __device__ __forceinline__ void ld_act_n(const T *p, float *out) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 f = ld4_act<T>(p + 4 * q);
            out[4 * q] = f.x; out[4 * q + 1] = f.y; out[4 * q + 2] = f.z; out[4 * q + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) out[q] = to_f<T>(p[q]);
    }
}
template <int N> __device__ __forceinline__ void ld_f32_n(const float *p, float *out) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 f = ld4(p + 4 * q);
            out[4 * q] = f.x; out[4 * q + 1] = f.y; out[4 * q + 2] = f.z; out[4 * q + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) out[q] = p[q];
    }
}

// z of N adjacent channels: x is the channel's column at flattened token t of
// sequence [s0, s1) (batch row b, position tau), w the channels' rows of conv_w
template <typename T, int N>
__device__ __forceinline__ void conv_z_n(const T *x, int64_t sb, int64_t st, int64_t b, int64_t tau, int64_t t,
                                         int64_t s0, const T *w, float *z) {
    float wv[N * kConvW];
    ld_act_n<T, N * kConvW>(w, wv);
    float xs[kConvW][N];
#pragma unroll
    for (int m = 0; m < kConvW; ++m) {
        const int64_t back = kConvW - 1 - m;
        if (t - back >= s0) {
            ld_act_n<T, N>(x + b * sb + (tau - back) * st, xs[m]);
        } else {
#pragma unroll
            for (int q = 0; q < N; ++q) xs[m][q] = 0.f;
        }
    }
#pragma unroll
    for (int q = 0; q < N; ++q) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < kConvW; ++m)
            if (t - (kConvW - 1 - m) >= s0) acc = fmaf(wv[q * kConvW + m], xs[m][q], acc);
        z[q] = acc;
    }
}

template <typename T, int CPL>
__global__ void __launch_bounds__(kProThreads) prologue_bwd_kernel(const BwdProblem bp, int64_t nA, int64_t nB) {
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    const int ch_qk = d.Hk * d.dk, ch_v = d.Hv * d.dv, ch = 2 * ch_qk + ch_v;
    const int64_t blk = blockIdx.x;
    if (blk < nA) {
        // ---- q / k: groups of lph lanes, one (token, head) each
        const int lph = d.dk / CPL;                    // lanes per head, a power of two <= 32
        const int lane = threadIdx.x & 31;
        const int64_t unit = (blk * kProThreads + threadIdx.x) / lph;
        const int i = (lane % lph) * CPL;              // first channel of this lane in the head
        const int64_t units = p.ntok * 2 * d.Hk;
        const bool act = unit < units;                 // whole groups: uniform within a group
        const int64_t t = act ? unit / (2 * d.Hk) : 0;
        const int hh = act ? (int)(unit - t * 2 * d.Hk) : 0;
        const bool isk = hh >= d.Hk;
        const int h = isk ? hh - d.Hk : hh;
        float z[CPL], y[CPL], dxn[CPL];
        float ss = 0.f;
        if (act) {
            int64_t s0, s1, b, tau;
            seq_of(d, p.cu, t, s0, s1);
            tok_pos(d, t, b, tau);
            const T *x = isk ? (const T *)p.k_raw + h * d.dk + i : (const T *)p.q_raw + h * d.dk + i;
            conv_z_n<T, CPL>(x, isk ? d.k_stride_b : d.q_stride_b, isk ? d.k_stride_t : d.q_stride_t, b, tau, t, s0,
                             (const T *)p.conv_w + (int64_t)((isk ? ch_qk : 0) + h * d.dk + i) * kConvW, z);
            const int G = d.Hv / d.Hk;
            const float *src = (isk ? bp.dk : bp.dq) + ((int64_t)h * G * p.ntok + t) * d.dk + i;
#pragma unroll
            for (int q = 0; q < CPL; ++q) dxn[q] = 0.f;
            for (int jj = 0; jj < G; ++jj) {
                float v[CPL];
                ld_f32_n<CPL>(src + (int64_t)jj * p.ntok * d.dk, v);
#pragma unroll
                for (int q = 0; q < CPL; ++q) dxn[q] += v[q];
            }
#pragma unroll
            for (int q = 0; q < CPL; ++q) {
                y[q] = z[q] * sigm(z[q]);
                ss = fmaf(y[q], y[q], ss);
            }
        } else {
#pragma unroll
            for (int q = 0; q < CPL; ++q) z[q] = y[q] = dxn[q] = 0.f;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            if (off < lph) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float rho = 1.0f / sqrtf(ss + d.l2_eps);
        float dot = 0.f;
#pragma unroll
        for (int q = 0; q < CPL; ++q) dot = fmaf(y[q] * rho, dxn[q], dot);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            if (off < lph) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        if (act) {
            float out[CPL];
#pragma unroll
            for (int q = 0; q < CPL; ++q) out[q] = rho * (dxn[q] - y[q] * rho * dot) * dsilu(z[q]);
            float *dst = bp.dz + t * ch + (isk ? ch_qk : 0) + h * d.dk + i;
            if constexpr (CPL % 4 == 0) {
#pragma unroll
                for (int q = 0; q < CPL / 4; ++q)
                    st4(dst + 4 * q, out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
            } else {
#pragma unroll
                for (int q = 0; q < CPL; ++q) dst[q] = out[q];
            }
        }
    } else if (blk < nA + nB) {
        // ---- v: 4 adjacent channels of one token
        const int64_t item = (blk - nA) * kProThreads + threadIdx.x;
        const int quads = ch_v / 4;
        if (item >= p.ntok * quads) return;
        const int64_t t = item / quads;
        const int cv = (int)(item - t * quads) * 4;
        int64_t s0, s1, b, tau;
        seq_of(d, p.cu, t, s0, s1);
        tok_pos(d, t, b, tau);
        float z[4];
        conv_z_n<T, 4>((const T *)p.v_raw + cv, d.v_stride_b, d.v_stride_t, b, tau, t, s0,
                       (const T *)p.conv_w + (int64_t)(2 * ch_qk + cv) * kConvW, z);
        const int jh = cv / d.dv;
        const int64_t r = (int64_t)jh * p.ntok + t;
        const float be = p.beta[r];
        const float4 g = ld4(bp.dR + r * d.dv + (cv - jh * d.dv));
        st4(bp.dz + t * ch + 2 * ch_qk + cv, be * g.x * dsilu(z[0]), be * g.y * dsilu(z[1]), be * g.z * dsilu(z[2]),
            be * g.w * dsilu(z[3]));
    } else {
        // ---- beta / decay of one (token, v head)
        const int64_t item = (blk - nA - nB) * kProThreads + threadIdx.x;
        if (item >= p.ntok * d.Hv) return;
        const int64_t t = item / d.Hv;
        const int h = (int)(item - t * d.Hv);
        int64_t b, tau;
        tok_pos(d, t, b, tau);
        const float av = to_f<T>(((const T *)p.a)[b * d.a_stride_b + tau * d.a_stride_t + h]);
        const float bv = to_f<T>(((const T *)p.b)[b * d.b_stride_b + tau * d.b_stride_t + h]);
        const int64_t r = (int64_t)h * p.ntok + t;
        const float be = sigm(bv);
        ((T *)bp.db)[t * d.Hv + h] = from_f<T>(bp.dbeta[r] * be * (1.0f - be));
        const float x = av + p.dt_bias[h], eA = expf(p.A_log[h]);
        const float dg = bp.dgam[r];
        const float dx = -dg * eA * sigm(x);
        ((T *)bp.da)[t * d.Hv + h] = from_f<T>(dx);
        bp.pa[r] = dx;
        bp.pa[(int64_t)d.Hv * p.ntok + r] = dg * (-eA * softplus_f(x));
    }
}

template <typename T, int CPL>
cudaError_t launch_prologue_bwd_c(const BwdProblem &bp, cudaStream_t s) {
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int64_t lph = d.dk / CPL;
    const int64_t nA = (p.ntok * 2 * d.Hk * lph + kProThreads - 1) / kProThreads;
    const int64_t nB = (p.ntok * (d.Hv * d.dv / 4) + kProThreads - 1) / kProThreads;
    const int64_t nC = (p.ntok * d.Hv + kProThreads - 1) / kProThreads;
    if (nA + nB + nC == 0) return cudaSuccess;
    prologue_bwd_kernel<T, CPL><<<(unsigned)(nA + nB + nC), kProThreads, 0, s>>>(bp, nA, nB);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prologue_bwd(const BwdProblem &bp, cudaStream_t s) {
    switch (bp.f.d.dk) {      // channels per lane: a head over at most one warp
    case 512: return launch_prologue_bwd_c<T, 16>(bp, s);
    case 256: return launch_prologue_bwd_c<T, 8>(bp, s);
    case 128: return launch_prologue_bwd_c<T, 4>(bp, s);
    case 64: return launch_prologue_bwd_c<T, 2>(bp, s);
    default: return launch_prologue_bwd_c<T, 1>(bp, s);
    }
}

// ------------------------------------------------------------ conv backward
// grid (blocks of kBwdConvTokens tokens, groups of 4 * kConvQuads channels);
// per channel, dx_t = sum_m w_m dz_{t+3-m} within the sequence, and the
// block's partial sums of dw_m = sum_t dz_t x_{t-3+m}. A thread owns 4
// adjacent channels (one tensor: the q|k|v boundaries are multiples of 16) and
// walks runs of kConvRun tokens: the run's dz rows and raw-input rows, with
// their 3-token halos, are all loaded before the run is computed. The CTA's
// kConvRuns token rows then add their partial sums in a fixed order.
constexpr int kConvQuads = 32;   // channel quads per CTA (x)
constexpr int kConvRuns = 4;     // token runs side by side (y)
constexpr int kConvRun = 8;      // tokens per run
static_assert(kBwdConvTokens % (kConvRuns * kConvRun) == 0, "conv backward token tiling");

template <typename T>
__global__ void __launch_bounds__(kConvQuads * kConvRuns) conv_bwd_kernel(const BwdProblem bp) {
    __shared__ float4 red[kConvRuns][kConvW][kConvQuads];
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    const int ch_qk = d.Hk * d.dk, ch_v = d.Hv * d.dv, ch = 2 * ch_qk + ch_v;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int c = (blockIdx.y * kConvQuads + tx) * 4;
    const bool active = c < ch;
    const T *x = (const T *)p.q_raw;
    T *dx = (T *)bp.dq_raw;
    int64_t sb = d.q_stride_b, st = d.q_stride_t, ostride = ch_qk;
    int c_in = c;
    if (c >= 2 * ch_qk) {
        x = (const T *)p.v_raw; sb = d.v_stride_b; st = d.v_stride_t; c_in = c - 2 * ch_qk;
        dx = (T *)bp.dv_raw; ostride = ch_v;
    } else if (c >= ch_qk) {
        x = (const T *)p.k_raw; sb = d.k_stride_b; st = d.k_stride_t; c_in = c - ch_qk;
        dx = (T *)bp.dk_raw;
    }
    // w[m] = tap m of the four channels
    float4 w[kConvW];
    {
        float wv[4 * kConvW];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = active ? ld4_act<T>((const T *)p.conv_w + (int64_t)c * kConvW + 4 * q)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            wv[4 * q] = f.x; wv[4 * q + 1] = f.y; wv[4 * q + 2] = f.z; wv[4 * q + 3] = f.w;
        }
#pragma unroll
        for (int m = 0; m < kConvW; ++m)
            w[m] = make_float4(wv[m], wv[kConvW + m], wv[2 * kConvW + m], wv[3 * kConvW + m]);
    }
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 dw[kConvW] = {z4, z4, z4, z4};
    int64_t s0 = 0, s1 = -1;
    const int64_t tb = (int64_t)blockIdx.x * kBwdConvTokens;
    for (int run = ty; run * kConvRun < kBwdConvTokens; run += kConvRuns) {
        const int64_t ta = tb + (int64_t)run * kConvRun;
        if (ta >= p.ntok) break;
        // dz rows ta .. ta + kConvRun + 2, raw-input rows ta - 3 .. ta + kConvRun - 1
        float4 g[kConvRun + kConvW - 1], xr[kConvRun + kConvW - 1];
#pragma unroll
        for (int k = 0; k < kConvRun + kConvW - 1; ++k) {
            const int64_t pz = ta + k, px = ta - (kConvW - 1) + k;
            g[k] = (active && pz < p.ntok) ? ld4(bp.dz + pz * ch + c) : z4;
            if (active && px >= 0 && px < p.ntok) {
                const int64_t b = p.cu ? 0 : px / d.T;
                xr[k] = ld4_act<T>(x + b * sb + (px - b * d.T) * st + c_in);
            } else {
                xr[k] = z4;
            }
        }
#pragma unroll
        for (int u = 0; u < kConvRun; ++u) {
            const int64_t t = ta + u;
            if (t >= p.ntok) break;
            if (t >= s1) seq_of(d, p.cu, t, s0, s1);
            float4 gx = z4;
#pragma unroll
            for (int m = 0; m < kConvW; ++m)
                if (t + (kConvW - 1 - m) < s1) gx = fma4(w[m], g[u + kConvW - 1 - m], gx);
            if (active) st4_act<T>(dx + t * ostride + c_in, gx);
#pragma unroll
            for (int m = 0; m < kConvW; ++m)
                if (t - (kConvW - 1 - m) >= s0) dw[m] = fma4(g[u], xr[u + m], dw[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < kConvW; ++m) red[ty][m][tx] = dw[m];
    __syncthreads();
    if (ty == 0 && active) {
        float out[4][kConvW];   // [channel][tap]
#pragma unroll
        for (int m = 0; m < kConvW; ++m) {
            float4 a = red[0][m][tx];
#pragma unroll
            for (int r = 1; r < kConvRuns; ++r) a = add4(a, red[r][m][tx]);
            out[0][m] = a.x; out[1][m] = a.y; out[2][m] = a.z; out[3][m] = a.w;
        }
        float4 *dst = reinterpret_cast<float4 *>(bp.pconv + ((int64_t)blockIdx.x * ch + c) * kConvW);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(out[q][0], out[q][1], out[q][2], out[q][3]);
    }
}

// out[i] = sum_{r < R} part[r * rs + i] for i < n, one thread per i, r in order
__global__ void __launch_bounds__(kThreads) sum_rows_kernel(const float *part, int64_t R, int64_t rs, int64_t n,
                                                            float *out) {
    const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= n) return;
    float acc = 0.f;
#pragma unroll 8
    for (int64_t r = 0; r < R; ++r) acc += part[r * rs + i];
    out[i] = acc;
}

// out[i] = sum_{r < R} part[r * rs + i * cs], one CTA per i, fixed order
__global__ void __launch_bounds__(kThreads) sum_kernel(const float *part, int64_t R, int64_t rs, int64_t cs,
                                                       float *out) {
    __shared__ float red[kThreads];
    const int64_t i = blockIdx.x;
    float acc = 0.f;
    for (int64_t r = threadIdx.x; r < R; r += kThreads) acc += part[r * rs + i * cs];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int s = kThreads / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[i] = red[0];
}

// ------------------------------------------------------------ launches
template <typename T, typename GTy, typename WT>
cudaError_t launch_rms(const BwdProblem &bp, cudaStream_t s) {
    const gdn_desc &d = bp.f.d;
    const int64_t rows = bp.f.ntok * d.Hv;
    if (rows == 0) return cudaSuccess;
    const int64_t nwarps = bwd_epi_warps(d);
    const unsigned blocks = (unsigned)((nwarps + kThreads / 32 - 1) / (kThreads / 32));
    switch (d.dv <= 32 ? 1 : d.dv / 32) {
    case 1: rms_bwd_kernel<T, GTy, WT, 1><<<blocks, kThreads, 0, s>>>(bp, rows, nwarps); break;
    case 2: rms_bwd_kernel<T, GTy, WT, 2><<<blocks, kThreads, 0, s>>>(bp, rows, nwarps); break;
    case 4: rms_bwd_kernel<T, GTy, WT, 4><<<blocks, kThreads, 0, s>>>(bp, rows, nwarps); break;
    case 8: rms_bwd_kernel<T, GTy, WT, 8><<<blocks, kThreads, 0, s>>>(bp, rows, nwarps); break;
    default: rms_bwd_kernel<T, GTy, WT, 16><<<blocks, kThreads, 0, s>>>(bp, rows, nwarps); break;
    }
    return cudaGetLastError();
}

template <typename T, typename GTy>
cudaError_t launch_rms_w(const BwdProblem &bp, cudaStream_t s) {
    return bp.f.d.norm_w_dtype == GDN_F32 ? launch_rms<T, GTy, float>(bp, s) : launch_rms<T, GTy, T>(bp, s);
}

// the serial kernels' dv tile: the widest of 64 / 32 / 16 columns within dv
// whose shared memory fits a CTA (measured fastest at the layer and
// long-sequence shapes: narrower tiles give more CTAs, but each CTA's chain is
// bound by its per-chunk loads and barriers rather than by its work)
int serial_tile(const gdn_desc &d) {
    if (d.dv >= 64 && serial_smem_bytes<64>(d.dk) <= 227 * 1024) return 64;
    if (d.dv >= 32 && serial_smem_bytes<32>(d.dk) <= 227 * 1024) return 32;
    return 16;
}

template <typename T, int NV>
cudaError_t launch_serial(const BwdProblem &bp, bool reverse, cudaStream_t s) {
    const gdn_desc &d = bp.f.d;
    const int ntiles = d.dv / NV;
    const int64_t blocks = (int64_t)d.N * d.Hv * ntiles;
    if (blocks == 0) return cudaSuccess;
    cudaError_t e;
    if (!reverse) {
        const size_t bytes = serial_smem_bytes<NV>(d.dk);
        e = cudaFuncSetAttribute(states_kernel<T, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        states_kernel<T, NV><<<(unsigned)blocks, 4 * NV, bytes, s>>>(bp, ntiles);
    } else {
        const size_t bytes = serial_smem_bytes<NV>(d.dk);
        e = cudaFuncSetAttribute(chain_bwd_kernel<T, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
        chain_bwd_kernel<T, NV><<<(unsigned)blocks, 4 * NV, bytes, s>>>(bp, ntiles);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_serial_nv(const BwdProblem &bp, bool reverse, cudaStream_t s) {
    switch (serial_tile(bp.f.d)) {
    case 64: return launch_serial<T, 64>(bp, reverse, s);
    case 32: return launch_serial<T, 32>(bp, reverse, s);
    default: return launch_serial<T, 16>(bp, reverse, s);
    }
}

template <typename K>
cudaError_t launch_per_chunk(K kernel, size_t bytes, const BwdProblem &bp, int64_t slots, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kernel<<<dim3((unsigned)slots, bp.f.d.Hv), kThreads, bytes, s>>>(bp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const BwdProblem &bp, cudaStream_t s) {
    const Problem &p = bp.f;
    const gdn_desc &d = p.d;
    const int64_t slots = chunk_slots(p);
    cudaError_t e = cudaSuccess;
    if (slots > 0 && (e = launch_per_chunk(mats_kernel<T>, mats_smem_bytes(), bp, slots, s)) != cudaSuccess) return e;
    if (sizeof(T) == 2 && p.ntok > 0 && chunk_tc_supports(d)) {
        // the forward's tensor-core chunk stage recomputes H0, Vn and O (fp32 stores)
        Problem pr = p;
        pr.rec_h0 = bp.h0;
        pr.rec_vn = bp.vn;
        pr.rec_o = bp.dO;
        pr.hT = nullptr;
        pr.pdl = false;
        if ((e = launch_chunk_tc_rec(pr, s)) != cudaSuccess) return e;
    } else {
        if ((e = launch_serial_nv<T>(bp, false, s)) != cudaSuccess) return e;
        if (slots > 0) {
            e = out_tc_supports(d) ? launch_out_tc(bp, slots, s)
                                   : launch_per_chunk(out_kernel<T>, out_smem_bytes(), bp, slots, s);
            if (e != cudaSuccess) return e;
        }
    }
    e = d.gate_dtype == GDN_F32 ? launch_rms_w<T, float>(bp, s) : launch_rms_w<T, T>(bp, s);
    if (e != cudaSuccess) return e;
    if (slots > 0) {
        e = dterms_tc_supports(d) ? launch_dterms_tc(bp, slots, s)
                                  : launch_per_chunk(dterms_kernel<T>, dterms_smem_bytes(), bp, slots, s);
        if (e != cudaSuccess) return e;
    }
    if ((e = launch_serial_nv<T>(bp, true, s)) != cudaSuccess) return e;
    if (slots > 0) {
        if (chunk_x_tc_supports(d)) {
            if ((e = launch_chunk_x_tc(bp, slots, s)) != cudaSuccess) return e;
            e = launch_per_chunk(chunk_grad_kernel<T, true>, grad_smem_bytes(), bp, slots, s);
        } else {
            e = launch_per_chunk(chunk_grad_kernel<T, false>, grad_smem_bytes(), bp, slots, s);
        }
        if (e != cudaSuccess) return e;
    }
    const int ch_qk = d.Hk * d.dk, ch_v = d.Hv * d.dv, ch = 2 * ch_qk + ch_v;
    if (p.ntok > 0) {
        if ((e = launch_prologue_bwd<T>(bp, s)) != cudaSuccess) return e;
        conv_bwd_kernel<T><<<dim3((unsigned)bwd_conv_blocks(d), (ch + 4 * kConvQuads - 1) / (4 * kConvQuads)),
                             dim3(kConvQuads, kConvRuns), 0, s>>>(bp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // parameter gradients: fixed-order sums of the partials (zero without tokens)
    const int64_t rows = p.ntok * d.Hv;
    sum_kernel<<<d.dv, kThreads, 0, s>>>(bp.pnorm, rows > 0 ? bwd_epi_warps(d) : 0, d.dv, 1, bp.dnorm_w);
    sum_rows_kernel<<<(ch * kConvW + kThreads - 1) / kThreads, kThreads, 0, s>>>(
        bp.pconv, p.ntok > 0 ? bwd_conv_blocks(d) : 0, (int64_t)ch * kConvW, (int64_t)ch * kConvW, bp.dconv_w);
    sum_kernel<<<d.Hv, kThreads, 0, s>>>(bp.pa, p.ntok, 1, p.ntok, bp.ddt_bias);
    sum_kernel<<<d.Hv, kThreads, 0, s>>>(bp.pa + (int64_t)d.Hv * p.ntok, p.ntok, 1, p.ntok, bp.dA_log);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdProblem &p, cudaStream_t s) {
    switch (p.f.d.dtype) {
    case GDN_F32: return launch_t<float>(p, s);
    case GDN_BF16: return launch_t<__nv_bfloat16>(p, s);
    default: return launch_t<__half>(p, s);
    }
}

}  // namespace gdn
