// gdn_epilogue.cu -- post-GDR gated RMSNorm of the GDN core forward.
//
// y = round_act(norm_w * o * rsqrt(mean(o^2) + eps)) * silu(gate), per
// (token, v head) row of dv values ("GDN Elementwise Fusion", post-GDR
// requirements: gate in the act dtype or fp32, possibly a strided view into the
// input projection with separate batch and token strides, consumed in place;
// "Execution and numerical behavior": the RMSNorm result is materialised in the
// activation dtype before the fp32 SiLU-gating multiply).
// HBM-bound streaming kernel: each row is read once (o, gate) and written once
// with 16-byte accesses where the gate view's alignment allows, scalar gate
// loads where it does not. A row spans at most one warp, so the mean of
// squares is a shuffle reduction.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;

template <typename T, typename G, typename W, int NVEC, bool GVEC>
__global__ void __launch_bounds__(kThreads) epilogue_kernel(const Problem p) {
    constexpr int VEC = Vec16<T>::N;
    constexpr int CPT = NVEC * VEC;
    __shared__ float nw[512];
    const gdn_desc &d = p.d;
    const int dv = d.dv;
    for (int i = threadIdx.x; i < dv; i += kThreads) nw[i] = to_f<W>(((const W *)p.norm_w)[i]);
    __syncthreads();

    const int lpr = dv / CPT;                  // lanes per row (power of two, <= 32)
    const int rows_per_block = kThreads / lpr;
    const int sub = threadIdx.x / lpr;         // row slot in the block
    const int cc = (threadIdx.x - sub * lpr) * CPT;
    const float inv_dv = 1.0f / (float)dv;
    const int64_t nrows = p.ntok * d.Hv;
    using S = typename Inter<T>::S;    // storage of o
    const S *o = (const S *)p.o;
    bool finite = true;
    const G *gate = (const G *)p.gate;
    T *out = (T *)p.out;

    for (int64_t r0 = (int64_t)blockIdx.x * rows_per_block; r0 < nrows;
         r0 += (int64_t)gridDim.x * rows_per_block) {
        const int64_t r = r0 + sub;
        const bool valid = r < nrows;
        float x[CPT], gv[CPT];
        if (valid) {
            const int64_t tok = r / d.Hv;
            const int h = (int)(r - tok * d.Hv);
#pragma unroll
            for (int v = 0; v < NVEC; ++v) load16_f<S>(o + r * dv + cc + v * VEC, x + v * VEC);
#pragma unroll
            for (int i = 0; i < CPT; ++i) finite = finite && isfinite(x[i]);
            const G *gp = gate + tok_offset(tok, d.T, d.gate_stride_b, d.gate_stride_t) + h * dv + cc;
            if (GVEC) {
                constexpr int GV = Vec16<G>::N;
#pragma unroll
                for (int v = 0; v < CPT; v += GV) load16_f<G>(gp + v, gv + v);
            } else {
#pragma unroll
                for (int i = 0; i < CPT; ++i) gv[i] = to_f<G>(gp[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < CPT; ++i) x[i] = gv[i] = 0.f;
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) ss = fmaf(x[i], x[i], ss);
        for (int off = lpr >> 1; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss * inv_dv + d.norm_eps);
        if (valid) {
            float y[CPT];
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const float rn = round_through<T>(nw[cc + i] * (x[i] * inv));
                y[i] = rn * silu_f(gv[i]);
            }
#pragma unroll
            for (int v = 0; v < NVEC; ++v) store16_f_cs<T>(out + r * dv + cc + v * VEC, y + v * VEC);
        }
    }
    // a non-finite gated-delta-rule output (unless an earlier stage already
    // reported a malformed cu_seqlens, after which o holds nothing meaningful)
    if (__syncthreads_or(!finite) && threadIdx.x == 0 && *p.status == GDN_OK)
        *p.status = GDN_ERR_DEVICE_RANGE;
}

template <typename T, typename G, typename W, int NVEC>
cudaError_t launch_g(const Problem &p, cudaStream_t s) {
    constexpr int CPT = NVEC * Vec16<T>::N;
    const int lpr = p.d.dv / CPT;
    const int rows_per_block = kThreads / lpr;
    const int64_t nrows = p.ntok * p.d.Hv;
    int64_t blocks = (nrows + rows_per_block - 1) / rows_per_block;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const size_t gs = sizeof(G);
    const bool gvec = ((uintptr_t)p.gate % 16 == 0) && ((p.d.gate_stride_b * gs) % 16 == 0) &&
                      ((p.d.gate_stride_t * gs) % 16 == 0) && ((CPT * gs) % 16 == 0);
    if (gvec) epilogue_kernel<T, G, W, NVEC, true><<<(unsigned)blocks, kThreads, 0, s>>>(p);
    else epilogue_kernel<T, G, W, NVEC, false><<<(unsigned)blocks, kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T, typename G, typename W>
cudaError_t launch_w(const Problem &p, cudaStream_t s) {
    constexpr int VEC = Vec16<T>::N;
    const int need = p.d.dv / 32;              // channels per lane so that a row fits a warp
    if (need <= VEC) return launch_g<T, G, W, 1>(p, s);
    if (need <= 2 * VEC) return launch_g<T, G, W, 2>(p, s);
    return launch_g<T, G, W, 4>(p, s);
}

template <typename T, typename G>
cudaError_t launch_gw(const Problem &p, cudaStream_t s) {
    if (p.d.norm_w_dtype == GDN_F32) return launch_w<T, G, float>(p, s);
    return launch_w<T, G, T>(p, s);
}

template <typename T>
cudaError_t launch_t(const Problem &p, cudaStream_t s) {
    if (p.d.gate_dtype == GDN_F32) return launch_gw<T, float>(p, s);
    return launch_gw<T, T>(p, s);
}

}  // namespace

cudaError_t launch_epilogue(const Problem &p, cudaStream_t s) {
    switch (p.d.dtype) {
    case GDN_F32: return launch_t<float>(p, s);
    case GDN_BF16: return launch_t<__nv_bfloat16>(p, s);
    default: return launch_t<__half>(p, s);
    }
}

}  // namespace gdn
