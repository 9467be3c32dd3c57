// gdn_epilogue.cu -- post-GDR gated RMSNorm of the GDN core forward.
//
// y = round_act(norm_w * o * rsqrt(mean(o^2) + eps)) * silu(gate), per
// (token, v head) row of dv values ("GDN Elementwise Fusion", post-GDR
// requirements: gate in the act dtype or fp32, possibly a strided view into the
// input projection with separate batch and token strides, consumed in place;
// "Execution and numerical behavior": the RMSNorm result is materialised in the
// activation dtype before the fp32 SiLU-gating multiply).
// HBM-bound streaming kernel: each thread owns the same column slice of a few
// consecutive rows and issues all of their loads first; each row is read once
// (o, gate) and written once with 16-byte accesses (scalar gate loads where the
// view's alignment does not allow 16 bytes). A row spans at most one warp, so
// the mean of squares is a shuffle reduction. The arithmetic runs on fp32
// pairs (one packed instruction per two columns).
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;

// Rows (token, v head) of one thread: R consecutive rows, so that one division
// locates the first and the rest follow by carrying the head index. Small
// problems take R = 2 (more, smaller CTAs: a shorter tail), large ones R = 4
// (more loads in flight per thread).
constexpr int64_t kManyRows = 1 << 20;

template <typename T, typename G, typename W, int NVEC, bool GVEC, int R>
__global__ void __launch_bounds__(kThreads) epilogue_kernel(const Problem p) {
    constexpr int VEC = Vec16<T>::N;
    constexpr int CPT = NVEC * VEC;            // columns per thread
    constexpr int NP = CPT / 2;                // column pairs per thread
    constexpr int GN = GVEC ? CPT * (int)sizeof(G) / 16 : 1;   // 16-byte gate vectors
    using S = typename Inter<T>::S;            // storage of o
    // norm weights, one padding slot after every CPT of them: lane l reads
    // [l*(CPT+1), +CPT) without bank conflicts
    __shared__ float nwp[512 + 512 / 4];
    const gdn_desc &d = p.d;
    const int dv = d.dv;
    for (int i = threadIdx.x; i < dv; i += kThreads) nwp[(i / CPT) * (CPT + 1) + i % CPT] = to_f<W>(((const W *)p.norm_w)[i]);
    pdl_wait();       // o (and the status word) of the chunk stage are complete

    const int lpr = dv / CPT;                  // lanes per row (power of two, <= 32)
    const int rows_per_pass = kThreads / lpr;
    const int sub = threadIdx.x / lpr;
    const int lane_in_row = threadIdx.x - sub * lpr;
    const int cc = lane_in_row * CPT;
    const int64_t nrows = p.ntok * d.Hv;
    const int64_t r0 = ((int64_t)blockIdx.x * rows_per_pass + sub) * R;

    // head of the first row, and its token as (batch row, token in the row) for
    // the gate view; 32-bit divisions unless the row count needs more
    int h, tt;
    int64_t bt;
    if (nrows <= 0x7fffffff) {
        const uint32_t q = (uint32_t)r0 / (uint32_t)d.Hv;
        h = (int)((uint32_t)r0 - q * (uint32_t)d.Hv);
        const uint32_t b = q / (uint32_t)d.T;
        tt = (int)(q - b * (uint32_t)d.T);
        bt = b;
    } else {
        const int64_t tok = r0 / d.Hv;
        h = (int)(r0 - tok * d.Hv);
        bt = tok / d.T;
        tt = (int)(tok - bt * d.T);
    }

    // every load of this thread first
    uint4 ox[R][NVEC];
    uint4 gx[R][GN];
    float gs[R][GVEC ? 1 : CPT];
#pragma unroll
    for (int k = 0; k < R; ++k) {
        if (r0 + k < nrows) {
            const uint4 *op = reinterpret_cast<const uint4 *>((const S *)p.o + (r0 + k) * dv + cc);
#pragma unroll
            for (int v = 0; v < NVEC; ++v) ox[k][v] = __ldcs(op + v);
            const G *gp = (const G *)p.gate + bt * d.gate_stride_b + tt * d.gate_stride_t + h * dv + cc;
            if (GVEC) {
#pragma unroll
                for (int v = 0; v < GN; ++v) gx[k][v] = __ldcs(reinterpret_cast<const uint4 *>(gp) + v);
            } else {
#pragma unroll
                for (int i = 0; i < (GVEC ? 1 : CPT); ++i) gs[k][i] = to_f<G>(gp[i]);
            }
        } else {
#pragma unroll
            for (int v = 0; v < NVEC; ++v) ox[k][v] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int v = 0; v < GN; ++v) gx[k][v] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < (GVEC ? 1 : CPT); ++i) gs[k][i] = 0.f;
        }
        if (++h == d.Hv) {
            h = 0;
            if (++tt == d.T) { tt = 0; ++bt; }
        }
    }
    __syncthreads();
    float2 w[NP];
    {
        const float *wv = nwp + lane_in_row * (CPT + 1);
#pragma unroll
        for (int i = 0; i < NP; ++i) w[i] = make_float2(wv[2 * i], wv[2 * i + 1]);
    }
    bool finite = true;
#pragma unroll
    for (int k = 0; k < R; ++k) {
        float2 x[NP];
#pragma unroll
        for (int v = 0; v < NVEC; ++v) Pairs<S>::unpack(ox[k][v], x + v * (VEC / 2));
        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) ss2 = fma2(x[i], x[i], ss2);
        float ss = ss2.x + ss2.y;
        for (int off = lpr >> 1; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        // a non-finite element makes the sum of squares non-finite
        finite = finite && isfinite(ss);
        const float2 inv = splat2(rsqrtf(ss * (1.0f / (float)dv) + d.norm_eps));
        if (r0 + k < nrows) {
            float2 g[NP];
            if (GVEC) {
                constexpr int GE = 16 / sizeof(G);
#pragma unroll
                for (int v = 0; v < GN; ++v) Pairs<G>::unpack(gx[k][v], g + v * (GE / 2));
            } else {
#pragma unroll
                for (int i = 0; i < NP; ++i) g[i] = make_float2(gs[k][GVEC ? 0 : 2 * i], gs[k][GVEC ? 0 : 2 * i + 1]);
            }
            float2 y[NP];
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const float2 rn = Pairs<T>::round(mul2(w[i], mul2(x[i], inv)));
                y[i] = mul2(rn, silu2_act<T>(g[i]));
            }
            uint4 *out = reinterpret_cast<uint4 *>((T *)p.out + (r0 + k) * dv + cc);
#pragma unroll
            for (int v = 0; v < NVEC; ++v) __stcs(out + v, Pairs<T>::pack(y + v * (VEC / 2)));
        }
    }
    // a non-finite gated-delta-rule output (unless an earlier stage already
    // reported a malformed cu_seqlens, after which o holds nothing meaningful)
    if (__syncthreads_or(!finite) && threadIdx.x == 0 && *p.status == GDN_OK)
        *p.status = GDN_ERR_DEVICE_RANGE;
}

template <typename T, typename G, typename W, int NVEC, int R>
cudaError_t launch_r(const Problem &p, cudaStream_t s) {
    constexpr int CPT = NVEC * Vec16<T>::N;
    const int lpr = p.d.dv / CPT;
    const int rows_per_block = kThreads / lpr * R;
    const int64_t nrows = p.ntok * p.d.Hv;
    const int64_t blocks = (nrows + rows_per_block - 1) / rows_per_block;
    const size_t gs = sizeof(G);
    const bool gvec = ((uintptr_t)p.gate % 16 == 0) && ((p.d.gate_stride_b * gs) % 16 == 0) &&
                      ((p.d.gate_stride_t * gs) % 16 == 0) && ((CPT * gs) % 16 == 0);
    auto kernel = gvec ? epilogue_kernel<T, G, W, NVEC, true, R> : epilogue_kernel<T, G, W, NVEC, false, R>;
    return launch_kernel(p.pdl, kernel, dim3((unsigned)blocks), dim3(kThreads), 0, s, p);
}

template <typename T, typename G, typename W, int NVEC>
cudaError_t launch_g(const Problem &p, cudaStream_t s) {
    if (p.ntok * p.d.Hv >= kManyRows) return launch_r<T, G, W, NVEC, 4>(p, s);
    return launch_r<T, G, W, NVEC, 2>(p, s);
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
