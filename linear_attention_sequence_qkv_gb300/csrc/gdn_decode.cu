// gdn_decode.cu -- one decode step of the GDN core: one new token per sequence.
//
// The forward's definitions applied to one more token of each sequence: the
// width-4 causal depthwise conv ("fused q/k/v short conv", flash-linear-attention
// PR #972, "Summary") over the sequence's last three raw inputs (a conv cache,
// advanced in place) and the token, SiLU, the per-head q/k L2 norm with eps 1e-6
// (Megatron-LM PR #5396, "Why"), beta = sigmoid(b), g = -exp(A_log) softplus(a +
// dt_bias), and one step of the gated delta rule
//     S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
// on the carried fp32 state (stored as H = S^T, [dk][dv]), written with
// u = H^T k as H_t = e^g H + k (beta (v - e^g u))^T. The gated RMSNorm is the
// forward's epilogue kernel over the B new tokens.
//
// Two kernels: decode_prep (conv + cache, norms, beta / decay; every channel is
// read and rewritten by one thread) and decode_state (one CTA per (sequence,
// v head, stripe of up to 128 columns of dv): each thread keeps 16 rows of 4
// adjacent columns in registers, so the state is read once and written once
// with 16-byte accesses). The step is bound by the state traffic, 8 bytes per
// element of S per token.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kPrepThreads = 512;   // most threads of a prep CTA: max(dk, 128) are launched
constexpr int kQuadRows = 16;       // state rows per thread (4 columns each)

// y = silu(conv) of channel c from the cache and the token x; advances the cache
template <typename T>
__device__ __forceinline__ float conv_token(T *cs, const T *w, int c, T x) {
    const float x3 = to_f<T>(cs[3 * c]), x2 = to_f<T>(cs[3 * c + 1]), x1 = to_f<T>(cs[3 * c + 2]);
    const float x0 = to_f<T>(x);
    float acc = to_f<T>(w[4 * c]) * x3;
    acc = fmaf(to_f<T>(w[4 * c + 1]), x2, acc);
    acc = fmaf(to_f<T>(w[4 * c + 2]), x1, acc);
    acc = fmaf(to_f<T>(w[4 * c + 3]), x0, acc);
    cs[3 * c] = cs[3 * c + 1];
    cs[3 * c + 1] = cs[3 * c + 2];
    cs[3 * c + 2] = x;
    return silu_f(acc);
}

// grid (B, 2*Hk q/k heads + v channel groups + 1 beta/decay unit)
template <typename T>
__global__ void __launch_bounds__(kPrepThreads) decode_prep_kernel(const DecodeProblem p, int units_v) {
    __shared__ float red[kPrepThreads / 32];
    const gdn_desc &d = p.d;
    const int n = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
    const int ch_qk = d.Hk * d.dk, ch_v = d.Hv * d.dv, ch = 2 * ch_qk + ch_v;
    T *cs = (T *)p.conv_state + (int64_t)n * ch * 3;
    const T *w = (const T *)p.conv_w;
    if (n == 0 && u == 0 && tid == 0) *p.status = GDN_OK;
    if (u < 2 * d.Hk) {                       // one q or k head
        const bool isk = u >= d.Hk;
        const int h = isk ? u - d.Hk : u;
        float y = 0.f;
        if (tid < d.dk) {
            const int cl = h * d.dk + tid;
            const T *x = (const T *)(isk ? p.k_raw : p.q_raw) + (int64_t)n * (isk ? d.k_stride_b : d.q_stride_b) + cl;
            y = conv_token<T>(cs, w, (isk ? ch_qk : 0) + cl, *x);
        }
        float ss = y * y;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < (d.dk + 31) / 32; ++i) tot += red[i];
        if (tid < d.dk) (isk ? p.k : p.q)[((int64_t)h * d.B + n) * d.dk + tid] = y * rsqrtf(tot + d.l2_eps);
    } else if (u < 2 * d.Hk + units_v) {      // a group of v channels
        const int cv = (u - 2 * d.Hk) * (int)blockDim.x + tid;
        if (cv < ch_v) {
            const T *x = (const T *)p.v_raw + (int64_t)n * d.v_stride_b + cv;
            p.v[(int64_t)n * ch_v + cv] = conv_token<T>(cs, w, 2 * ch_qk + cv, *x);
        }
    } else {                                  // beta and decay of every v head
        for (int h = tid; h < d.Hv; h += blockDim.x) {
            const float av = to_f<T>(((const T *)p.a)[(int64_t)n * d.a_stride_b + h]);
            const float bv = to_f<T>(((const T *)p.b)[(int64_t)n * d.b_stride_b + h]);
            p.beta[(int64_t)n * d.Hv + h] = sigmoid_f(bv);
            p.g[(int64_t)n * d.Hv + h] = -expf(p.A_log[h]) * softplus_f(av + p.dt_bias[h]);
        }
    }
}

// grid (B * Hv, dv / (4 nq)); block nq x (dk / kQuadRows) threads: thread
// (qd, slice) owns columns [4 qd, +4) of the CTA's stripe and rows
// [slice * kQuadRows, +kQuadRows) of the state of (n, j), in registers
template <typename S>
__global__ void __launch_bounds__(256, 2) decode_state_kernel(const DecodeProblem p, int nq) {
    extern __shared__ float dsm[];
    const gdn_desc &d = p.d;
    const int dk = d.dk, dv = d.dv;
    const int qd = threadIdx.x % nq, slice = threadIdx.x / nq;
    const int slices = blockDim.x / nq;
    const int nj = blockIdx.x;                // n * Hv + j
    const int n = nj / d.Hv, j = nj - n * d.Hv;
    const int hk = j / (d.Hv / d.Hk);
    const int c = (blockIdx.y * nq + qd) * 4;
    float *qs = dsm, *ks = dsm + dk;
    float4 *red = reinterpret_cast<float4 *>(dsm + 2 * dk);   // [slices][nq]
    for (int i = threadIdx.x; i < dk; i += blockDim.x) {
        qs[i] = p.q[((int64_t)hk * d.B + n) * dk + i];
        ks[i] = p.k[((int64_t)hk * d.B + n) * dk + i];
    }
    __syncthreads();
    const int r0 = slice * kQuadRows;
    const int rs = dv / 4;                    // row stride in float4
    float4 *H = reinterpret_cast<float4 *>(p.state + (int64_t)nj * dk * dv + (int64_t)r0 * dv + c);
    float4 h[kQuadRows];
#pragma unroll
    for (int i = 0; i < kQuadRows; ++i) h[i] = H[i * rs];
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kQuadRows; ++i) {
        const float kk = ks[r0 + i];
        u.x = fmaf(h[i].x, kk, u.x);
        u.y = fmaf(h[i].y, kk, u.y);
        u.z = fmaf(h[i].z, kk, u.z);
        u.w = fmaf(h[i].w, kk, u.w);
    }
    red[slice * nq + qd] = u;
    __syncthreads();
    float4 ut = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < slices; ++s) {
        const float4 t = red[s * nq + qd];
        ut.x += t.x; ut.y += t.y; ut.z += t.z; ut.w += t.w;
    }
    const float eg = expf(p.g[nj]), bt = p.beta[nj];
    const float4 v = *reinterpret_cast<const float4 *>(p.v + (int64_t)n * d.Hv * dv + (int64_t)j * dv + c);
    const float4 r = make_float4(bt * (v.x - eg * ut.x), bt * (v.y - eg * ut.y), bt * (v.z - eg * ut.z),
                                 bt * (v.w - eg * ut.w));
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kQuadRows; ++i) {
        const float kk = ks[r0 + i], qq = qs[r0 + i];
        float4 hn;
        hn.x = fmaf(eg, h[i].x, kk * r.x);
        hn.y = fmaf(eg, h[i].y, kk * r.y);
        hn.z = fmaf(eg, h[i].z, kk * r.z);
        hn.w = fmaf(eg, h[i].w, kk * r.w);
        H[i * rs] = hn;
        o.x = fmaf(hn.x, qq, o.x);
        o.y = fmaf(hn.y, qq, o.y);
        o.z = fmaf(hn.z, qq, o.z);
        o.w = fmaf(hn.w, qq, o.w);
    }
    __syncthreads();                          // every thread has read u's partial sums
    red[slice * nq + qd] = o;
    __syncthreads();
    if (slice == 0) {
        float4 ot = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < slices; ++s) {
            const float4 t = red[s * nq + qd];
            ot.x += t.x; ot.y += t.y; ot.z += t.z; ot.w += t.w;
        }
        S *dst = (S *)p.o + (int64_t)nj * dv + c;
        dst[0] = from_f<S>(ot.x * d.scale);
        dst[1] = from_f<S>(ot.y * d.scale);
        dst[2] = from_f<S>(ot.z * d.scale);
        dst[3] = from_f<S>(ot.w * d.scale);
    }
}

template <typename T>
cudaError_t launch_t(const DecodeProblem &p, cudaStream_t s) {
    const gdn_desc &d = p.d;
    const int ch_v = d.Hv * d.dv;
    // a q or k head per CTA (dk threads, at least 128 so that the v groups are not tiny)
    const int pt = d.dk > 128 ? d.dk : 128;
    const int units_v = (ch_v + pt - 1) / pt;
    decode_prep_kernel<T><<<dim3((unsigned)d.B, 2 * d.Hk + units_v + 1), pt, 0, s>>>(p, units_v);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // column quads per CTA: up to 128 columns, and at most 256 threads (two CTAs
    // per SM, so that one's stores overlap the other's loads)
    const int slices = d.dk / kQuadRows;
    int nq = d.dv / 4;
    if (nq > 32) nq = 32;
    if (nq * slices > 256) nq = 256 / slices;
    const int threads = nq * slices;
    const size_t smem = (size_t)2 * d.dk * sizeof(float) + (size_t)threads * sizeof(float4);
    using S = typename Inter<T>::S;
    decode_state_kernel<S><<<dim3((unsigned)((int64_t)d.B * d.Hv), d.dv / (4 * nq)), threads, smem, s>>>(p, nq);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem &p, cudaStream_t s) {
    switch (p.d.dtype) {
    case GDN_F32: return launch_t<float>(p, s);
    case GDN_BF16: return launch_t<__nv_bfloat16>(p, s);
    default: return launch_t<__half>(p, s);
    }
}

}  // namespace gdn
