// gdn_prologue.cu -- pre-GDR prologue of the GDN core forward.
//
// One kernel covers every pre-GDR step ("GDN Elementwise Fusion", option table:
// causal convolution, SiLU, layout transforms, Q/K L2 normalisation, head
// expansion, beta and decay preparation):
//   * a width-4 causal depthwise conv over the concatenated [q|k|v] channels,
//     then SiLU ("fused q/k/v short conv", flash-linear-attention PR #972,
//     "Summary": one depthwise conv over concatenated channels equals three);
//   * per-head L2 norm of q and k, x * rsqrt(sum x^2 + eps), eps = 1e-6
//     ("fold q/k L2-norm into the gated_delta_rule kernel", Megatron-LM PR #5396,
//     "Why"); q and k leave as fp32, or for 2-byte activations as two fp16
//     planes hi + lo carrying about fp32 precision;
//   * beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias) and the
//     inclusive cumulative sum of g inside each 64-token chunk.
// Grid: x = chunk slot (one 64-token chunk of one sequence), y = (channel group
// of q, k or v: 128 threads x 16-byte vectors) x (token slice of the chunk), the
// last y = beta/decay group. Every input row is read once plus a 3-token halo per
// slice (L2 hits), with coalesced 16-byte loads all issued up front; q/k/v are
// written head-major [H][Ntok][d] for the chunk kernels.
#include <type_traits>

#include "gdn_common.cuh"

namespace gdn {
namespace {

// CTA sizes: 128 threads, or 192 where that leaves no idle warp in the channel
// groups and 128 does not (six 256-channel heads: 1536 q channels = 192 x 8)
constexpr int kThreads = 128;

// ------------------------------------------------------------------ K0
// Packed sequences: validate cu_seqlens and build chunk_off[n] = number of
// 64-token chunks in sequences 0..n-1. A malformed array sets the status word
// and leaves an empty chunk table, so later kernels touch nothing.
__global__ void __launch_bounds__(1024) seqlens_scan_kernel(const int32_t *__restrict__ cu, int N,
                                                            int T, int32_t *__restrict__ chunk_off,
                                                            int32_t *__restrict__ status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x;
    int bad = 0;
    for (int n = tid; n < N; n += blockDim.x)
        if (cu[n + 1] < cu[n]) bad = 1;
    if (tid == 0 && (cu[0] != 0 || cu[N] != T)) bad = 1;
    bad = __syncthreads_or(bad);
    if (bad) {
        for (int n = tid; n <= N; n += blockDim.x) chunk_off[n] = 0;
        if (tid == 0) *status = GDN_ERR_DEVICE_SEQLENS;
        return;
    }
    if (tid == 0) {
        carry_s = 0;
        *status = GDN_OK;
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        const int c = n < N ? (cu[n + 1] - cu[n] + kChunk - 1) / kChunk : 0;
        int x = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            warp_sums[lane] = s;  // inclusive prefix over warps
        }
        __syncthreads();
        const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + carry_s;
        if (n < N) chunk_off[n] = before + x - c;
        __syncthreads();
        if (tid == blockDim.x - 1) carry_s = before + x;
        __syncthreads();
    }
    if (tid == 0) chunk_off[N] = carry_s;
}

struct PrologueArgs {
    Problem p;
    int groups_qk;   // channel groups of q (= of k)
    int groups_v;    // channel groups of v
};

// ------------------------------------------------------------ conv group
// One CTA covers one channel group (128 threads x CPT channels) of one token
// slice (TOKS tokens) of one chunk. Each thread copies the TOKS + 3 rows of its
// channels (16-byte vectors, zero-filled before the sequence start) into shared
// memory with cp.async, all in flight at once without holding registers, then
// runs the 4-tap window over them.
template <int NVEC, int TH> struct ConvShape {
    static constexpr int TOKS = 16 / NVEC;
    static constexpr int ROWS = TOKS + kConvW - 1;
    static constexpr int SLICES = kChunk / TOKS;
    static constexpr size_t SMEM = (size_t)ROWS * NVEC * TH * 16;
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem), "r"(ok ? 16 : 0)
                 : "memory");
}
// wait until at most N of this thread's copy groups are still in flight
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// f(integral_constant<int, U>) for U = 0 .. N-1, unrolled at compile time
template <int U, int N, typename F> __device__ __forceinline__ void static_for(F &&f) {
    if constexpr (U < N) {
        f(std::integral_constant<int, U>{});
        static_for<U + 1, N>(f);
    }
}

template <typename T, int NVEC, bool NORM, bool PRE, int TH>
__device__ __forceinline__ void conv_group(const PrologueArgs &A, const ChunkLoc &c, int gy,
                                           uint4 *stage) {
    constexpr int VEC = Vec16<T>::N;
    constexpr int CPT = NVEC * VEC;           // channels per thread
    constexpr int NP = CPT / 2;               // channel pairs per thread
    constexpr int PV = VEC / 2;               // pairs per 16-byte vector
    using Shape = ConvShape<NVEC, TH>;
    constexpr int TOKS = Shape::TOKS;
    constexpr int ROWS = Shape::ROWS;
    using S = typename Inter<T>::S;
    const Problem &p = A.p;
    const gdn_desc &d = p.d;
    const int tid = threadIdx.x;
    const int slice = gy % Shape::SLICES;
    int g = gy / Shape::SLICES;
    const int t_begin = slice * TOKS;
    if (t_begin >= c.len) return;
    const int ntok = min(TOKS, c.len - t_begin);

    // which tensor / channel range
    const T *src;
    S *dst;
    int64_t sb, st;
    int nch, hd, w_base;
    const int ch_qk = d.Hk * d.dk;
    if (g < A.groups_qk) {
        src = (const T *)p.q_raw; dst = (S *)p.q; sb = d.q_stride_b; st = d.q_stride_t;
        nch = ch_qk; hd = d.dk; w_base = 0;
    } else if ((g -= A.groups_qk) < A.groups_qk) {
        src = (const T *)p.k_raw; dst = (S *)p.k; sb = d.k_stride_b; st = d.k_stride_t;
        nch = ch_qk; hd = d.dk; w_base = ch_qk;
    } else {
        g -= A.groups_qk;
        src = (const T *)p.v_raw; dst = (S *)p.v; sb = d.v_stride_b; st = d.v_stride_t;
        nch = d.Hv * d.dv; hd = d.dv; w_base = 2 * ch_qk;
    }
    const int c0 = g * (TH * CPT) + tid * CPT;
    const bool active = c0 < nch;
    // a warp with no channel has nothing to do (no block barrier follows)
    if (!__any_sync(0xffffffffu, active)) return;
    const int lanes_per_head = hd / CPT;      // <= 32 for q/k by construction

    // rows into shared memory, one copy group per row:
    // stage[(r * NVEC + v) * TH + tid]. Rows before the sequence start are
    // zeros, or the prefix rows (the raw inputs of the three earlier tokens).
    const int64_t first = c.tok0 + t_begin - (kConvW - 1);
    const int64_t brow = p.cu ? 0 : c.n;     // batch row of this sequence
    const T *rp = src + brow * sb + (first - brow * (int64_t)d.T) * st + (active ? c0 : 0);
    const int64_t ch_all = 2 * (int64_t)ch_qk + (int64_t)d.Hv * d.dv;
    const T *pre = PRE ? (const T *)p.conv_prefix + (int64_t)c.n * (kConvW - 1) * ch_all + w_base + (active ? c0 : 0)
                       : nullptr;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const bool in_rows = active && r < ntok + kConvW - 1;
        const bool ok = in_rows && first + r >= c.seq0;
        // prefix row index: 0 = oldest of the three tokens before seq0
        const int64_t pr = first + r - (c.seq0 - (kConvW - 1));
        const bool okp = PRE && in_rows && !ok && pr >= 0;
#pragma unroll
        for (int v = 0; v < NVEC; ++v)
            cp_async16(&stage[(r * NVEC + v) * TH + tid],
                       ok ? (const void *)(rp + r * st + v * VEC)
                          : (okp ? (const void *)(pre + pr * ch_all + v * VEC) : (const void *)src),
                       ok || okp);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    // conv taps of my channels as pairs (overlaps the copies)
    float2 w[NP][kConvW];
    if (active) {
        const T *wp = (const T *)p.conv_w + (int64_t)(w_base + c0) * kConvW;
        float wf[CPT * kConvW];
#pragma unroll
        for (int i = 0; i < CPT * kConvW; i += VEC) load16_f<T>(wp + i, wf + i);
#pragma unroll
        for (int i = 0; i < NP; ++i)
#pragma unroll
            for (int j = 0; j < kConvW; ++j)
                w[i][j] = make_float2(wf[(2 * i) * kConvW + j], wf[(2 * i + 1) * kConvW + j]);
    } else {
#pragma unroll
        for (int i = 0; i < NP; ++i)
#pragma unroll
            for (int j = 0; j < kConvW; ++j) w[i][j] = make_float2(0.f, 0.f);
    }

    auto row = [&](int r, float2 *out) {   // each thread reads only its own rows
#pragma unroll
        for (int v = 0; v < NVEC; ++v) Pairs<T>::unpack(stage[(r * NVEC + v) * TH + tid], out + v * PV);
    };
    const int head = c0 / hd;
    const int dd = c0 - head * hd;
    S *dbase = dst + ((int64_t)head * p.ntok + c.tok0 + t_begin) * hd + dd;
    // q/k of 2-byte activations: hi plane here, lo plane `plane` elements further
    constexpr bool split = NORM && sizeof(S) == 2;
    const int64_t plane = (int64_t)d.Hk * p.ntok * d.dk;

    float2 x3[NP], x2[NP], x1[NP];
    // token u of the slice: the window (x3, x2, x1) plus row u + 3
    auto body = [&](auto uc) {
        constexpr int u = decltype(uc)::value;
        float2 x0[NP], y[NP];
        row(u + kConvW - 1, x0);
        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            float2 acc = mul2(w[i][0], x3[i]);
            acc = fma2(w[i][1], x2[i], acc);
            acc = fma2(w[i][2], x1[i], acc);
            acc = fma2(w[i][3], x0[i], acc);
            // q/k keep ~fp32 precision (hi + lo planes); v is stored at 16 bits
            y[i] = NORM ? silu2_acc(acc) : silu2_act<S>(acc);
            if (NORM) ss2 = fma2(y[i], y[i], ss2);
            x3[i] = x2[i];
            x2[i] = x1[i];
            x1[i] = x0[i];
        }
        if (NORM) {
            float ss = ss2.x + ss2.y;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                if (off < lanes_per_head) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float2 inv = splat2(rsqrtf(ss + d.l2_eps));
#pragma unroll
            for (int i = 0; i < NP; ++i) y[i] = mul2(y[i], inv);
        }
        if (active) {
            uint4 *op = reinterpret_cast<uint4 *>(dbase + (int64_t)u * hd);
#pragma unroll
            for (int v = 0; v < NVEC; ++v) op[v] = Pairs<S>::pack(y + v * PV);
            if (split) {   // lo plane: what fp16 rounding of y left out
                float2 lo[NP];
#pragma unroll
                for (int i = 0; i < NP; ++i) lo[i] = fma2(Pairs<S>::round(y[i]), splat2(-1.0f), y[i]);
                uint4 *lp = reinterpret_cast<uint4 *>(dbase + (int64_t)u * hd + plane);
#pragma unroll
                for (int v = 0; v < NVEC; ++v) lp[v] = Pairs<S>::pack(lo + v * PV);
            }
        }
    };
    // rows 0..2, then token u as soon as row u + 3 has landed
    cp_async_wait<ROWS - 3>();
    row(0, x3);
    row(1, x2);
    row(2, x1);
    static_for<0, TOKS>([&](auto uc) {
        constexpr int u = decltype(uc)::value;
        if (u < ntok) {                       // uniform across the block
            cp_async_wait<TOKS - 1 - u>();
            body(uc);
        }
    });
}

// ------------------------------------------------------- beta/decay group
template <typename T, int TH>
__device__ __forceinline__ void gate_group(const Problem &p, const ChunkLoc &c, float *smem) {
    float (*gs)[33] = reinterpret_cast<float (*)[33]>(smem);
    float (*bs)[33] = reinterpret_cast<float (*)[33]>(smem + kChunk * 33);
    const gdn_desc &d = p.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int h0 = 0; h0 < d.Hv; h0 += 32) {
        const int nh = min(32, d.Hv - h0);
        for (int idx = tid; idx < kChunk * 32; idx += TH) {
            const int i = idx >> 5, hh = idx & 31;
            float gv = 0.f, bv = 0.f;
            if (i < c.len && hh < nh) {
                const int64_t tok = c.tok0 + i;
                const int h = h0 + hh;
                const float av = to_f<T>(((const T *)p.a)[tok_offset(tok, d.T, d.a_stride_b, d.a_stride_t) + h]);
                const float bb = to_f<T>(((const T *)p.b)[tok_offset(tok, d.T, d.b_stride_b, d.b_stride_t) + h]);
                bv = sigmoid_f(bb);
                gv = -expf(p.A_log[h]) * softplus_f(av + p.dt_bias[h]);
            }
            gs[i][hh] = gv;
            bs[i][hh] = bv;
        }
        __syncthreads();
        using GT = typename Inter<T>::G;
        GT *gamma = (GT *)p.gamma;
        for (int hh = warp; hh < nh; hh += TH / 32) {
            const GT g0 = gs[2 * lane][hh], g1 = gs[2 * lane + 1][hh];
            GT x = g0 + g1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const GT y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            const GT excl = x - (g0 + g1);
            const int64_t row = (int64_t)(h0 + hh) * p.ntok + c.tok0;
            if (2 * lane < c.len) {
                gamma[row + 2 * lane] = excl + g0;
                p.beta[row + 2 * lane] = bs[2 * lane][hh];
            }
            if (2 * lane + 1 < c.len) {
                gamma[row + 2 * lane + 1] = excl + g0 + g1;
                p.beta[row + 2 * lane + 1] = bs[2 * lane + 1][hh];
            }
        }
        __syncthreads();
    }
}

template <typename T, int NVEC, bool PRE, int TH>
__global__ void __launch_bounds__(TH) prologue_kernel(const PrologueArgs A) {
    extern __shared__ uint4 stage[];
    pdl_trigger();    // the chunk stage's CTAs may become resident during the last wave
    const Problem &p = A.p;
    if (p.cu == nullptr) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.status = GDN_OK;
    } else if (*p.status != GDN_OK) {
        return;
    }
    ChunkLoc c;
    if (!locate_chunk(blockIdx.x, p.cu, p.chunk_off, p.d.N, p.d.T, c)) return;
    const int gy = blockIdx.y;
    if (gy == (2 * A.groups_qk + A.groups_v) * ConvShape<NVEC, TH>::SLICES) gate_group<T, TH>(p, c, (float *)stage);
    else if (gy < 2 * A.groups_qk * ConvShape<NVEC, TH>::SLICES) conv_group<T, NVEC, true, PRE, TH>(A, c, gy, stage);
    else conv_group<T, NVEC, false, PRE, TH>(A, c, gy, stage);
}

template <typename T, int NVEC, int TH>
cudaError_t launch_th(const Problem &p, cudaStream_t s) {
    constexpr int CPT = NVEC * Vec16<T>::N;
    PrologueArgs A;
    A.p = p;
    const int gc = TH * CPT;
    A.groups_qk = (p.d.Hk * p.d.dk + gc - 1) / gc;
    A.groups_v = (p.d.Hv * p.d.dv + gc - 1) / gc;
    using Shape = ConvShape<NVEC, TH>;
    static_assert(Shape::SMEM >= 2 * kChunk * 33 * 4, "gate group scratch");
    dim3 grid((unsigned)chunk_slots(p), (2 * A.groups_qk + A.groups_v) * Shape::SLICES + 1);
    // the prefix reads are compiled in only where a prefix is given
    auto kernel = p.conv_prefix ? prologue_kernel<T, NVEC, true, TH> : prologue_kernel<T, NVEC, false, TH>;
    if (Shape::SMEM > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Shape::SMEM);
        if (e != cudaSuccess) return e;
    }
    kernel<<<grid, TH, Shape::SMEM, s>>>(A);
    return cudaGetLastError();
}

template <typename T, int NVEC>
cudaError_t launch_t(const Problem &p, cudaStream_t s) {
    constexpr int CPT = NVEC * Vec16<T>::N;
    const int th_qk = p.d.Hk * p.d.dk / CPT, th_v = p.d.Hv * p.d.dv / CPT;   // threads per tensor
    if ((th_qk % 128 != 0 || th_v % 128 != 0) && th_qk % 192 == 0 && th_v % 192 == 0)
        return launch_th<T, NVEC, 192>(p, s);
    return launch_th<T, NVEC, kThreads>(p, s);
}

}  // namespace

cudaError_t launch_seqlens_scan(const Problem &p, cudaStream_t s) {
    seqlens_scan_kernel<<<1, 1024, 0, s>>>(p.cu, p.d.N, p.d.T, p.chunk_off, p.status);
    return cudaGetLastError();
}

// A q/k head must fit in one warp's lanes: channels per thread >= dk / 32.
cudaError_t launch_prologue(const Problem &p, cudaStream_t s) {
    const int need = p.d.dk / 32;
    switch (p.d.dtype) {
    case GDN_F32:
        if (need <= 4) return launch_t<float, 1>(p, s);
        if (need <= 8) return launch_t<float, 2>(p, s);
        return launch_t<float, 4>(p, s);
    case GDN_BF16:
        if (need <= 8) return launch_t<__nv_bfloat16, 1>(p, s);
        return launch_t<__nv_bfloat16, 2>(p, s);
    default:
        if (need <= 8) return launch_t<__half, 1>(p, s);
        return launch_t<__half, 2>(p, s);
    }
}

}  // namespace gdn
