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
#include "gdn_common.cuh"

namespace gdn {
namespace {

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
template <int NVEC> struct ConvShape {
    static constexpr int TOKS = 16 / NVEC;
    static constexpr int ROWS = TOKS + kConvW - 1;
    static constexpr int SLICES = kChunk / TOKS;
    static constexpr size_t SMEM = (size_t)ROWS * NVEC * kThreads * 16;
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem), "r"(ok ? 16 : 0)
                 : "memory");
}

template <typename T, int NVEC, bool NORM>
__device__ __forceinline__ void conv_group(const PrologueArgs &A, const ChunkLoc &c, int gy,
                                           uint4 *stage) {
    constexpr int VEC = Vec16<T>::N;
    constexpr int CPT = NVEC * VEC;           // channels per thread
    using Shape = ConvShape<NVEC>;
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
    bool norm;
    const int ch_qk = d.Hk * d.dk;
    if (g < A.groups_qk) {
        src = (const T *)p.q_raw; dst = (S *)p.q; sb = d.q_stride_b; st = d.q_stride_t;
        nch = ch_qk; hd = d.dk; w_base = 0; norm = true;
    } else if ((g -= A.groups_qk) < A.groups_qk) {
        src = (const T *)p.k_raw; dst = (S *)p.k; sb = d.k_stride_b; st = d.k_stride_t;
        nch = ch_qk; hd = d.dk; w_base = ch_qk; norm = true;
    } else {
        g -= A.groups_qk;
        src = (const T *)p.v_raw; dst = (S *)p.v; sb = d.v_stride_b; st = d.v_stride_t;
        nch = d.Hv * d.dv; hd = d.dv; w_base = 2 * ch_qk; norm = false;
    }
    const int c0 = g * (kThreads * CPT) + tid * CPT;
    const bool active = c0 < nch;
    const int lanes_per_head = hd / CPT;      // <= 32 for q/k by construction
    (void)norm;

    // rows into shared memory: stage[(r * NVEC + v) * kThreads + tid]
    const int64_t first = c.tok0 + t_begin - (kConvW - 1);
    const int64_t brow = p.cu ? 0 : c.n;     // batch row of this sequence
    const T *rp = src + brow * sb + (first - brow * (int64_t)d.T) * st + (active ? c0 : 0);
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const bool ok = active && r < ntok + kConvW - 1 && first + r >= c.seq0;
#pragma unroll
        for (int v = 0; v < NVEC; ++v)
            cp_async16(&stage[(r * NVEC + v) * kThreads + tid], ok ? (const void *)(rp + r * st + v * VEC)
                                                                   : (const void *)src, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // conv taps of my channels (overlaps the copies)
    float w[CPT][kConvW];
    if (active) {
        const T *wp = (const T *)p.conv_w + (int64_t)(w_base + c0) * kConvW;
#pragma unroll
        for (int i = 0; i < CPT * kConvW; i += VEC) {
            float tmp[VEC];
            load16_f<T>(wp + i, tmp);
#pragma unroll
            for (int j = 0; j < VEC; ++j) w[(i + j) / kConvW][(i + j) % kConvW] = tmp[j];
        }
    } else {
#pragma unroll
        for (int i = 0; i < CPT; ++i)
#pragma unroll
            for (int j = 0; j < kConvW; ++j) w[i][j] = 0.f;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");   // each thread reads only its own rows

    auto row = [&](int r, float *out) {
#pragma unroll
        for (int v = 0; v < NVEC; ++v) unpack16<T>(stage[(r * NVEC + v) * kThreads + tid], out + v * VEC);
    };
    float x3[CPT], x2[CPT], x1[CPT];
    row(0, x3);
    row(1, x2);
    row(2, x1);

    const int head = c0 / hd;
    const int dd = c0 - head * hd;
    S *dbase = dst + ((int64_t)head * p.ntok + c.tok0 + t_begin) * hd + dd;
    // q/k of 2-byte activations: hi plane here, lo plane `plane` elements further
    const bool split = NORM && sizeof(S) == 2;
    const int64_t plane = (int64_t)d.Hk * p.ntok * d.dk;

#pragma unroll 4
    for (int u = 0; u < ntok; ++u) {          // uniform across the block
        float x0[CPT], y[CPT];
        row(u + kConvW - 1, x0);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            float acc = w[i][0] * x3[i];
            acc = fmaf(w[i][1], x2[i], acc);
            acc = fmaf(w[i][2], x1[i], acc);
            acc = fmaf(w[i][3], x0[i], acc);
            // q/k keep ~fp32 precision (hi + lo planes); v is stored at 16 bits
            y[i] = NORM ? silu_f(acc) : silu_act<S>(acc);
            ss = fmaf(y[i], y[i], ss);
            x3[i] = x2[i];
            x2[i] = x1[i];
            x1[i] = x0[i];
        }
        if (NORM) {
            for (int off = lanes_per_head >> 1; off >= 1; off >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss + d.l2_eps);
#pragma unroll
            for (int i = 0; i < CPT; ++i) y[i] *= inv;
        }
        if (active) {
            S *op = dbase + (int64_t)u * hd;
#pragma unroll
            for (int v = 0; v < NVEC; ++v) store16_f<S>(op + v * VEC, y + v * VEC);
            if (split) {   // lo plane: what fp16 rounding of y left out
                float lo[CPT];
#pragma unroll
                for (int i = 0; i < CPT; ++i) lo[i] = y[i] - round_through<S>(y[i]);
#pragma unroll
                for (int v = 0; v < NVEC; ++v) store16_f<S>(op + plane + v * VEC, lo + v * VEC);
            }
        }
    }
}

// ------------------------------------------------------- beta/decay group
template <typename T>
__device__ __forceinline__ void gate_group(const Problem &p, const ChunkLoc &c, float *smem) {
    float (*gs)[33] = reinterpret_cast<float (*)[33]>(smem);
    float (*bs)[33] = reinterpret_cast<float (*)[33]>(smem + kChunk * 33);
    const gdn_desc &d = p.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int h0 = 0; h0 < d.Hv; h0 += 32) {
        const int nh = min(32, d.Hv - h0);
        for (int idx = tid; idx < kChunk * 32; idx += kThreads) {
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
        for (int hh = warp; hh < nh; hh += kThreads / 32) {
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

template <typename T, int NVEC>
__global__ void __launch_bounds__(kThreads) prologue_kernel(const PrologueArgs A) {
    extern __shared__ uint4 stage[];
    const Problem &p = A.p;
    if (p.cu == nullptr) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *p.status = GDN_OK;
    } else if (*p.status != GDN_OK) {
        return;
    }
    ChunkLoc c;
    if (!locate_chunk(blockIdx.x, p.cu, p.chunk_off, p.d.N, p.d.T, c)) return;
    const int gy = blockIdx.y;
    if (gy == (2 * A.groups_qk + A.groups_v) * ConvShape<NVEC>::SLICES) gate_group<T>(p, c, (float *)stage);
    else if (gy < 2 * A.groups_qk * ConvShape<NVEC>::SLICES) conv_group<T, NVEC, true>(A, c, gy, stage);
    else conv_group<T, NVEC, false>(A, c, gy, stage);
}

template <typename T, int NVEC>
cudaError_t launch_t(const Problem &p, cudaStream_t s) {
    constexpr int CPT = NVEC * Vec16<T>::N;
    PrologueArgs A;
    A.p = p;
    const int gc = kThreads * CPT;
    A.groups_qk = (p.d.Hk * p.d.dk + gc - 1) / gc;
    A.groups_v = (p.d.Hv * p.d.dv + gc - 1) / gc;
    using Shape = ConvShape<NVEC>;
    static_assert(Shape::SMEM >= 2 * kChunk * 33 * 4, "gate group scratch");
    dim3 grid((unsigned)chunk_slots(p), (2 * A.groups_qk + A.groups_v) * Shape::SLICES + 1);
    if (Shape::SMEM > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(prologue_kernel<T, NVEC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Shape::SMEM);
        if (e != cudaSuccess) return e;
    }
    prologue_kernel<T, NVEC><<<grid, kThreads, Shape::SMEM, s>>>(A);
    return cudaGetLastError();
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
