// gdn_backward_tc.cu -- the dv contractions of the backward's per-chunk
// gradients on the tensor cores (tcgen05, bf16 operands, fp32 accumulators).
//
// Per (chunk slot, v head) the per-chunk gradient kernel needs three products
// over dv (see gdn_backward.cu for the chunk form):
//     X1 = dO' H0^T,  X2 = dR0 H0^T,  X3 = Vn dH1^T      (each 64 x dk)
// Here they are two M = 128 products accumulated in tensor memory:
//     [dO'; dR0] H0^T  -> TMEM columns [0, dk)      (rows 0..63 X1, 64..127 X2)
//     [Vn;  0  ] dH1^T -> TMEM columns [256, 256+dk) (rows 0..63 X3)
// over 64-column blocks of dv. The fp32 operands are rounded to bf16 (fp32's
// exponent range: gradients of any scale) and written by the CTA's threads
// into 128-byte-swizzled K-major tiles; one thread issues the MMAs. The
// results go to the workspace ([slot][Hv][3][64][dk] fp32) together with
// <H0, dH1>, which the same loads give for free. Shapes: dk <= 256, dv a
// multiple of 64; 2-byte activations (fp32 activations keep the fp32 path).
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kXThreads = 128;      // one thread per TMEM lane / tile row
constexpr int kC2 = kChunk * kChunk; // elements of a 64 x 64 chunk matrix

// kind::f16 instruction descriptor with bf16 A and B, fp32 D, both K-major:
// [4,6) D format 1 = f32, [7,10) A format 1 = bf16, [10,13) B format 1 = bf16,
// [17,23) N >> 3, [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void st4f(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

__device__ __forceinline__ uint32_t bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 64 fp32 from src (null: zeros) rounded to bf16 into row r of a swizzled tile
__device__ __forceinline__ void put_row(unsigned char *tile, int r, const float *src) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (src) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(src + 8 * q));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(src + 8 * q + 4));
            u = make_uint4(bf2(a.x, a.y), bf2(a.z, a.w), bf2(b.x, b.y), bf2(b.z, b.w));
        }
        *reinterpret_cast<uint4 *>(tile + sw128_off(r, 8 * q)) = u;
    }
}

// rows r of H0 and dH1 into their tiles, accumulating their dot product
__device__ __forceinline__ void put_rows2(unsigned char *th, unsigned char *tg, int r, const float *h,
                                          const float *g, float &hd) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(h + 8 * q));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(h + 8 * q + 4));
        const float4 c = __ldg(reinterpret_cast<const float4 *>(g + 8 * q));
        const float4 e = __ldg(reinterpret_cast<const float4 *>(g + 8 * q + 4));
        hd = fmaf(a.x, c.x, fmaf(a.y, c.y, fmaf(a.z, c.z, fmaf(a.w, c.w, hd))));
        hd = fmaf(b.x, e.x, fmaf(b.y, e.y, fmaf(b.z, e.z, fmaf(b.w, e.w, hd))));
        *reinterpret_cast<uint4 *>(th + sw128_off(r, 8 * q)) = make_uint4(bf2(a.x, a.y), bf2(a.z, a.w), bf2(b.x, b.y),
                                                                          bf2(b.z, b.w));
        *reinterpret_cast<uint4 *>(tg + sw128_off(r, 8 * q)) = make_uint4(bf2(c.x, c.y), bf2(c.z, c.w), bf2(e.x, e.y),
                                                                          bf2(e.z, e.w));
    }
}

__global__ void __launch_bounds__(kXThreads, 1) chunk_x_kernel(const BwdProblem bp) {
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ float red[kXThreads / 32];
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
    unsigned char *A12 = sm, *A3 = sm + 16384, *BH = sm + 32768, *BD = BH + dk * 128;
    const int t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(&tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    const float *dOg = bp.dO + ((size_t)j * p.ntok + tok0) * dv;
    const float *dRg = bp.dR + ((size_t)j * p.ntok + tok0) * dv;
    const float *Vng = bp.vn + ((size_t)j * p.ntok + tok0) * dv;
    const float *H0 = bp.h0 + ((size_t)slot * Hv + j) * dk * dv;
    const float *dH1 = bp.dh1 + ((size_t)slot * Hv + j) * dk * dv;
    const uint32_t idesc = idesc_bf16(128, dk);
    const uint64_t da12 = sw128_desc(smem_u32(A12), 16, 1024), da3 = sw128_desc(smem_u32(A3), 16, 1024);
    const uint64_t dbh = sw128_desc(smem_u32(BH), 16, 1024), dbd = sw128_desc(smem_u32(BD), 16, 1024);
    float hd = 0.f;
    if (t >= 64) put_row(A3, t, nullptr);     // rows 64..127 of [Vn; 0] stay zero
    bool ok = true;
    int step = 0;
    for (int kb = 0; kb < dv; kb += 64, ++step) {
        const int i = t & 63;
        put_row(A12, t, i < L ? (t < 64 ? dOg : dRg) + (int64_t)i * dv + kb : nullptr);
        if (t < 64) put_row(A3, t, t < L ? Vng + (int64_t)t * dv + kb : nullptr);
        for (int r = t; r < dk; r += kXThreads)
            put_rows2(BH, BD, r, H0 + (size_t)r * dv + kb, dH1 + (size_t)r * dv + kb, hd);
        fence_async_smem();                   // the tiles are read by the tensor cores
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {   // K = 16 per MMA: the start advances 32 bytes
                mma_f16(tbase, da12 + 2 * ks, dbh + 2 * ks, idesc, (kb | ks) != 0);
                mma_f16(tbase + 256, da3 + 2 * ks, dbd + 2 * ks, idesc, (kb | ks) != 0);
            }
            mma_commit(&bar);
        }
        // every thread waits for the products before the tiles are rewritten
        const bool done = mbar_wait(&bar, (uint32_t)step & 1);
        fence_after_sync();
        if (__syncthreads_or(!done)) {
            ok = false;
            break;
        }
    }
    if (ok) {
        float *X = bp.xbuf + ((size_t)slot * Hv + j) * 3 * 64 * dk;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float *row12 = t < 64 ? X + (size_t)t * dk : X + 64 * (size_t)dk + (size_t)(t - 64) * dk;
        for (int c = 0; c < dk; c += 32) {
            float v[32];
            tmem_ld32(tbase + lane_off + c, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) st4f(row12 + c + 4 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            if (warp < 2) {                    // rows 0..63 of the second product
                tmem_ld32(tbase + 256 + lane_off + c, v);
                float *row3 = X + 128 * (size_t)dk + (size_t)t * dk + c;
#pragma unroll
                for (int q = 0; q < 8; ++q) st4f(row3 + 4 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, off);
        if ((t & 31) == 0) red[warp] = hd;
    } else {
        // the products did not complete in time: report, wait (bounded) once more
        // for what is in flight, then free the tensor memory
        if (t == 0) *p.status = GDN_ERR_DEVICE_TIMEOUT;
        mbar_wait(&bar, (uint32_t)step & 1);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (ok && t == 0) bp.hdbuf[(size_t)slot * Hv + j] = red[0] + red[1] + red[2] + red[3];
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------ outputs O
// O = scale ((diag(e^gam) Q) H0 + Pm Vn) of a (chunk slot, v head) as one
// tensor-memory accumulation (M = 128: rows 0..63 the chunk's tokens, 64..127
// zero): A K-major (e^gam Q over 64-wide dk blocks, then Pm), B MN-major (rows
// of H0, then Vn; dv in 64-column blocks 8 KB apart), N = dv in MMAs of at
// most 256 columns. fp16 operands: these are forward quantities of bounded
// size (unit-norm q, the state, the new values), where fp16's three extra
// mantissa bits over bf16 keep O close to the forward's. Writes o (fp32,
// [Hv][ntok][dv]) for the RMSNorm backward.
constexpr int kOThreads = 256;

__device__ __forceinline__ uint32_t h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 8 fp32 at src (16-byte aligned) -> fp16 into a 128-byte-swizzled tile
__device__ __forceinline__ void put8(unsigned char *dst, const float *src, float scale) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(src + 4));
    *reinterpret_cast<uint4 *>(dst) = make_uint4(h2(scale * a.x, scale * a.y), h2(scale * a.z, scale * a.w),
                                                 h2(scale * b.x, scale * b.y), h2(scale * b.z, scale * b.w));
}

__global__ void __launch_bounds__(kOThreads, 1) out_tc_kernel(const BwdProblem bp) {
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ float egs[kChunk];
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
    unsigned char *At = sm, *Bt = sm + 16384;          // A: 128 x 64 K-major; B: 64 K-rows x dv MN-major
    const int t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    if (t < kChunk) {
        const int i = t < L ? t : L - 1;
        egs[t] = expf(((const float *)p.gamma)[(int64_t)j * p.ntok + tok0 + i]);
    }
    if (warp == 0) tmem_alloc(&tslot, 512);
    // rows 64..127 of A are zero for every product
    for (int idx = t; idx < 64 * 8; idx += kOThreads)
        *reinterpret_cast<uint4 *>(At + sw128_off(64 + idx / 8, 8 * (idx % 8))) = make_uint4(0u, 0u, 0u, 0u);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    const __half *qh = (const __half *)p.q + ((int64_t)hk * p.ntok + tok0) * dk;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const float *H0 = bp.h0 + ((size_t)slot * Hv + j) * dk * dv;
    const float *Pm = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2 + kC2;
    const float *Vng = bp.vn + ((size_t)j * p.ntok + tok0) * dv;
    const int nmma = dv > 256 ? 2 : 1, nw = dv > 256 ? 256 : dv;
    const uint32_t idesc = idesc_f16(128, nw, false, true);   // fp16 A K-major, B MN-major
    const uint64_t da = sw128_desc(smem_u32(At), 16, 1024), db = sw128_desc(smem_u32(Bt), 8192, 1024);
    // B tile: rows kr of src (row stride dv; null rows beyond nrows) into the MN-major layout
    auto put_b = [&](const float *src, int nrows) {
        for (int idx = t; idx < 64 * (dv / 8); idx += kOThreads) {
            const int kr = idx / (dv / 8), n0 = 8 * (idx % (dv / 8));
            unsigned char *dst = Bt + (n0 / 64) * 8192 + sw128_off(kr, n0 % 64);
            if (kr < nrows) put8(dst, src + (int64_t)kr * dv + n0, 1.f);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    bool ok = true;
    const int steps = dk / 64 + 1;                     // dk blocks of (e^gam Q) H0, then Pm Vn
    for (int st = 0; st < steps && ok; ++st) {
        if (st < steps - 1) {
            const int kb = 64 * st;
            for (int idx = t; idx < 64 * 8; idx += kOThreads) {   // e^gam Q, rows 0..63
                const int i = idx / 8, c = 8 * (idx % 8);
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (i < L) {
                    float h[8], l[8];
                    unpack16<__half>(*reinterpret_cast<const uint4 *>(qh + (int64_t)i * dk + kb + c), h);
                    unpack16<__half>(*reinterpret_cast<const uint4 *>(qh + (int64_t)i * dk + kb + c + plane), l);
                    const float e = egs[i];
                    u = make_uint4(h2(e * (h[0] + l[0]), e * (h[1] + l[1])), h2(e * (h[2] + l[2]), e * (h[3] + l[3])),
                                   h2(e * (h[4] + l[4]), e * (h[5] + l[5])), h2(e * (h[6] + l[6]), e * (h[7] + l[7])));
                }
                *reinterpret_cast<uint4 *>(At + sw128_off(i, c)) = u;
            }
            put_b(H0 + (size_t)kb * dv, 64);
        } else {
            for (int idx = t; idx < 64 * 8; idx += kOThreads) {   // Pm
                const int i = idx / 8, c = 8 * (idx % 8);
                put8(At + sw128_off(i, c), Pm + i * kChunk + c, 1.f);
            }
            put_b(Vng, L);
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                for (int h = 0; h < nmma; ++h)
                    mma_f16(tbase + 256 * h, da + 2 * ks, db + (uint64_t)((2048 * ks + 32768 * h) >> 4), idesc,
                            (st | ks) != 0);
            mma_commit(&bar);
        }
        const bool done = mbar_wait(&bar, (uint32_t)st & 1);
        fence_after_sync();
        if (__syncthreads_or(!done)) ok = false;
    }
    if (ok) {
        // rows 0..63: warps 0, 1 (columns of the first half) and 4, 5 (second half)
        const int q4 = warp & 3, half = warp >> 2;
        if (q4 < 2) {
            const int i = 32 * q4 + (t & 31);
            const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
            for (int c = half * (dv / 2); c < (half + 1) * (dv / 2); c += 32) {
                float v[32];
                tmem_ld32(tbase + lane_off + c, v);
                if (i < L) {
                    float *dst = bp.dO + ((size_t)j * p.ntok + tok0 + i) * dv + c;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st4f(dst + 4 * q, d.scale * v[4 * q], d.scale * v[4 * q + 1], d.scale * v[4 * q + 2],
                             d.scale * v[4 * q + 3]);
                }
            }
        }
    } else {
        if (t == 0) *p.status = GDN_ERR_DEVICE_TIMEOUT;
        mbar_wait(&bar, (uint32_t)(steps - 1) & 1);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------ dO' terms
// U = (diag(e^gam) Q)^T dO' ([dk][dv] per chunk slot and v head) and
// W = Pm^T dO' ([64][dv] rows of the chunk's tokens): both contract over the
// chunk's 64 tokens, so B = dO' (64 token rows x dv, MN-major) is built once and
// each 128-row block of U, then W, is one tensor-memory product. The A
// operands are the transposes of token-major data, i.e. MN-major tiles whose
// rows are tokens (64 M columns per 8 KB block). dO' is a gradient (any scale),
// so the operands are bf16, each split into hi = bf16(x) and lo = bf16(x - hi):
// hi.hi + hi.lo + lo.hi carries about 16 significant bits (W and U feed the
// reverse chain directly).

// x -> (hi, lo) bf16 pairs of two values
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}
__device__ __forceinline__ void split8(const float *v, uint4 &hi, uint4 &lo) {
    split2(v[0], v[1], hi.x, lo.x);
    split2(v[2], v[3], hi.y, lo.y);
    split2(v[4], v[5], hi.z, lo.z);
    split2(v[6], v[7], hi.w, lo.w);
}

__global__ void __launch_bounds__(kOThreads, 1) dterms_tc_kernel(const BwdProblem bp) {
    extern __shared__ unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ float egs[kChunk];
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
    // A hi / lo: 64 token rows x 128 M (two 8 KB blocks each); B hi / lo: 64 x dv
    unsigned char *Ah = sm, *Al = sm + 16384, *Bh = sm + 32768, *Bl = Bh + 64 * (size_t)dv * 2;
    const int t = threadIdx.x, warp = t >> 5;
    if (t == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    if (t < kChunk) {
        const int i = t < L ? t : L - 1;
        egs[t] = expf(((const float *)p.gamma)[(int64_t)j * p.ntok + tok0 + i]);
    }
    if (warp == 0) tmem_alloc(&tslot, 512);
    // B = dO' rows (tokens i < L), MN-major
    const float *dOg = bp.dO + ((size_t)j * p.ntok + tok0) * dv;
    for (int idx = t; idx < 64 * (dv / 8); idx += kOThreads) {
        const int kr = idx / (dv / 8), n0 = 8 * (idx % (dv / 8));
        uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
        if (kr < L) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(dOg + (int64_t)kr * dv + n0));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(dOg + (int64_t)kr * dv + n0 + 4));
            const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            split8(v, hi, lo);
        }
        const uint32_t off = (n0 / 64) * 8192 + sw128_off(kr, n0 % 64);
        *reinterpret_cast<uint4 *>(Bh + off) = hi;
        *reinterpret_cast<uint4 *>(Bl + off) = lo;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tslot;
    const __half *qh = (const __half *)p.q + ((int64_t)hk * p.ntok + tok0) * dk;
    const int64_t plane = (int64_t)d.Hk * p.ntok * dk;
    const float *Pm = bp.mats + ((size_t)slot * Hv + j) * 3 * kC2 + kC2;
    float *U = bp.uq + ((size_t)slot * Hv + j) * dk * dv;
    const int nmma = dv > 256 ? 2 : 1, nw = dv > 256 ? 256 : dv;
    const uint32_t idesc = idesc_bf16(128, nw) | (1u << 15) | (1u << 16);   // A and B MN-major
    const uint64_t dah = sw128_desc(smem_u32(Ah), 8192, 1024), dal = sw128_desc(smem_u32(Al), 8192, 1024);
    const uint64_t dbh = sw128_desc(smem_u32(Bh), 8192, 1024), dbl = sw128_desc(smem_u32(Bl), 8192, 1024);
    const int ublocks = (dk + 127) / 128;
    bool ok = true;
    for (int blk = 0; blk <= ublocks && ok; ++blk) {
        const bool isw = blk == ublocks;                // the last block is W
        // A rows = tokens (K), 128 M columns: dk indices [128 blk, +128) of e^gam Q, or Pm^T rows
        for (int idx = t; idx < 64 * 16; idx += kOThreads) {
            const int kr = idx / 16, m0 = 8 * (idx % 16);
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (isw) {
                if (m0 < kChunk) {                      // Pm^T: A[m][i] = Pm[m][i], row m of Pm
                    const float4 a = __ldg(reinterpret_cast<const float4 *>(Pm + kr * kChunk + m0));
                    const float4 b = __ldg(reinterpret_cast<const float4 *>(Pm + kr * kChunk + m0 + 4));
                    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
                }
            } else {
                const int dd = 128 * blk + m0;
                if (kr < L && dd < dk) {
                    float h[8], l[8];
                    unpack16<__half>(*reinterpret_cast<const uint4 *>(qh + (int64_t)kr * dk + dd), h);
                    unpack16<__half>(*reinterpret_cast<const uint4 *>(qh + (int64_t)kr * dk + dd + plane), l);
                    const float e = egs[kr];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = e * (h[u] + l[u]);
                }
            }
            uint4 hi, lo;
            split8(v, hi, lo);
            const uint32_t off = (m0 / 64) * 8192 + sw128_off(kr, m0 % 64);
            *reinterpret_cast<uint4 *>(Ah + off) = hi;
            *reinterpret_cast<uint4 *>(Al + off) = lo;
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)             // K = 16 tokens per MMA: 2048 bytes per step
                for (int h = 0; h < nmma; ++h) {
                    const uint64_t ak = (uint64_t)((2048 * ks) >> 4), bk = (uint64_t)((2048 * ks + 32768 * h) >> 4);
                    mma_f16(tbase + 256 * h, dah + ak, dbh + bk, idesc, ks != 0);
                    mma_f16(tbase + 256 * h, dah + ak, dbl + bk, idesc, 1);
                    mma_f16(tbase + 256 * h, dal + ak, dbh + bk, idesc, 1);
                }
            mma_commit(&bar);
        }
        const bool done = mbar_wait(&bar, (uint32_t)blk & 1);
        fence_after_sync();
        if (__syncthreads_or(!done)) {
            ok = false;
            break;
        }
        // read out: row = TMEM lane (warp % 4), columns split between warps < 4 and >= 4
        const int q4 = warp & 3, half = warp >> 2;
        const int row = 32 * q4 + (t & 31);
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool useful = isw ? q4 < 2 : 128 * blk + 32 * q4 < dk;   // warp-uniform
        if (useful) {
            for (int c = half * (dv / 2); c < (half + 1) * (dv / 2); c += 32) {
                float v[32];
                tmem_ld32(tbase + lane_off + c, v);
                float *dst = nullptr;
                if (isw) {
                    if (row < L) dst = bp.wv + ((size_t)j * p.ntok + tok0 + row) * dv + c;
                } else {
                    dst = U + (size_t)(128 * blk + row) * dv + c;
                }
                if (dst) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) st4f(dst + 4 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
        }
        // the tensor-memory reads are done before the next block's products
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    if (!ok) {
        if (t == 0) *p.status = GDN_ERR_DEVICE_TIMEOUT;
        mbar_wait(&bar, (uint32_t)ublocks & 1);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace

bool dterms_tc_supports(const gdn_desc &d) {
    return d.dtype != GDN_F32 && d.dk % 64 == 0 && d.dv % 64 == 0 && d.dv <= 512 && d.dv >= 64;
}

cudaError_t launch_dterms_tc(const BwdProblem &bp, int64_t slots, cudaStream_t s) {
    const gdn_desc &d = bp.f.d;
    const size_t bytes = 1024 + 32768 + 2 * 64 * (size_t)d.dv * 2;
    cudaError_t e = cudaFuncSetAttribute(dterms_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dterms_tc_kernel<<<dim3((unsigned)slots, d.Hv), kOThreads, bytes, s>>>(bp);
    return cudaGetLastError();
}

bool out_tc_supports(const gdn_desc &d) {
    return d.dtype != GDN_F32 && d.dk % 64 == 0 && d.dv % 64 == 0 && d.dv <= 512 && d.dv >= 64;
}

cudaError_t launch_out_tc(const BwdProblem &bp, int64_t slots, cudaStream_t s) {
    const gdn_desc &d = bp.f.d;
    const size_t bytes = 1024 + 16384 + 64 * (size_t)d.dv * 2;
    cudaError_t e = cudaFuncSetAttribute(out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    out_tc_kernel<<<dim3((unsigned)slots, d.Hv), kOThreads, bytes, s>>>(bp);
    return cudaGetLastError();
}

bool chunk_x_tc_supports(const gdn_desc &d) {
    return d.dtype != GDN_F32 && (d.dk == 64 || d.dk == 128 || d.dk == 256) && d.dv % 64 == 0;
}

cudaError_t launch_chunk_x_tc(const BwdProblem &bp, int64_t slots, cudaStream_t s) {
    const gdn_desc &d = bp.f.d;
    const size_t bytes = 1024 + 32768 + 2 * (size_t)d.dk * 128;
    cudaError_t e = cudaFuncSetAttribute(chunk_x_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    chunk_x_kernel<<<dim3((unsigned)slots, d.Hv), kXThreads, bytes, s>>>(bp);
    return cudaGetLastError();
}

}  // namespace gdn
