// gdn_chunk_tc.cu -- chunked gated delta rule on the tcgen05 tensor cores
// (bf16/fp16 activations; fp16 operands, fp32 accumulators in tensor memory).
//
// Per chunk of 64 tokens (gam = in-chunk cumulative decay, H = S^T [dk][dv]):
//   A   = strict_lower( beta_i exp(gam_i - gam_j) k_i.k_j ),  P = lower( exp(gam_i - gam_j) q_i.k_j )
//   T   = (I + A)^{-1}
//   R   = diag(beta) (V - diag(exp(gam)) K H)
//   [Vn; P Vn] = [T; P T] R
//   O   = diag(exp(gam)) Q H + P Vn
//   H  <- exp(gam_L) H + K^T diag(exp(gam_L - gam)) Vn
// Two kernels:
//  * prep (one CTA per chunk and v head, fully parallel): [K;Q] K^T on the
//    tensor cores in split precision (q and k arrive as fp16 hi + lo planes;
//    hi*hi + hi*lo + lo*hi recovers ~fp32 dot products, which the output RMSNorm
//    needs for nearly orthogonal q, k), decay masks, the 64x64 unit-triangular
//    solve on CUDA cores in fp32, then P T on the tensor cores. Writes the
//    [T; P T] tile (128 x 64 fp16, 16 KB) already in the 128-byte-swizzled
//    layout, so the chain kernel fetches it with one bulk copy. For the
//    transposed chain (gdn_chain_tm.cu) the per-token factors of the row
//    updates and the output scale are folded into the tile instead:
//    [diag(e^{gam_L - gam}) T diag(beta); scale P T diag(beta)], whose product
//    with V - diag(e^gam) K H is [Vn'; scale P Vn].
//  * chain (one CTA of 8 warps per sequence, v head and 64-column dv tile): the
//    state slice H [dk][64] stays in registers in fp32 across chunks (warps w
//    and w+4 read the same tensor-memory lanes and split the columns; an fp16
//    copy in shared memory feeds the next MMA); per chunk three dependent MMAs
//    [K; Q] H, [T; P T] R and dH = K^T Vn', then H = e^{gam_L} H + dH. Inputs of
//    chunk c+1 (and c+2) are fetched by TMA while chunk c computes.
// Every wait on an mbarrier gives up after about a second; the kernel then
// records GDN_ERR_DEVICE_TIMEOUT in the status word, waits (bounded) for its own
// copies and MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int LDA = kChunk + 1;

struct PrepMaps {
    CUtensorMap q_hi, q_lo, k_hi, k_lo;
};
struct ChainMaps {
    CUtensorMap q_hi, k_hi, v;
};

__device__ __forceinline__ void set_timeout(const Problem &p) {
    atomicCAS(p.status, GDN_OK, GDN_ERR_DEVICE_TIMEOUT);
}

// 32 columns [c0, c0 + 32) of a swizzled tile row, fp32 -> fp16
__device__ __forceinline__ void store_half_row_f16(unsigned char *tile, int row, int c0, const float *v32) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u;
        __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v32[8 * c + 2 * e], v32[8 * c + 2 * e + 1]);
        *reinterpret_cast<uint4 *>(tile + sw128_off(row, c0 + 8 * c)) = u;
    }
}
// 32 fp32 to a 16-byte-aligned global row slice
__device__ __forceinline__ void store_row_f32(float *dst, const float *v32) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_float4(v32[4 * q], v32[4 * q + 1], v32[4 * q + 2], v32[4 * q + 3]);
}

// ================================================================ prep kernel
// One CTA per (q/k head, chunk slot): the products of the chunk's keys and
// queries are shared by the v heads of the q/k head (GQA), so they are loaded
// and multiplied once; the decay masks, the solve and P T are per v head.
constexpr int kPrepThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;   // 8 warps: warps w and w+4 share TMEM lanes, split columns
constexpr int kLdc = kChunk + 4;    // column stride of A (column-major, 16-byte aligned columns)
// v heads solved per pass (the solve scratch holds this many), a template
// parameter of the kernel. One keeps the CTA's shared memory at ~58 KB and its
// TMEM at 128 columns, so that three CTAs share an SM and hide each other's copy
// and barrier latency; two heads per pass under GQA (two CTAs per SM) measured
// slower on the packed workload (6.55 against 5.83 ms for the chunk stage).

struct PrepSmem {
    int blocks;            // dk / 64
    int bpp;               // dk blocks per load phase (operand buffers hold bpp blocks: one)
    size_t hi, lo, kp, Ac, Ts, Ws, tp, gam, bet, bars, total;
    __host__ __device__ PrepSmem(int dk, int ph) {
        blocks = dk / 64;
        bpp = 1;                                     // 40 KB of operands per phase
        size_t o = 0;
        hi = o; o += (size_t)bpp * 2 * kTileBytes;
        lo = o; o += (size_t)bpp * 2 * kTileBytes;
        kp = o; o += (size_t)bpp * kTileBytes;       // K of the previous chunk (hi)
        // the solve's fp32 scratch reuses the operand buffers once S1 and X are done:
        // A (column-major), T (row-major), W = A21 T11 (row-major 32x33), per v head
        Ac = 0;
        Ts = Ac + (size_t)ph * kChunk * kLdc * 4;
        Ws = Ts + (size_t)ph * kChunk * LDA * 4;
        const size_t solve_end = Ws + (size_t)ph * 32 * 33 * 4;
        if (solve_end > o) o = solve_end;
        o = (o + 1023) & ~(size_t)1023;
        // the [T; P] tile over A's scratch (A is dead once T21 is formed; T stays)
        tp = 0;
        gam = o; o += ph * kChunk * 4;
        bet = o; o += ph * kChunk * 4;
        bars = o; o += 64;
        total = o + 1024;    // slack for aligning the base to 1024 B
    }
};

// IMM: the test mode of the waits (gdn_set_wait_test_mode), a separate instance so
// that the normal one carries nothing of it. FOLD: the tile with beta and
// e^{gam_L - gam} folded in, for the transposed chain. MINB: CTAs per SM the
// registers allow: four (64 registers) when the prep has the GPU to itself, three
// (80 registers, fewer spills) beside a chain segment, where four CTAs slowed the
// chain through the memory system more than they sped the prep.
template <int PH, bool IMM, bool FOLD, int MINB>
__global__ void __launch_bounds__(kPrepThreads, MINB) chunk_prep_kernel(const __grid_constant__ PrepMaps maps,
                                                                     const Problem p, int64_t nslots,
                                                                     unsigned char *tpt, int64_t slot_base) {
    extern __shared__ unsigned char smraw[];
    pdl_wait();       // the prologue's q, k, beta, gamma (and status) are complete
    pdl_trigger();
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const gdn_desc &d = p.d;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & 127;                 // TMEM lane = tile row
    const int c0 = (tid >> 7) * 32;            // its 32 of the 64 columns
    const int hk = blockIdx.y;
    const int G = d.Hv / d.Hk;
    const int64_t slot = blockIdx.x + slot_base;   // a segment's slots start at slot_base
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    ChunkLoc c;
    if (!locate_chunk(slot, p.cu, p.chunk_off, d.N, d.T, c)) return;
    constexpr int kPassHeads = PH;
    const PrepSmem L(d.dk, PH);
    unsigned char *hi = sm + L.hi, *lo = sm + L.lo, *kp = sm + L.kp, *tp = sm + L.tp;
    float *Ac = (float *)(sm + L.Ac), *Ts = (float *)(sm + L.Ts), *Ws = (float *)(sm + L.Ws);
    float *gam = (float *)(sm + L.gam), *bet = (float *)(sm + L.bet);
    uint64_t *bar_load = (uint64_t *)(sm + L.bars), *bar_mma = bar_load + 1;
    uint32_t *tslot = (uint32_t *)(bar_load + 2);
    __shared__ volatile int s_err;
    const bool has_prev = c.tok0 > c.seq0;     // not the first chunk of its sequence
    // per v head: [T; P T] then X (X is written for the first v head of the group only)
    auto out_of = [&](int jv) { return tpt + ((int64_t)jv * nslots + slot) * kPrepOut; };

    if (tid == 0) {
        s_err = 0;
        mbar_init(bar_load, 1);
        mbar_init(bar_mma, 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(tslot, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t lane_addr = tbase + ((uint32_t)((warp & 3) * 32) << 16) + c0;
    const int nphase = L.blocks / L.bpp;
    uint32_t load_phase = 0, mma_phase = 0;
    bool load_out = false, mma_out = false;
    // cumulative decay and beta of v heads g0, g0 + 1 of the group (their global
    // loads overlap the operand copies for the first pass)
    auto load_gb = [&](int g0) {
        if (tid < kPassHeads * kChunk) {
            const int h = tid >> 6, i = tid & (kChunk - 1);
            if (g0 + h < G) {
                const int64_t base = (int64_t)(hk * G + g0 + h) * p.ntok + c.tok0;
                // kept as gam * log2(e): every mask entry is then one ex2 of a difference
                gam[tid] = ((const float *)p.gamma)[base + (i < c.len ? i : c.len - 1)] * kLog2e;
                bet[tid] = i < c.len ? p.beta[base + i] : 0.f;
            }
        }
    };
    load_gb(0);

    // S1 = [Kh;Qh] Kh^T + [Kh;Qh] Kl^T + [Kl;Ql] Kh^T  -> TMEM cols [0, 64), and
    // X = [Kh;Qh] Kh_prev^T -> cols [64, 128) (later reused by P T), dk blocks streamed through the
    // operand buffers bpp at a time
    for (int ph = 0; ph < nphase; ++ph) {
        if (tid == 0) {
            mbar_expect_tx(bar_load, (uint32_t)L.bpp * (has_prev ? 5 : 4) * kTileBytes);
            const int y = (int)((int64_t)hk * p.ntok + c.tok0);
            for (int q = 0; q < L.bpp; ++q) {
                const int b = ph * L.bpp + q;
                tma_load_2d(hi + q * 2 * kTileBytes, &maps.k_hi, 64 * b, y, bar_load);
                tma_load_2d(hi + q * 2 * kTileBytes + kTileBytes, &maps.q_hi, 64 * b, y, bar_load);
                tma_load_2d(lo + q * 2 * kTileBytes, &maps.k_lo, 64 * b, y, bar_load);
                tma_load_2d(lo + q * 2 * kTileBytes + kTileBytes, &maps.q_lo, 64 * b, y, bar_load);
                if (has_prev) tma_load_2d(kp + q * kTileBytes, &maps.k_hi, 64 * b, y - kChunk, bar_load);
            }
        }
        load_out = true;
        if (!mbar_wait(bar_load, load_phase & 1, IMM)) s_err = 1;
        load_phase++;
        __syncthreads();
        if (s_err) goto cleanup;
        load_out = false;
        if (tid == 0) {
            const uint32_t id = idesc_f16(128, 64, false, false);
            // descriptors built once; a K step adds 32 bytes (2 in the start field)
            const uint64_t dh = sw128_desc(smem_u32(hi), 16, 1024), dl = sw128_desc(smem_u32(lo), 16, 1024);
            const uint64_t dp = sw128_desc(smem_u32(kp), 16, 1024);
            for (int q = 0; q < L.bpp; ++q)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t off = (uint64_t)((q * 2 * kTileBytes) >> 4) + 2 * ks;
                    const uint64_t ah = dh + off, al = dl + off;
                    mma_f16(tbase, ah, ah, id, (ph | q | ks) != 0);
                    mma_f16(tbase, ah, al, id, 1);
                    mma_f16(tbase, al, ah, id, 1);
                    if (has_prev)
                        mma_f16(tbase + 64, ah, dp + (uint64_t)((q * kTileBytes) >> 4) + 2 * ks, id, (ph | q | ks) != 0);
                }
            mma_commit(bar_mma);
        }
        mma_out = true;
        // the buffers are reused by the next phase (and by the solve) once these MMAs are done
        if (!mbar_wait(bar_mma, mma_phase & 1, IMM)) s_err = 1;
        mma_phase++;
        __syncthreads();
        if (s_err) goto cleanup;
        mma_out = false;
    }
    fence_after_sync();

    if (has_prev) {   // X -> workspace, fp16, already in the 128-byte-swizzled tile layout
        float v[32];
        tmem_ld32(lane_addr + 64, v);
        unsigned char *xo = out_of(hk * G) + kTPTBytes;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 u;
            __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
            *reinterpret_cast<uint4 *>(xo + sw128_off(row, c0 + 8 * q)) = u;
        }
    }
    // S1 stays in TMEM cols [0, 64) for every v head of the group

    for (int g0 = 0; g0 < G; g0 += kPassHeads) {
        const int nh = G - g0 < kPassHeads ? G - g0 : kPassHeads;
        if (g0 > 0) load_gb(g0);
        __syncthreads();
        // A = beta_i e^{gam_i - gam_j} k_i.k_j below the diagonal, stored column-major
        if (row < kChunk) {
            float s1[32];
            tmem_ld32(lane_addr, s1);
            for (int h = 0; h < nh; ++h) {
                const float gi = gam[h * kChunk + row], bi = bet[h * kChunk + row];
                float *Ah = Ac + h * kChunk * kLdc;
                const float4 *g4 = reinterpret_cast<const float4 *>(gam + h * kChunk + c0);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 gj = g4[q4];
                    const float gv[4] = {gj.x, gj.y, gj.z, gj.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q = 4 * q4 + e, jj = c0 + q;
                        Ah[jj * kLdc + row] = jj < row ? bi * ex2_approx(gi - gv[e]) * s1[q] : 0.f;
                    }
                }
            }
        }
        __syncthreads();
        // T = (I + A)^{-1} in two levels. The 32x32 diagonal blocks first: one warp
        // per (v head, block), thread jc solving column jc by forward substitution
        // with the column in registers; after step m, row m is final and updates
        // the rows below it with column m of A (the same address for every thread).
        if (tid < nh * kChunk) {
            const int h = tid >> 6, b = (tid >> 5) & 1, jc = tid & 31;
            const float *Ab = Ac + h * kChunk * kLdc + 32 * b * kLdc + 32 * b;
            float2 acc[16];                    // rows 2k, 2k + 1 of the block
#pragma unroll
            for (int k = 0; k < 16; ++k) acc[k] = make_float2(2 * k == jc ? 1.f : 0.f, 2 * k + 1 == jc ? 1.f : 0.f);
#pragma unroll
            for (int m = 0; m < 31; ++m) {
                const float tm = (m & 1) ? acc[m >> 1].y : acc[m >> 1].x;
                const float2 nt = make_float2(-tm, -tm);
                const float4 *col = reinterpret_cast<const float4 *>(Ab + m * kLdc);
                // rows up to m hold A = 0 in this column, so whole float4 groups are safe
#pragma unroll
                for (int q = (m + 1) >> 2; q < 8; ++q) {
                    const float4 a = col[q];
                    acc[2 * q] = fma2(make_float2(a.x, a.y), nt, acc[2 * q]);
                    acc[2 * q + 1] = fma2(make_float2(a.z, a.w), nt, acc[2 * q + 1]);
                }
            }
            float *Th = Ts + h * kChunk * LDA + 32 * b * LDA + 32 * b;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                Th[(2 * k) * LDA + jc] = acc[k].x;
                Th[(2 * k + 1) * LDA + jc] = acc[k].y;
                if (b == 0) {                  // the upper right block of T is zero
                    Th[(2 * k) * LDA + 32 + jc] = 0.f;
                    Th[(2 * k + 1) * LDA + 32 + jc] = 0.f;
                }
            }
        }
        __syncthreads();
        // ... then T21 = -T22 (A21 T11): two 32x32x32 products, each thread a 4x2 tile
        const int mt = tid & 127, mh = tid >> 7;
        const int i0 = (mt >> 4) * 4, j0 = (mt & 15) * 2;
        if (mh < nh) {                         // W = A21 T11 (T11 is zero above its diagonal)
            const float *Ah = Ac + mh * kChunk * kLdc;
            const float *Th = Ts + mh * kChunk * LDA;
            float2 w[4] = {};
#pragma unroll 8
            for (int k = 0; k < 32; ++k) {
                const float4 a = *reinterpret_cast<const float4 *>(Ah + k * kLdc + 32 + i0);
                const float2 t = make_float2(Th[k * LDA + j0], Th[k * LDA + j0 + 1]);
                w[0] = fma2(make_float2(a.x, a.x), t, w[0]);
                w[1] = fma2(make_float2(a.y, a.y), t, w[1]);
                w[2] = fma2(make_float2(a.z, a.z), t, w[2]);
                w[3] = fma2(make_float2(a.w, a.w), t, w[3]);
            }
            float *Wh = Ws + mh * 32 * 33;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                Wh[(i0 + r) * 33 + j0] = w[r].x;
                Wh[(i0 + r) * 33 + j0 + 1] = w[r].y;
            }
        }
        __syncthreads();
        if (mh < nh) {                         // T21 = -T22 W (T22 is zero above its diagonal)
            const float *Wh = Ws + mh * 32 * 33;
            float *Th = Ts + mh * kChunk * LDA;
            float2 t21[4] = {};
#pragma unroll 8
            for (int k = 0; k < 32; ++k) {
                const float2 wk = make_float2(Wh[k * 33 + j0], Wh[k * 33 + j0 + 1]);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float t22 = Th[(32 + i0 + r) * LDA + 32 + k];
                    t21[r] = fma2(make_float2(t22, t22), wk, t21[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                Th[(32 + i0 + r) * LDA + j0] = -t21[r].x;
                Th[(32 + i0 + r) * LDA + j0 + 1] = -t21[r].y;
            }
        }
        __syncthreads();
        for (int h = 0; h < nh; ++h) {
            // [T; P] tile: T rows from the solve, P = e^{gam_i - gam_j} q_i.k_j (j <= i)
            {
                float v[32];
                if (row < kChunk) {
                    const float *Th = Ts + h * kChunk * LDA + row * LDA + c0;
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = Th[q];
                } else {
                    const int i = row - kChunk;
                    const float gi = gam[h * kChunk + i];
                    float s1[32];
                    tmem_ld32(lane_addr, s1);
                    const float4 *g4 = reinterpret_cast<const float4 *>(gam + h * kChunk + c0);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const float4 gj = g4[q4];
                        const float gv[4] = {gj.x, gj.y, gj.z, gj.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int q = 4 * q4 + e, jj = c0 + q;
                            v[q] = jj <= i ? ex2_approx(gi - gv[e]) * s1[q] : 0.f;
                        }
                    }
                }
                store_half_row_f16(tp, row, c0, v);
            }
            fence_async_smem();
            __syncthreads();
            // P T: A = [T; P] (K-major), B = T (MN-major, rows 0..63 of the same tile) -> cols [64, 128)
            if (tid == 0) {
                const uint32_t id = idesc_f16(128, 64, false, true);
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(tbase + 64, sw128_desc(smem_u32(tp) + 32 * ks, 16, 1024),
                            sw128_desc(smem_u32(tp) + 2048 * ks, 8192, 1024), id, ks != 0);
                mma_commit(bar_mma);
            }
            mma_out = true;
            if (!mbar_wait(bar_mma, mma_phase & 1, IMM)) s_err = 1;
            mma_phase++;
            __syncthreads();
            if (s_err) goto cleanup;
            mma_out = false;
            fence_after_sync();
            if (row >= kChunk) {   // P T replaces P in rows 64..127
                float v[32];
                tmem_ld32(lane_addr + 64, v);
                if (FOLD) {        // P' = scale P T diag(beta)
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] *= d.scale * bet[h * kChunk + c0 + q];
                }
                store_half_row_f16(tp, row, c0, v);
            } else if (FOLD) {     // diag(e^{gam_L - gam}) T diag(beta) in rows 0..63 (P T has read T)
                // gam is clamped to the chunk's last token, so gam[63] is gam_L
                const float er = ex2_approx(gam[h * kChunk + kChunk - 1] - gam[h * kChunk + row]);
                const float *Th = Ts + h * kChunk * LDA + row * LDA + c0;
                float v[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = er * Th[q] * bet[h * kChunk + c0 + q];
                store_half_row_f16(tp, row, c0, v);
            }
            fence_before_sync();
            __syncthreads();
            {
                uint4 *dst = reinterpret_cast<uint4 *>(out_of(hk * G + g0 + h));
                const uint4 *src = reinterpret_cast<const uint4 *>(tp);
                for (int e = tid; e < (int)(kTPTBytes / 16); e += kPrepThreads) dst[e] = src[e];
            }
            __syncthreads();   // tp is rewritten for the next v head
        }
    }

cleanup:
    if (s_err) {
        if (tid == 0) {
            set_timeout(p);
            if (load_out) mbar_wait(bar_load, load_phase & 1);
            if (mma_out) mbar_wait(bar_mma, mma_phase & 1);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 128);
}

// =============================================================== chain kernel
// Shared memory of the chain kernel: two stages of [K;Q] (dk/64 blocks of 16 KB)
// plus X (16 KB); one [T; P T] tile; the fp16 state copy h16 (B operand of
// [K;Q] h16); R and Vn' tiles.
struct ChainSmem {
    int blocks;
    int stages;            // 3 where they fit (dk <= 128), else 2
    size_t stage_bytes, x, tpt, h16, r16, vn16, bars, total;
    __host__ __device__ ChainSmem(int dk) {
        blocks = dk / 64;
        x = (size_t)blocks * 2 * kTileBytes;        // inside a stage, after the stack
        stage_bytes = x + kXBytes;
        stages = dk <= 128 ? 3 : 2;
        size_t o = (size_t)stages * stage_bytes;
        tpt = o; o += kTPTBytes;
        h16 = o; o += (size_t)(dk < 128 ? 128 : dk) * 128;
        r16 = o; o += kTileBytes;
        vn16 = o; o += kTileBytes;
        bars = o; o += 256;   // B_COUNT barriers and the TMEM slot
        total = o + 1024;
    }
};

// Warp roles. Warps 0..7 ("row warps"): lanes = rows of the 128-row MMA
// results, warps w and w+4 split the 64 columns; rows 0..63 produce R and Vn',
// rows 64..127 the output. Warps 8..15 ("state warps", same lane split) update
// the fp32 state kept in tensor memory and write its fp16 copy. Warp 16 issues
// every MMA, warp 17 every TMA copy. Roles meet on mbarriers (one arrival per
// warp).
//
// With H_c = e^{gL_c} H_{c-1} + K_c^T Vn'_c, the first product of chunk c splits as
//   [K_c; Q_c] H_{c-1} = [K_c; Q_c] (e^{gL_{c-1}} H_{c-2}) + X_c Vn'_{c-1},
//   X_c = [K_c; Q_c] K_{c-1}^T (from the prep kernel),
// so only X_c Vn'_{c-1} (4 MMAs) waits for the previous chunk; the dk-deep part
// and the state update run beside the critical path.
constexpr int kRowWarps = 8, kStateWarps = 8;
constexpr int kMmaWarp = kRowWarps + kStateWarps;
constexpr int kLoadWarp = kMmaWarp + 1;
constexpr int kChainThreads = (kLoadWarp + 1) * 32;
// B_LOAD s / B_LQ s: the K part / the Q + X part of stage s landed; B_QF s / B_KF s:
// the products reading stage s's Q + X part / K part are done (its refill may start).
constexpr int kMaxStages = 3;
enum ChainBar { B_LOAD0 = 0, B_LQ0 = B_LOAD0 + kMaxStages, B_TPT = B_LQ0 + kMaxStages, B_QF0, B_KF0 = B_QF0 + kMaxStages,
                B_C1 = B_KF0 + kMaxStages, B_R, B_C2, B_VN, B_O, B_C4, B_H, B_DRAIN, B_COUNT };

// NS stages: 3 where they fit (dk <= 128), else 2. REC: the backward's
// recompute, storing the state at each chunk's start, Vn and O in fp32.
// IMM: the test mode of the waits (gdn_set_wait_test_mode), a separate instance
template <int NS, bool REC = false, bool IMM = false>
__global__ void __launch_bounds__(kChainThreads, 1)
chunk_chain_kernel(const __grid_constant__ ChainMaps maps, const Problem p, int ntiles,
                   int64_t nslots, const unsigned char *prep_out, int cbase, int cmax) {
    extern __shared__ unsigned char smraw[];
    pdl_wait();       // the prep tiles (and everything before them) are complete
    pdl_trigger();
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const gdn_desc &d = p.d;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;          // TMEM lane
    const int c0 = ((warp >> 2) & 1) * 32;     // its 32 of the 64 columns
    int bid = blockIdx.x;
    const int tile = bid % ntiles;
    bid /= ntiles;
    const int j = bid % d.Hv;
    const int n = bid / d.Hv;
    if (p.cu != nullptr && *p.status != GDN_OK) return;
    const int dk = d.dk, dv = d.dv, Hv = d.Hv;
    const int G = Hv / d.Hk;                   // v heads per q/k head
    const int hk = j / G;
    const int v0 = tile * 64;
    // chunks [cbase, cbase + cmax) of the sequence: a segment of it, or all of it;
    // h0 / hT are the state before / after the segment
    const int64_t sstart = p.cu ? (int64_t)p.cu[n] : (int64_t)n * d.T;
    const int64_t seq1 = p.cu ? (int64_t)p.cu[n + 1] : sstart + d.T;
    const int64_t seq0 = sstart + (int64_t)cbase * kChunk;
    const int64_t left = seq1 > seq0 ? (seq1 - seq0 + kChunk - 1) / kChunk : 0;
    const int nchunks = (int)(left < cmax ? left : cmax);
    const int64_t slot0 = (p.cu ? (int64_t)p.chunk_off[n] : (int64_t)n * ((d.T + kChunk - 1) / kChunk)) + cbase;
    const ChainSmem L(dk);
    const int halves = dk >= 128 ? dk / 128 : 1;  // M=128 row groups of the state
    unsigned char *tptb = sm + L.tpt, *h16 = sm + L.h16, *r16 = sm + L.r16, *vn16 = sm + L.vn16;
    uint64_t *bar = (uint64_t *)(sm + L.bars);
    uint32_t *tslot = (uint32_t *)(bar + B_COUNT);
    __shared__ volatile int s_err;
    const size_t sbase = ((size_t)n * Hv + j) * dk * dv;
    const float *gw = (const float *)p.gamma + (int64_t)j * p.ntok;
    const float *bw = p.beta + (int64_t)j * p.ntok;
    const __half *vw = (const __half *)p.v + (int64_t)j * p.ntok * dv;
    __half *o = (__half *)p.o;
    const bool state_warp = warp >= kRowWarps && warp < kMmaWarp;
    // row hrow, columns c0..c0+31 of this tile in the recompute's state at chunk c's start
    auto rec_h0_row = [&](int c, int hrow) {
        return p.rec_h0 + ((size_t)(slot0 + c) * Hv + j) * dk * dv + (size_t)hrow * dv + v0 + c0;
    };

    if (tid == 0) {
        s_err = 0;
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&bar[B_LOAD0 + i], 1);
            mbar_init(&bar[B_LQ0 + i], 1);
            mbar_init(&bar[B_QF0 + i], 1);
            mbar_init(&bar[B_KF0 + i], 1);
        }
        mbar_init(&bar[B_TPT], 1);
        mbar_init(&bar[B_C1], 1);
        mbar_init(&bar[B_C2], 1);
        mbar_init(&bar[B_C4], 1);
        mbar_init(&bar[B_R], 4);     // row warps of rows 0..63: 0, 1, 4, 5
        mbar_init(&bar[B_VN], 4);
        mbar_init(&bar[B_O], 4);     // row warps of rows 64..127: 2, 3, 6, 7
        mbar_init(&bar[B_H], kStateWarps);
        mbar_init(&bar[B_DRAIN], 1);
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // TMEM: D1 (two buffers) at 0 / 64, D2 at 128, H (fp32) at 320 + 64 h
    auto tD1 = [&](int c) { return tbase + lane_off + c0 + 64 * (c & 1); };
    const uint32_t tD2 = tbase + 128 + lane_off + c0;
    const uint32_t tH = tbase + 320 + lane_off + c0;

    auto chunk_tok0 = [&](int c) { return seq0 + (int64_t)c * kChunk; };
    auto chunk_len = [&](int c) {
        const int64_t r = seq1 - chunk_tok0(c);
        return r < kChunk ? (int)r : kChunk;
    };
    auto gamma_last = [&](int c) { return gw[chunk_tok0(c) + chunk_len(c) - 1]; };
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (s_err) return false;
        if (!mbar_wait(&bar[b], parity, IMM)) { s_err = 1; return false; }
        return true;
    };
    auto warp_arrive = [&](int b) {
        fence_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[b]);
    };
    // state warps: fp32 state into TMEM and its fp16 copy (chunk 0's B operand)
    if (state_warp) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int hrow = 128 * h + row;
            if (h >= halves) break;
            float t[32];
            if (hrow < dk && p.h0) {
                const float4 *src = reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)hrow * dv + v0 + c0);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 f = src[q];
                    t[4 * q] = f.x; t[4 * q + 1] = f.y; t[4 * q + 2] = f.z; t[4 * q + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) t[q] = 0.f;
            }
            tmem_st32(tH + 64 * h, t);
            if (hrow < dk) store_half_row_f16(h16, hrow, c0, t);
            if (REC && hrow < dk && nchunks > 0) store_row_f32(rec_h0_row(0, hrow), t);
        }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // per load barrier (B_LOAD s, B_LQ s, B_TPT): the parity of the last phase the TMA
    // thread armed, or -1; kept in shared memory, read only by the drain
    __shared__ int s_armed[B_TPT + 1];
    if (tid <= B_TPT) s_armed[tid] = -1;
    __syncthreads();
    if (warp == kLoadWarp) {
        // -------------------------------------------------------- TMA warp
        if (lane == 0) {
            // a stage is [K_b; Q_b] for each 64-column block b, then X; its K part is
            // read until C4 of the chunk, its Q and X parts only until C1
            auto load_k = [&](int c) {
                const int s = c % NS;
                unsigned char *st = sm + s * L.stage_bytes;
                const int yk = (int)((int64_t)hk * p.ntok + chunk_tok0(c));
                mbar_expect_tx(&bar[B_LOAD0 + s], (uint32_t)L.blocks * kTileBytes);
                s_armed[B_LOAD0 + s] = (c / NS) & 1;
                for (int b = 0; b < L.blocks; ++b)
                    tma_load_2d(st + b * 2 * kTileBytes, &maps.k_hi, 64 * b, yk, &bar[B_LOAD0 + s]);
            };
            auto load_qx = [&](int c) {
                const int s = c % NS;
                unsigned char *st = sm + s * L.stage_bytes;
                const int yk = (int)((int64_t)hk * p.ntok + chunk_tok0(c));
                const bool with_x = c > 0;
                mbar_expect_tx(&bar[B_LQ0 + s], (uint32_t)L.blocks * kTileBytes + (with_x ? kXBytes : 0));
                s_armed[B_LQ0 + s] = (c / NS) & 1;
                for (int b = 0; b < L.blocks; ++b)
                    tma_load_2d(st + b * 2 * kTileBytes + kTileBytes, &maps.q_hi, 64 * b, yk, &bar[B_LQ0 + s]);
                if (with_x)
                    bulk_load(st + L.x, prep_out + ((int64_t)(hk * G) * nslots + slot0 + c) * kPrepOut + kTPTBytes,
                              kXBytes, &bar[B_LQ0 + s]);
            };
            auto load_tpt = [&](int c) {
                mbar_expect_tx(&bar[B_TPT], kTPTBytes);
                s_armed[B_TPT] = c & 1;
                bulk_load(tptb, prep_out + ((int64_t)j * nslots + slot0 + c) * kPrepOut, kTPTBytes, &bar[B_TPT]);
            };
            constexpr int ns = NS;
            for (int c = 0; c < ns && c < nchunks; ++c) {
                load_k(c);
                load_qx(c);
                if (c == 0) load_tpt(0);
            }
            // Each wait below is for the phase right after the one this thread last
            // consumed, and the barrier cannot complete the next one before this
            // thread's refill: B_QF s / B_KF s are re-armed only by the products of
            // chunk c + ns, which need the parts loaded here; B_C2 only by chunk
            // c+1's C2, which needs its [T; P T] load.
            for (int c = 0; c + 1 < nchunks; ++c) {
                const int s = c % ns;
                const uint32_t ph = (uint32_t)(c / ns) & 1;
                // Q and X of chunk c+ns into chunk c's stage once C1 of chunk c is done
                if (c + ns < nchunks) {
                    if (!wait(B_QF0 + s, ph)) break;
                    load_qx(c + ns);
                }
                // [T; P T] of chunk c+1 once C2 of chunk c has read the buffer
                if (!wait(B_C2, c & 1)) break;
                load_tpt(c + 1);
                // K of chunk c+ns once its last reader (C4 of chunk c) is done
                if (c + ns < nchunks) {
                    if (!wait(NS == 2 ? B_C4 : B_KF0 + s, NS == 2 ? (uint32_t)(c & 1) : ph)) break;
                    load_k(c + ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------- MMA warp
        if (lane == 0) {
            const uint32_t id_k = idesc_f16(128, 64, false, true);   // A K-major, B MN-major
            const uint32_t id_m = idesc_f16(128, 64, true, true);    // A MN-major (K^T), B MN-major
            // descriptors are computed once; a K step adds a constant to the start field
            const uint64_t d_st0 = sw128_desc(smem_u32(sm), 16, 1024);
            const uint64_t d_h16 = sw128_desc(smem_u32(h16), 8192, 1024);
            const uint64_t d_vn = sw128_desc(smem_u32(vn16), 8192, 1024);
            const uint64_t d_r = sw128_desc(smem_u32(r16), 8192, 1024);
            const uint64_t d_tpt = sw128_desc(smem_u32(tptb), 16, 1024);
            // dk = 64 has a single 64-row block: LBO 0 repeats it as rows 64..127 (ignored)
            const uint64_t d_kt0 = sw128_desc(smem_u32(sm), dk >= 128 ? 2 * kTileBytes : 0, 1024);
            const uint32_t stage16 = (uint32_t)(L.stage_bytes >> 4), x16 = (uint32_t)(L.x >> 4);
            // H += K_c^T Vn'_c, into the state the state warps already scaled by e^{gL_c}
            auto issue_c4 = [&](int c) {
                const uint64_t a0 = d_kt0 + (c % NS) * stage16;
                for (int h = 0; h < halves; ++h)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tbase + 320 + 64 * h, a0 + (uint64_t)((h * 4 * kTileBytes + 2048 * ks) >> 4),
                                d_vn + (uint64_t)((2048 * ks) >> 4), id_m, 1);
                mma_commit(&bar[B_C4]);
                if (NS > 2) mma_commit(&bar[B_KF0 + c % NS]);   // the stage's K part is free
            };
            auto issue_c1a = [&](int c) {  // D1 = [K; Q] h16
                const uint64_t a0 = d_st0 + (c % NS) * stage16;
                for (int b = 0; b < L.blocks; ++b)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tbase + 64 * (c & 1), a0 + (uint64_t)((b * 2 * kTileBytes + 32 * ks) >> 4),
                                d_h16 + (uint64_t)(((b * 4 + ks) * 2048) >> 4), id_k, (b | ks) != 0);
            };
            int c = 0;
            for (; c < nchunks; ++c) {
                const int s = c % NS;
                const uint32_t ph = (uint32_t)(c / NS) & 1;
                if (!wait(B_LOAD0 + s, ph) || !wait(B_LQ0 + s, ph)) break;
                if (c >= 1 && !wait(B_H, (c - 1) & 1)) break;     // h16 = e^{gL_{c-1}} H_{c-2}
                fence_after_sync();
                issue_c1a(c);
                if (c >= 1) {
                    // C1b: D1 += X Vn'_{c-1} (the only product that waits for chunk c-1)
                    if (!wait(B_VN, (c - 1) & 1)) break;
                    fence_after_sync();
                    const uint64_t ax = d_st0 + s * stage16 + x16;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tbase + 64 * (c & 1), ax + (uint64_t)((32 * ks) >> 4),
                                d_vn + (uint64_t)((2048 * ks) >> 4), id_k, 1);
                }
                mma_commit(&bar[B_C1]);
                mma_commit(&bar[B_QF0 + s]);      // stage s's Q and X parts are free
                if (c >= 1) issue_c4(c - 1);
                // C2: D2 = [T; P T] R
                if (!wait(B_TPT, c & 1) || !wait(B_R, c & 1)) break;
                if (c >= 1 && !wait(B_O, (c - 1) & 1)) break;     // D2 of chunk c-1 consumed
                fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(tbase + 128, d_tpt + (uint64_t)((32 * ks) >> 4),
                            d_r + (uint64_t)((2048 * ks) >> 4), id_k, ks != 0);
                mma_commit(&bar[B_C2]);
            }
            if (c == nchunks && nchunks > 0) {   // state update of the last chunk
                if (wait(B_VN, (nchunks - 1) & 1) && wait(B_H, (nchunks - 1) & 1)) {
                    fence_after_sync();
                    issue_c4(nchunks - 1);
                }
            }
        }
        __syncwarp();
    } else if (warp < kRowWarps) {
        // ---------------------------------------------------------- row warps
        const bool top = row < kChunk;
        const int r = top ? row : row - kChunk;   // token within the chunk
        // operands of the next chunk, prefetched into registers: V row slice,
        // gamma and beta of this row, the chunk's last gamma
        uint4 vq[4];
        float g_r = 0.f, b_r = 0.f, g_l = 0.f;
        auto prefetch = [&](int c) {
            const int64_t t0 = chunk_tok0(c);
            const int len = chunk_len(c);
            const int i = r < len ? r : len - 1;
            g_r = gw[t0 + i];
            g_l = gw[t0 + len - 1];
            if (top) {
                b_r = r < len ? bw[t0 + r] : 0.f;
                const uint4 *src = reinterpret_cast<const uint4 *>(vw + (t0 + i) * dv + v0 + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) vq[q] = r < len ? src[q] : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        if (nchunks > 0) prefetch(0);
        for (int c = 0; c < nchunks; ++c) {
            const int64_t t0 = chunk_tok0(c);
            const int len = chunk_len(c);
            const float gr = g_r, br = b_r, gl = g_l;
            if (top) {
                float vv[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) unpack16<__half>(vq[q], vv + 8 * q);
                // E1: R = beta (V - e^gam K H) -> r16
                if (!wait(B_C1, c & 1)) break;
                fence_after_sync();
                float a[32];
                tmem_ld32(tD1(c), a);
                const float eg = __expf(gr);
#pragma unroll
                for (int q = 0; q < 32; ++q) a[q] = br * (vv[q] - eg * a[q]);
                store_half_row_f16(r16, r, c0, a);
                warp_arrive(B_R);
                // E2a: Vn' = e^{gam_L - gam} Vn -> vn16
                if (!wait(B_C2, c & 1)) break;
                fence_after_sync();
                tmem_ld32(tD2, a);
                const float sc = __expf(gl - gr);
#pragma unroll
                for (int q = 0; q < 32; ++q) a[q] *= sc;
                store_half_row_f16(vn16, r, c0, a);
                warp_arrive(B_VN);
                if (REC) {
                    // D2 stays until this warp's next B_R arrival lets the next C2 in;
                    // the load is warp-collective, only the store depends on the row
                    tmem_ld32(tD2, a);
                    if (r < len) store_row_f32(p.rec_vn + ((int64_t)j * p.ntok + t0 + r) * dv + v0 + c0, a);
                }
                // the next chunk's operands only now: the proxy fence of an arrival
                // waits for this thread's loads in flight, so none may be pending
                // at the two arrivals on the serial path
                if (c + 1 < nchunks) prefetch(c + 1);
            } else {
                // E2b: O = e^gam (Q H) + P Vn -> o   (off the critical path)
                if (c + 1 < nchunks) prefetch(c + 1);
                if (!wait(B_C2, c & 1)) break;
                fence_after_sync();
                float a[32], b2[32];
                tmem_ld32(tD1(c), a);
                tmem_ld32(tD2, b2);
                // no shared-memory writes to publish: order the tensor-memory reads only
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_O]);
                if (REC && r < len) {
                    const float eg = __expf(gr);
#pragma unroll
                    for (int q = 0; q < 32; ++q) a[q] = fmaf(eg, a[q], b2[q]) * d.scale;
                    store_row_f32(p.rec_o + ((int64_t)j * p.ntok + t0 + r) * dv + v0 + c0, a);
                } else if (!REC && r < len) {
                    const float eg = __expf(gr);
                    uint4 *dst = reinterpret_cast<uint4 *>(o + ((t0 + r) * Hv + j) * (int64_t)dv + v0 + c0);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint4 u;
                        __half2 *hh = reinterpret_cast<__half2 *>(&u);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            hh[e] = __floats2half2_rn(fmaf(eg, a[8 * ch + 2 * e], b2[8 * ch + 2 * e]) * d.scale,
                                                      fmaf(eg, a[8 * ch + 2 * e + 1], b2[8 * ch + 2 * e + 1]) * d.scale);
                        dst[ch] = u;
                    }
                }
            }
        }
    } else if (state_warp) {
        // -------------------------------------------------------- state warps
        // Once H_c is complete (C4 of chunk c done): H <- e^{gL_{c+1}} H_c in place,
        // so that C4 of chunk c+1 accumulates onto it, and its fp16 copy h16 (the
        // B operand of chunk c+2's first product).
        auto final_state = [&]() {
            for (int h = 0; h < halves; ++h) {
                const int hrow = 128 * h + row;
                if (hrow >= dk) continue;
                float t[32];
                tmem_ld32(tH + 64 * h, t);
                float4 *dst = reinterpret_cast<float4 *>(p.hT + sbase + (size_t)hrow * dv + v0 + c0);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float4(t[4 * q], t[4 * q + 1], t[4 * q + 2], t[4 * q + 3]);
            }
        };
        // rec_c >= 0: the state read is H0 of chunk rec_c (REC only)
        auto scale_state = [&](float e, bool copy, int rec_c) {
            for (int h = 0; h < halves; ++h) {
                const int hrow = 128 * h + row;
                if (hrow >= dk) continue;
                float t[32];
                tmem_ld32(tH + 64 * h, t);
                if (REC && rec_c >= 0) store_row_f32(rec_h0_row(rec_c, hrow), t);
#pragma unroll
                for (int q = 0; q < 32; ++q) t[q] *= e;
                tmem_st32(tH + 64 * h, t);
                if (copy) store_half_row_f16(h16, hrow, c0, t);
            }
        };
        if (nchunks > 0) {
            // chunk 0's first product has read h16 = H_init: scale for chunk 0's
            // update and publish e^{gL_0} H_init for chunk 1
            if (wait(B_C1, 0)) {
                scale_state(__expf(gamma_last(0)), nchunks > 1, -1);
                warp_arrive(B_H);
                for (int c = 0; c < nchunks; ++c) {
                    const float gl_next = c + 1 < nchunks ? gamma_last(c + 1) : 0.f;
                    if (!wait(B_C4, c & 1)) break;
                    fence_after_sync();
                    if (c + 1 < nchunks) {
                        scale_state(__expf(gl_next), c + 2 < nchunks, c + 1);
                        warp_arrive(B_H);
                    }
                }
                if (p.hT && !s_err) final_state();
            }
        } else if (p.hT) {               // empty sequence: final state = initial state
            final_state();
        }
    }
    __syncthreads();
    if (s_err) {
        // drain, with bounded waits, before the tensor memory is freed: every MMA the
        // MMA thread issued (one more commit covers them all) and the last armed phase
        // of every load barrier
        if (tid == kMmaWarp * 32) {
            set_timeout(p);
            mma_commit(&bar[B_DRAIN]);
            mbar_wait(&bar[B_DRAIN], 0);
        }
        if (tid == kLoadWarp * 32)
            for (int b = 0; b <= B_TPT; ++b)
                if (s_armed[b] >= 0) mbar_wait(&bar[b], (uint32_t)s_armed[b]);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ===================================================================== host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return (PFN_cuTensorMapEncodeTiled_v12000)f;
    }();
    return fn;
}


// Segmented schedule of a long single sequence: one high-priority stream per
// device for the chain segments and the events that order them against the
// prep segments on the caller's stream, created on first use and kept (events
// are re-recorded by every call; the enqueue runs under the mutex, so one
// call's records are waited on before another call records them again).
constexpr int kMaxSegments = 16;
struct SideStream {
    cudaStream_t hp = nullptr;
    cudaEvent_t ev[kMaxSegments + 2] = {};
    bool ready = false;
};
std::mutex g_side_mu;
SideStream g_side[64];

SideStream *side_stream(int dev) {   // caller holds g_side_mu
    if (dev < 0 || dev >= 64) return nullptr;
    SideStream &ss = g_side[dev];
    if (ss.ready) return &ss;
    int lo = 0, hi = 0;
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithPriority(&ss.hp, cudaStreamNonBlocking, hi) != cudaSuccess) return nullptr;
    for (auto &e : ss.ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ss.ready = true;
    return &ss;
}

// v heads per solve pass of the prep kernel, and its instance
int prep_pass_heads(const gdn_desc &) { return 1; }
using PrepFn = void (*)(const PrepMaps, const Problem, int64_t, unsigned char *, int64_t);
template <int MINB>
PrepFn prep_instance(bool imm, bool fold) {
    return fold ? (imm ? chunk_prep_kernel<1, true, true, MINB> : chunk_prep_kernel<1, false, true, MINB>)
                : (imm ? chunk_prep_kernel<1, true, false, MINB> : chunk_prep_kernel<1, false, false, MINB>);
}
// three_per_sm: beside a chain segment, or a grid that fits one round of three
PrepFn prep_kernel(int, bool imm, bool fold, bool three_per_sm = false) {
    return three_per_sm ? prep_instance<3>(imm, fold) : prep_instance<4>(imm, fold);
}

int max_dyn_smem() {
    int dev = 0, v = 232448;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return v;
}

}  // namespace

bool encode_tile_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
    return encode_tile_map_pitch(m, base, rows, cols, cols * 2);
}

bool encode_tile_map_pitch(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint64_t pitch) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool chunk_tc_supports(const gdn_desc &d) {
    return (d.dtype == GDN_BF16 || d.dtype == GDN_F16) && (d.dk == 64 || d.dk == 128 || d.dk == 256) &&
           d.dv >= 64 && d.dv % 64 == 0;
}

// The prep tiles, and for a single sequence the state between two segments of
// its chain (see launch_chunk_tc).
size_t chunk_tc_workspace(const gdn_desc &d) {
    if (!chunk_tc_supports(d)) return 0;
    const size_t seg_state = d.N == 1 ? (size_t)d.Hv * d.dk * d.dv * sizeof(float) : 0;
    return (size_t)d.Hv * (size_t)chunk_slot_bound(d) * kPrepOut + seg_state;
}

cudaError_t launch_chunk_tc(const Problem &p, cudaStream_t s) {
    const gdn_desc &d = p.d;
    const int64_t nslots_alloc = chunk_slot_bound(d);
    const int64_t nslots = chunk_slots(p);
    if (nslots > nslots_alloc || p.tpt == nullptr) return cudaErrorInvalidValue;
    unsigned char *tpt = (unsigned char *)p.tpt;
    const int64_t plane = (int64_t)d.Hk * p.ntok * d.dk;
    if (p.ntok > 0) {
        PrepMaps pm;
        const __half *q = (const __half *)p.q, *k = (const __half *)p.k;
        if (!encode_tile_map(&pm.q_hi, q, (uint64_t)d.Hk * p.ntok, d.dk) ||
            !encode_tile_map(&pm.q_lo, q + plane, (uint64_t)d.Hk * p.ntok, d.dk) ||
            !encode_tile_map(&pm.k_hi, k, (uint64_t)d.Hk * p.ntok, d.dk) ||
            !encode_tile_map(&pm.k_lo, k + plane, (uint64_t)d.Hk * p.ntok, d.dk))
            return cudaErrorInvalidValue;
        const int ph = prep_pass_heads(d);
        const PrepSmem ps(d.dk, ph);
        // a grid that fits in one round of three CTAs per SM takes the 80-register instance
        int dev = 0, nsm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            nsm = 0;
        const bool one_round = nslots * d.Hk <= 3 * (int64_t)nsm;
        auto prep = prep_kernel(ph, p.wait_immediate != 0, chain_tm_supports(d), one_round);
        cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ps.total);
        if (e != cudaSuccess) return e;
        if (nslots > 0) {
            e = launch_kernel(p.pdl, prep, dim3((unsigned)nslots, d.Hk), dim3(kPrepThreads), ps.total, s,
                              pm, p, nslots_alloc, tpt, (int64_t)0);
            if (e != cudaSuccess) return e;
        }
    }
    if (chain_tm_supports(d))
        return launch_chain_tm(p, s, tpt, nslots_alloc, 0, 0x7fffffff, p.pdl && p.ntok > 0,
                               (unsigned)((int64_t)d.N * d.Hv * chain_tm_tiles(d)));
    ChainMaps cm;
    if (p.ntok > 0) {
        if (!encode_tile_map(&cm.q_hi, p.q, (uint64_t)d.Hk * p.ntok, d.dk) ||
            !encode_tile_map(&cm.k_hi, p.k, (uint64_t)d.Hk * p.ntok, d.dk) ||
            !encode_tile_map(&cm.v, p.v, (uint64_t)d.Hv * p.ntok, d.dv))
            return cudaErrorInvalidValue;
    } else {
        memset(&cm, 0, sizeof(cm));
    }
    const int maxs = max_dyn_smem();
    const ChainSmem cs(d.dk);
    // the kernel holds all 512 TMEM columns: request enough shared memory that a
    // second CTA never shares the SM (its allocation would wait for this one)
    const size_t smem = cs.total > (size_t)(maxs / 2 + 1024) ? cs.total : (size_t)(maxs / 2 + 1024);
    if ((int)smem > maxs) return cudaErrorInvalidValue;
    auto chain = p.wait_immediate ? (cs.stages == 3 ? chunk_chain_kernel<3, false, true> : chunk_chain_kernel<2, false, true>)
                                  : (cs.stages == 3 ? chunk_chain_kernel<3> : chunk_chain_kernel<2>);
    cudaError_t e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int ntiles = d.dv / 64;
    const int64_t blocks = (int64_t)d.N * d.Hv * ntiles;
    if (blocks == 0) return cudaSuccess;
    return launch_kernel(p.pdl && p.ntok > 0, chain, dim3((unsigned)blocks), dim3(kChainThreads), smem, s, cm, p, ntiles,
                         nslots_alloc, (const unsigned char *)tpt, 0, 0x7fffffff);
}

// The backward's recompute: the same prep and chain launches on one stream, the
// chain instantiated with the stores of the state at every chunk's start, Vn and
// O in fp32 (p.rec_h0 / rec_vn / rec_o) in place of the 16-bit o.
cudaError_t launch_chunk_tc_rec(const Problem &p, cudaStream_t s) {
    const gdn_desc &d = p.d;
    if (!p.rec_h0 || !p.rec_vn || !p.rec_o) return cudaErrorInvalidValue;
    const int64_t nslots_alloc = chunk_slot_bound(d);
    const int64_t nslots = chunk_slots(p);
    if (nslots > nslots_alloc || p.tpt == nullptr || p.ntok == 0) return cudaErrorInvalidValue;
    unsigned char *tpt = (unsigned char *)p.tpt;
    const int64_t plane = (int64_t)d.Hk * p.ntok * d.dk;
    PrepMaps pm;
    ChainMaps cm;
    const __half *q = (const __half *)p.q, *k = (const __half *)p.k;
    if (!encode_tile_map(&pm.q_hi, q, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&pm.q_lo, q + plane, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&pm.k_hi, k, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&pm.k_lo, k + plane, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&cm.q_hi, p.q, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&cm.k_hi, p.k, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&cm.v, p.v, (uint64_t)d.Hv * p.ntok, d.dv))
        return cudaErrorInvalidValue;
    const int ph = prep_pass_heads(d);
    const PrepSmem ps(d.dk, ph);
    auto prep = prep_kernel(ph, p.wait_immediate != 0, false);   // the 64-column chain's tile
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ps.total);
    if (e != cudaSuccess) return e;
    prep<<<dim3((unsigned)nslots, d.Hk), kPrepThreads, ps.total, s>>>(pm, p, nslots_alloc, tpt, (int64_t)0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int maxs = max_dyn_smem();
    const ChainSmem cs(d.dk);
    const size_t smem = cs.total > (size_t)(maxs / 2 + 1024) ? cs.total : (size_t)(maxs / 2 + 1024);
    if ((int)smem > maxs) return cudaErrorInvalidValue;
    auto chain = cs.stages == 3 ? chunk_chain_kernel<3, true> : chunk_chain_kernel<2, true>;
    if ((e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    const int ntiles = d.dv / 64;
    const int64_t blocks = (int64_t)d.N * d.Hv * ntiles;
    if (blocks == 0) return cudaSuccess;
    chain<<<(unsigned)blocks, kChainThreads, smem, s>>>(cm, p, ntiles, nslots_alloc, tpt, 0, 0x7fffffff);
    return cudaGetLastError();
}

// One long sequence whose chain occupies at most half of the SMs: the chunks are
// cut into segments; the prep of every segment runs on the caller's stream, the
// chain of segment k on a high-priority side stream once the prep of segment k
// is done, so that the prep of segment k+1 uses the SMs the chain leaves idle.
// The state crosses segments through the workspace (the chain's h0 / hT).
bool chunk_tc_segmented(const Problem &p) {
    const gdn_desc &d = p.d;
    if (p.single_stream || p.cu != nullptr || d.N != 1 || p.ntok == 0) return false;
    const int64_t nch = (d.T + kChunk - 1) / kChunk;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    const int64_t chain_ctas = (int64_t)d.Hv * (chain_tm_supports(d) ? chain_tm_tiles(d) : d.dv / 64);
    return nch >= 256 && chain_ctas * 2 <= nsm;
}

cudaError_t launch_chunk_tc_segmented(const Problem &p, cudaStream_t s) {
    const gdn_desc &d = p.d;
    const int64_t nslots_alloc = chunk_slot_bound(d);
    const int nch = (int)((d.T + kChunk - 1) / kChunk);
    const int seg = (nch + kMaxSegments - 1) / kMaxSegments > 64 ? (nch + kMaxSegments - 1) / kMaxSegments : 64;
    const int nseg = (nch + seg - 1) / seg;
    unsigned char *tpt = (unsigned char *)p.tpt;
    float *seg_state = (float *)(tpt + (size_t)d.Hv * nslots_alloc * kPrepOut);
    const int64_t plane = (int64_t)d.Hk * p.ntok * d.dk;
    PrepMaps pm;
    ChainMaps cm;
    const __half *q = (const __half *)p.q, *k = (const __half *)p.k;
    if (!encode_tile_map(&pm.q_hi, q, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&pm.q_lo, q + plane, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&pm.k_hi, k, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&pm.k_lo, k + plane, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&cm.q_hi, p.q, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&cm.k_hi, p.k, (uint64_t)d.Hk * p.ntok, d.dk) ||
        !encode_tile_map(&cm.v, p.v, (uint64_t)d.Hv * p.ntok, d.dv))
        return cudaErrorInvalidValue;
    const int ph = prep_pass_heads(d);
    const PrepSmem ps(d.dk, ph);
    auto prep = prep_kernel(ph, p.wait_immediate != 0, chain_tm_supports(d), true);
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ps.total);
    if (e != cudaSuccess) return e;
    const int maxs = max_dyn_smem();
    const ChainSmem cs(d.dk);
    const size_t smem = cs.total > (size_t)(maxs / 2 + 1024) ? cs.total : (size_t)(maxs / 2 + 1024);
    if ((int)smem > maxs) return cudaErrorInvalidValue;
    auto chain = p.wait_immediate ? (cs.stages == 3 ? chunk_chain_kernel<3, false, true> : chunk_chain_kernel<2, false, true>)
                                  : (cs.stages == 3 ? chunk_chain_kernel<3> : chunk_chain_kernel<2>);
    if ((e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return e;
    const int ntiles = d.dv / 64;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream *ss = side_stream(dev);
    if (!ss) return cudaErrorInvalidValue;
    // the side stream starts after everything already queued on the caller's
    if ((e = cudaEventRecord(ss->ev[0], s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->hp, ss->ev[0], 0)) != cudaSuccess) return e;
    for (int g = 0; g < nseg; ++g) {
        const int cb = g * seg, cn = nch - cb < seg ? nch - cb : seg;
        prep<<<dim3((unsigned)cn, d.Hk), kPrepThreads, ps.total, s>>>(pm, p, nslots_alloc, tpt, (int64_t)cb);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = cudaEventRecord(ss->ev[1 + g], s)) != cudaSuccess) return e;
    }
    for (int g = 0; g < nseg; ++g) {
        const int cb = g * seg, cn = nch - cb < seg ? nch - cb : seg;
        if ((e = cudaStreamWaitEvent(ss->hp, ss->ev[1 + g], 0)) != cudaSuccess) return e;
        Problem pg = p;
        pg.h0 = g == 0 ? p.h0 : seg_state;
        pg.hT = g == nseg - 1 ? p.hT : seg_state;
        if (chain_tm_supports(d)) {
            e = launch_chain_tm(pg, ss->hp, tpt, nslots_alloc, cb, cn, false, (unsigned)(d.Hv * chain_tm_tiles(d)));
        } else {
            chain<<<(unsigned)(d.Hv * ntiles), kChainThreads, smem, ss->hp>>>(cm, pg, ntiles, nslots_alloc, tpt,
                                                                              cb, cn);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
    }
    // the caller's stream continues once the last chain segment is done
    if ((e = cudaEventRecord(ss->ev[1 + nseg], ss->hp)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(s, ss->ev[1 + nseg], 0);
}

}  // namespace gdn
