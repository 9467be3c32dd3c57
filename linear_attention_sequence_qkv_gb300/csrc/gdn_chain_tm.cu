// gdn_chain_tm.cu -- the serial state pass of the chunked gated delta rule for
// dk <= 128 on the tcgen05 tensor cores, transposed so that 128 dv columns of
// the state are the 128 rows (TMEM lanes) of every product, and the state and
// the per-chunk operands stay in tensor memory.
//
// With H = S^T [dk][dv], and per chunk c of 64 tokens gam = in-chunk cumulative
// decay, gL = its last value, and the prep kernel's tiles [T; P T] and
// X_c = [K_c; Q_c] K_{c-1}^T (see gdn_chunk_tc.cu):
//   D1^T  = H_{c-1}^T [K_c; Q_c]^T
//         = (e^{gL_{c-1}} H_{c-2})^T [K_c; Q_c]^T + Vn'^T_{c-1} X_c^T
//   R~^T  = (V - diag(e^gam) K H_{c-1})^T                  (K half of D1^T)
//   D2^T  = R~^T [T'; P']^T                                (N = 128)
//   Vn'^T = top half of D2^T
//   O^T   = (Q H_{c-1})^T diag(e^gam) + bottom half of D2^T  (Q half of D1^T)
// where the prep kernel's tile already holds T' = diag(e^{gL - gam}) T diag(beta)
// and P' = scale P T diag(beta), so the row warps apply no per-token factor but
// e^gam. V^T reaches tensor memory through one more product, V^T I (the V tile
// as an MN-major A operand, a 64 x 64 identity as B), into D2's top half, which is
// free between the row warps' read of Vn'_{c-1} and the second product of chunk
// c: the row warps read V^T and K H with one tensor-memory load.
//   H_c^T = e^{gL_c} H_{c-1}^T + Vn'^T_c K_c
// Each product has M = 128 dv rows and takes its A operand from tensor memory
// (the fp16 copy of the state, R^T or Vn'^T, each written by the warps with
// tcgen05.st); only its B operand ([K; Q], X, [T; P T]) comes from shared memory,
// where a TMA warp stages it ahead of use. So the hand-offs on the serial path
// (D1 -> R -> D2 -> Vn' -> next D1) are tensor-memory loads and stores with no
// shared-memory round trip. The V tile also arrives by TMA; the outputs leave
// through a swizzled staging tile (16x256b tensor-memory loads give each thread
// token pairs of two dv rows, which stmatrix stores transposed) and TMA tensor
// stores. The per-token factor e^gam reaches the warps as broadcast reads of small
// per-warp arrays rather than shuffles.
//
// EPI instance (gdn_forward with dv = 128, chain_tm_fuses_epilogue): one CTA holds
// every dv of a token, so the output step (gated RMSNorm) runs here: the out warps
// read the staged o rows back in the separate output kernel's layout, repeat its
// arithmetic and order of sums (bit for bit the same out), and the tile leaves as
// out; the gate tile arrives by TMA in place of the second V slot.
//
// Every wait on an mbarrier gives up after about a second; the CTA then records
// GDN_ERR_DEVICE_TIMEOUT, waits (bounded) for its own copies and products in
// flight, frees its tensor memory and returns.
#include <cuda.h>

#include <cstring>

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using namespace tc;

// warps 0..7: R and Vn' (the serial path); 8..15: state scaling and outputs;
// 16: MMA issue; 17: TMA
constexpr int kRowW = 8, kOutW = 8;
constexpr int kMmaW = kRowW + kOutW, kTmaW = kMmaW + 1;
constexpr int kTmThreads = (kTmaW + 1) * 32;

// tensor-memory columns (lanes = the tile's 128 dv rows), each region aligned to its size
constexpr uint32_t kTH = 0;      // H^T fp32, dk columns
constexpr uint32_t kTD2 = 128;   // D2^T: [T R | P T R], 128 fp32 columns
constexpr uint32_t kTD1 = 256;   // D1^T: [K H | Q H], 128 fp32 columns
constexpr uint32_t kTH16 = 384;  // fp16 copy of (scaled) H^T, dk/2 columns
constexpr uint32_t kTR = 448;    // R^T fp16, 32 columns
constexpr uint32_t kTVN = 480;   // Vn'^T fp16, 32 columns

struct TmMaps {
    CUtensorMap q_hi, k_hi, v, o;
    CUtensorMap gate, out;   // the fused output step only
};

// T_FULL s / T_FREE s: operand stage s ([K; Q]) landed / free again (after the state
// update that reads its K last); T_PFULL p / T_PFREE p: prep slot p (X and [T; P T])
// landed / read by the chunk's second product; T_VFULL v / T_VFREE v: V tile slot v
// landed / read by the row warps; T_OFREE / T_OSTAGE: the output staging tile may be
// written / holds a chunk's outputs (T_VFREE is committed by the product V^T I). Products: T_C1 (D1 = [K H | Q H] done), T_C4 (the
// state update done), T_C2 (D2 = [T R | P T R] done). Warps: T_R (R^T stored, D1's K half
// read), T_VN (Vn'^T stored, D2's top read), T_H (the scaled state's fp16 copy stored and
// D1's Q half read: the next chunk's first products may start), T_O (D2's bottom read).
constexpr int kPSlots = 2, kVSlots = 2;
enum TmBar { T_FULL0 = 0, T_FREE0 = 4, T_PFULL0 = 8, T_PFREE0 = T_PFULL0 + kPSlots, T_VFULL0 = T_PFREE0 + kPSlots,
             T_VFREE0 = T_VFULL0 + kVSlots, T_C1 = T_VFREE0 + kVSlots, T_C2, T_C4, T_R, T_VN, T_O, T_H, T_OFREE,
             T_OSTAGE, T_GFULL, T_GFREE, T_OFULL, T_DRAIN, T_COUNT };
static_assert(T_FREE0 >= T_FULL0 + 4 && T_PFULL0 >= T_FREE0 + 4, "barrier ranges overlap");

// EPI (the output step fused): one V slot, and a gate tile in the second one's place
template <int DK, bool EPI>
struct TmSmem {
    static constexpr int kStages = DK == 128 ? 3 : 4;
    static constexpr int kVS = EPI ? 1 : kVSlots;
    static constexpr uint32_t kBlocks = DK / 64;
    static constexpr uint32_t kStage = kBlocks * 2 * kTileBytes;   // [K_b; Q_b] for each 64-column dk block
    static constexpr uint32_t kP = kStages * kStage;                // kPSlots x (X, [T; P T])
    static constexpr uint32_t kPSlot = kXBytes + kTPTBytes;
    static constexpr uint32_t kV = kP + kPSlots * kPSlot;           // kVS V tiles (64 tokens x 128 dv)
    static constexpr uint32_t kO = kV + kVS * 2 * kTileBytes;       // output staging tile (64 tokens x 128 dv)
    static constexpr uint32_t kG = kO + 2 * kTileBytes;             // gate tile (64 tokens x 128 dv), EPI only
    static constexpr uint32_t kI = kG + (EPI ? 2 * kTileBytes : 0); // 64 x 64 fp16 identity (K-major)
    static constexpr uint32_t kArr = kI + kTileBytes;               // per-warp e^gam of the chunk's tokens
    static constexpr uint32_t kBars = kArr + 16 * 32 * 4;
    static constexpr uint32_t kTotal = kBars + 256 + 1024;          // + barriers, + slack to align the base
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// IMM: the test mode of the waits (gdn_set_wait_test_mode), a separate instance
template <int DK, bool IMM, bool EPI>
__global__ void __launch_bounds__(kTmThreads, 1)
chain_tm_kernel(const __grid_constant__ TmMaps maps, const Problem p, int ntiles, int64_t nslots,
                const unsigned char *prep_out, int cbase, int cmax) {
    using L = TmSmem<DK, EPI>;
    constexpr int NS = L::kStages;
    constexpr int VS = L::kVS;
    constexpr int HC = DK / 2;            // state columns per state warp (two warps per lane group)
    extern __shared__ unsigned char smraw[];
    pdl_wait();        // the prep tiles (and everything before them) are complete
    pdl_trigger();
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const gdn_desc &d = p.d;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3;
    const int vrow = quad * 32 + lane;           // this thread's dv row (TMEM lane)
    const int half = (warp >> 2) & 1;            // row / out warps: tokens [32 half, 32 half + 32)
    int bid = blockIdx.x;
    const int tile = bid % ntiles;
    bid /= ntiles;
    const int j = bid % d.Hv;
    const int n = bid / d.Hv;
    const int dv = d.dv, Hv = d.Hv;
    const int G = Hv / d.Hk;
    const int hk = j / G;
    const int v0 = tile * 128;
    uint64_t *bar = (uint64_t *)(sm + L::kBars);
    uint32_t *tslot = (uint32_t *)(bar + T_COUNT);
    // this warp's e^gam of its half's 32 tokens of the current chunk
    float *arr = (float *)(sm + L::kArr) + (warp < 16 ? warp : 0) * 32;
    __shared__ volatile int s_err;
    __shared__ int s_skip;
    if (tid == 0) s_skip = p.cu != nullptr && *p.status != GDN_OK;
    __syncthreads();
    if (s_skip) return;
    // chunks [cbase, cbase + cmax) of the sequence (a segment of it, or all of it)
    const int64_t sstart = p.cu ? (int64_t)p.cu[n] : (int64_t)n * d.T;
    const int64_t seq1 = p.cu ? (int64_t)p.cu[n + 1] : sstart + d.T;
    const int64_t seq0 = sstart + (int64_t)cbase * kChunk;
    const int64_t left = seq1 > seq0 ? (seq1 - seq0 + kChunk - 1) / kChunk : 0;
    const int nch = (int)(left < cmax ? left : cmax);
    const int64_t slot0 = (p.cu ? (int64_t)p.chunk_off[n] : (int64_t)n * ((d.T + kChunk - 1) / kChunk)) + cbase;
    const size_t sbase = ((size_t)n * Hv + j) * DK * dv;
    const float *gw = (const float *)p.gamma + (int64_t)j * p.ntok;
    auto tok0 = [&](int c) { return seq0 + (int64_t)c * kChunk; };
    auto clen = [&](int c) {
        const int64_t r = seq1 - tok0(c);
        return r < kChunk ? (int)r : kChunk;
    };

    if (tid == 0) {
        s_err = 0;
        for (int i = 0; i < T_COUNT; ++i) {
            const bool warps8 = i == T_R || i == T_VN || i == T_O || i == T_H || i == T_OSTAGE || i == T_GFREE ||
                                i == T_OFULL;
            mbar_init(&bar[i], warps8 ? 8 : 1);
        }
        mbar_init_fence();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // a phase that has completed costs one barrier test; the error flag is read only
    // when it has not
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (IMM ? mbar_test_now(&bar[b], parity) : mbar_test(&bar[b], parity)) return true;
        if (s_err) return false;
        if (!mbar_wait(&bar[b], parity, IMM)) { s_err = 1; return false; }
        return true;
    };
    auto warp_arrive = [&](int b) {   // after this warp's tensor-memory accesses
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[b]);
    };
    const bool out_warp = warp >= kRowW && warp < kMmaW;
    // state warps: H^T (row vrow, dk columns [half*HC, half*HC + HC)) and its fp16 copy
    if (out_warp) {
#pragma unroll
        for (int q = 0; q < HC / 32; ++q) {
            float t[32], h[16];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int dd = half * HC + 32 * q + k;
                t[k] = p.h0 ? p.h0[sbase + (size_t)dd * dv + v0 + vrow] : 0.f;
            }
            tmem_st32(tbase + lane_off + kTH + half * HC + 32 * q, t);
#pragma unroll
            for (int k = 0; k < 16; ++k) h[k] = __uint_as_float(pack_h2(t[2 * k], t[2 * k + 1]));
            tmem_st16(tbase + lane_off + kTH16 + half * (HC / 2) + 16 * q, h);
        }
    }
    {   // the identity B operand of V^T I: element (n, k) = [n == k], 128-byte swizzled rows
        unsigned char *idt = sm + L::kI;
        for (int e = tid; e < kChunk * 8; e += kTmThreads) {
            const int n = e >> 3, jc = e & 7;   // row n, 16-byte chunk jc (k = 8 jc .. 8 jc + 7)
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if ((n >> 3) == jc) (&u.x)[(n & 7) >> 1] = (n & 1) ? 0x3C000000u : 0x00003C00u;
            *reinterpret_cast<uint4 *>(idt + n * 128 + ((jc ^ (n & 7)) << 4)) = u;
        }
        fence_async_smem();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    int tma_armed = 0, p_armed = 0, v_armed = 0, g_armed = 0;   // chunks whose loads the TMA thread issued
    if (warp == kTmaW) {
        // ------------------------------------------------------------ TMA warp
        if (lane == 0) {
            auto load_kq = [&](int c) {
                const int s = c % NS;
                unsigned char *st = sm + s * L::kStage;
                const int y = (int)((int64_t)hk * p.ntok + tok0(c));
                mbar_expect_tx(&bar[T_FULL0 + s], L::kStage);
                for (int b = 0; b < (int)L::kBlocks; ++b) {
                    tma_load_2d(st + b * 2 * kTileBytes, &maps.k_hi, 64 * b, y, &bar[T_FULL0 + s]);
                    tma_load_2d(st + b * 2 * kTileBytes + kTileBytes, &maps.q_hi, 64 * b, y, &bar[T_FULL0 + s]);
                }
            };
            auto load_prep = [&](int c) {   // X (not for a first chunk) and [T; P T]
                const int ps = c % kPSlots;
                unsigned char *dst = sm + L::kP + ps * L::kPSlot;
                mbar_expect_tx(&bar[T_PFULL0 + ps], kTPTBytes + (c > 0 ? kXBytes : 0));
                if (c > 0)
                    bulk_load(dst, prep_out + ((int64_t)(hk * G) * nslots + slot0 + c) * kPrepOut + kTPTBytes,
                              kXBytes, &bar[T_PFULL0 + ps]);
                bulk_load(dst + kXBytes, prep_out + ((int64_t)j * nslots + slot0 + c) * kPrepOut, kTPTBytes,
                          &bar[T_PFULL0 + ps]);
            };
            auto load_v = [&](int c) {
                const int sv = c % VS;
                unsigned char *dst = sm + L::kV + sv * 2 * kTileBytes;
                const int y = (int)((int64_t)j * p.ntok + tok0(c));
                mbar_expect_tx(&bar[T_VFULL0 + sv], 2 * kTileBytes);
                tma_load_2d(dst, &maps.v, v0, y, &bar[T_VFULL0 + sv]);
                tma_load_2d(dst + kTileBytes, &maps.v, v0 + 64, y, &bar[T_VFULL0 + sv]);
            };
            // the fused output step's gate rows of chunk c (rows past the tensor read zeros)
            auto load_gate = [&](int c) {
                const int y = (int)tok0(c);
                mbar_expect_tx(&bar[T_GFULL], 2 * kTileBytes);
                tma_load_2d(sm + L::kG, &maps.gate, j * dv + v0, y, &bar[T_GFULL]);
                tma_load_2d(sm + L::kG + kTileBytes, &maps.gate, j * dv + v0 + 64, y, &bar[T_GFULL]);
            };
            for (int c = 0; c < nch; ++c) {
                // stage c % NS is free once the state update of chunk c - NS is done
                if (c >= NS && !wait(T_FREE0 + c % NS, (uint32_t)((c / NS) - 1) & 1)) break;
                load_kq(c);
                tma_armed = c + 1;
                // V slot c % 2 once the row warps have read chunk c - 2's V
                if (c >= VS && !wait(T_VFREE0 + c % VS, (uint32_t)((c / VS) - 1) & 1)) break;
                load_v(c);
                v_armed = c + 1;
                // prep slot c % 2 once the second product of chunk c - 2 has read it
                if (c >= kPSlots && !wait(T_PFREE0 + c % kPSlots, (uint32_t)((c / kPSlots) - 1) & 1)) break;
                load_prep(c);
                p_armed = c + 1;
                if (EPI) {
                    // the gate tile once the out warps have read chunk c - 1's
                    if (c >= 1 && !wait(T_GFREE, (uint32_t)(c - 1) & 1)) break;
                    load_gate(c);
                    g_armed = c + 1;
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaW) {
        // ------------------------------------------------------------ MMA warp
        if (lane == 0) {
            const uint32_t id128 = idesc_f16(128, 128, false, false);
            const uint32_t idH = idesc_f16(128, DK, false, true);   // B = K, MN-major (dk contiguous)
            // descriptors are built once; an offset adds (bytes >> 4) to the start field
            // (shared addresses stay below 2^18, so the 14-bit field never carries)
            const uint64_t dK0 = sw128_desc(smem_u32(sm), 16, 1024);              // K-major tiles
            const uint64_t dKt0 = sw128_desc(smem_u32(sm), 2 * kTileBytes, 1024); // K as MN-major B
            const uint64_t stg = L::kStage >> 4, pslot = L::kPSlot >> 4;
            const uint64_t dP0 = dK0 + (L::kP >> 4);
            // V^T I into D2's top half: A = the V slot (dv contiguous: MN-major, two 64-wide
            // dv blocks a tile apart), B = the identity; the V slot is free once it is done
            const uint32_t idV = idesc_f16(128, 64, true, false);
            const uint64_t dV0 = sw128_desc(smem_u32(sm + L::kV), kTileBytes, 1024);
            const uint64_t dI = sw128_desc(smem_u32(sm + L::kI), 16, 1024);
            auto cvv = [&](int sv) {
                const uint64_t a0 = dV0 + (uint64_t)sv * ((2 * kTileBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(tbase + kTD2, a0 + (uint64_t)(128 * kk), dI + (uint64_t)(2 * kk), idV, kk != 0);
                mma_commit(&bar[T_VFREE0 + sv]);
            };
            // D1 = H16^T [K; Q]^T over dk ([K_b; Q_b] is a 128-row K-major tile per block)
            auto c1a = [&](int s) {
                const uint64_t b0 = dK0 + s * stg;
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks)
                    mma_f16_ta(tbase + kTD1, tbase + kTH16 + 8 * ks,
                               b0 + (uint64_t)(((ks >> 2) * 2 * kTileBytes + 32 * (ks & 3)) >> 4), id128, ks != 0);
            };
            // D1 += Vn'^T_{c-1} X^T (X: 128 rows of [K_c; Q_c] tokens x 64 tokens of c-1)
            auto c1b = [&](int ps) {
                const uint64_t b0 = dP0 + ps * pslot;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16_ta(tbase + kTD1, tbase + kTVN + 8 * kk, b0 + (uint64_t)(2 * kk), id128, 1);
            };
            // H^T += Vn'^T K (K of stage s as an MN-major B: tokens are K, dk is N)
            auto c4 = [&](int s) {
                const uint64_t b0 = dKt0 + s * stg;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16_ta(tbase + kTH, tbase + kTVN + 8 * kk, b0 + (uint64_t)(128 * kk), idH, 1);
                mma_commit(&bar[T_FREE0 + s]);
            };
            // the barriers each step needs are tested together (one round trip)
            auto wait2 = [&](int b1, uint32_t p1, int b2, uint32_t p2) -> bool {
                if (mbar_test2<IMM>(&bar[b1], p1, &bar[b2], p2)) return true;
                return wait(b1, p1) && wait(b2, p2);
            };
            auto wait3 = [&](int b1, uint32_t p1, int b2, uint32_t p2, int b3, uint32_t p3) -> bool {
                if (mbar_test3<IMM>(&bar[b1], p1, &bar[b2], p2, &bar[b3], p3)) return true;
                return wait(b1, p1) && wait(b2, p2) && wait(b3, p3);
            };
            int c = 0;
            for (; c < nch; ++c) {
                const int s = c % NS, ps = c % kPSlots, sv = c % VS;
                const uint32_t fs = (uint32_t)(c / NS) & 1, fp = (uint32_t)(c / kPSlots) & 1,
                               fv = (uint32_t)(c / VS) & 1, f1 = (uint32_t)(c - 1) & 1;
                // the stage, the prep slot and (c >= 1) H16 = e^{gL_{c-1}} H_{c-2} with D1's Q
                // half of chunk c-1 read by the out warps (its K half was read before R_{c-1}):
                // D1 may be overwritten while the second product of chunk c-1 still runs
                if (c >= 1 ? !wait3(T_FULL0 + s, fs, T_PFULL0 + ps, fp, T_H, f1)
                           : !wait2(T_FULL0 + s, fs, T_PFULL0 + ps, fp))
                    break;
                fence_after_sync();
                c1a(s);
                // Vn'_{c-1} (D2's top half read) and the V tile of chunk c
                if (c >= 1 ? !wait2(T_VN, f1, T_VFULL0 + sv, fv) : !wait(T_VFULL0 + sv, fv)) break;
                fence_after_sync();
                if (c >= 1) c1b(ps);
                cvv(sv);   // V^T of chunk c into D2's top half
                mma_commit(&bar[T_C1]);
                if (c >= 1) c4((c - 1) % NS);
                // C4 of chunk c-1 (for c = 0: the first product, which read H16 = H_init)
                mma_commit(&bar[T_C4]);
                // R_c, and D2 of chunk c-1 read by the out warps
                if (c >= 1 ? !wait2(T_R, (uint32_t)c & 1, T_O, f1) : !wait(T_R, (uint32_t)c & 1)) break;
                fence_after_sync();
                const uint64_t bt = dP0 + ps * pslot + (kXBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16_ta(tbase + kTD2, tbase + kTR + 8 * kk, bt + (uint64_t)(2 * kk), id128, kk != 0);
                mma_commit(&bar[T_C2]);
                mma_commit(&bar[T_PFREE0 + ps]);
            }
            if (c == nch && nch > 0) {   // the state update of the last chunk
                if (wait(T_VN, (uint32_t)(nch - 1) & 1) && wait(T_H, (uint32_t)(nch - 1) & 1)) {
                    fence_after_sync();
                    c4((nch - 1) % NS);
                    mma_commit(&bar[T_C4]);
                }
            }
        }
        __syncwarp();
    } else if (warp < kRowW) {
        // ------------------------------------------------------------ row warps
        // lane l loads the decay of token 32 half + l two chunks ahead (one chunk is
        // shorter than a DRAM round trip). beta and e^{gam_L - gam} are folded into
        // the prep tile and V^T is in D2's top half, so R~ = V - e^gam (K H) and the
        // tile's product is Vn' itself.
        float A = 0.f, B = 0.f;
        auto prefetch = [&](int c, float &x) {
            const int64_t t0 = tok0(c);
            const int len = clen(c);
            const int i = 32 * half + lane;
            x = gw[t0 + (i < len ? i : len - 1)];
        };
        const float4 *a4 = reinterpret_cast<const float4 *>(arr);
        // a chunk's e^gam, one per lane, published to the warp's array
        auto publish = [&](float g) {
            __syncwarp();                 // the previous chunk's reads of the array are done
            arr[lane] = __expf(g);
            __syncwarp();
        };
        if (nch > 0) prefetch(0, A);
        if (nch > 1) prefetch(1, B);
        if (nch > 0) publish(A);
        for (int c = 0; c < nch; ++c) {
            // R~^T = V - e^gam (K H) for this half's 32 tokens (tokens past the sequence's
            // end hold other rows' values: beta = 0 in the tile removes them)
            if (!wait(T_C1, (uint32_t)c & 1)) break;
            fence_after_sync();
            float a[32], v[32];
            tmem_ld32x2(tbase + lane_off + kTD1 + 32 * half, tbase + lane_off + kTD2 + 32 * half, a, v);
            float r[16];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 e4 = a4[m];
                const float2 x0 = fma2(make_float2(-e4.x, -e4.y), make_float2(a[4 * m], a[4 * m + 1]),
                                       make_float2(v[4 * m], v[4 * m + 1]));
                const float2 x1 = fma2(make_float2(-e4.z, -e4.w), make_float2(a[4 * m + 2], a[4 * m + 3]),
                                       make_float2(v[4 * m + 2], v[4 * m + 3]));
                r[2 * m] = __uint_as_float(pack_h2(x0.x, x0.y));
                r[2 * m + 1] = __uint_as_float(pack_h2(x1.x, x1.y));
            }
            tmem_st16(tbase + lane_off + kTR + 16 * half, r);
            warp_arrive(T_R);
            // Vn'^T: the top half of D2, to fp16
            if (!wait(T_C2, (uint32_t)c & 1)) break;
            fence_after_sync();
            tmem_ld32(tbase + lane_off + kTD2 + 32 * half, a);
#pragma unroll
            for (int m = 0; m < 16; ++m) r[m] = __uint_as_float(pack_h2(a[2 * m], a[2 * m + 1]));
            tmem_st16(tbase + lane_off + kTVN + 16 * half, r);
            warp_arrive(T_VN);
            A = B;                                   // chunk c + 1 (loaded a chunk ago)
            if (c + 2 < nch) prefetch(c + 2, B);
            if (c + 1 < nch) publish(A);
        }
    } else if (out_warp) {
        // ------------------------------------------------ state and output warps
        __half *o = (__half *)p.o;
        auto store_final = [&]() {
#pragma unroll
            for (int q = 0; q < HC / 32; ++q) {
                float t[32];
                tmem_ld32(tbase + lane_off + kTH + half * HC + 32 * q, t);
#pragma unroll
                for (int k = 0; k < 32; ++k) p.hT[sbase + (size_t)(half * HC + 32 * q + k) * dv + v0 + vrow] = t[k];
            }
        };
        // the decay of this lane's token and the chunk's last decay
        auto decays = [&](int c, float &g_tok, float &g_last) {
            const int64_t t0 = tok0(c);
            const int len = clen(c);
            const int i = 32 * half + lane;
            g_tok = gw[t0 + (i < len ? i : len - 1)];
            g_last = gw[t0 + len - 1];
        };
        // one thread issues the output tile's tensor stores; nfree / nstage count the
        // phases of T_OFREE / T_OSTAGE
        const bool storer = warp == kRowW && lane == 0;
        int nfree = 0, nstage = 0;
        // the fused output step: this thread's 8 norm weights (dv 8 (lane % 16) ..) as pairs
        const bool bf16_act = d.dtype == GDN_BF16;
        bool out_finite = true;
        float2 nw[4] = {};
        if (EPI) {
            const int cw = v0 + 8 * (lane & 15);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float w0, w1;
                if (d.norm_w_dtype == GDN_F32) {
                    w0 = ((const float *)p.norm_w)[cw + 2 * i];
                    w1 = ((const float *)p.norm_w)[cw + 2 * i + 1];
                } else if (bf16_act) {
                    w0 = __bfloat162float(((const __nv_bfloat16 *)p.norm_w)[cw + 2 * i]);
                    w1 = __bfloat162float(((const __nv_bfloat16 *)p.norm_w)[cw + 2 * i + 1]);
                } else {
                    w0 = __half2float(((const __half *)p.norm_w)[cw + 2 * i]);
                    w1 = __half2float(((const __half *)p.norm_w)[cw + 2 * i + 1]);
                }
                nw[i] = make_float2(w0, w1);
            }
        }
        // two chunks ahead: chunk c's values move into place at the end of iteration c - 1,
        // one iteration after their loads were issued, so no move waits on a load in flight
        float g_tok = 0.f, g_last = 0.f, g_tok_n = 0.f, g_last_n = 0.f;
        if (nch > 0) decays(0, g_tok, g_last);
        if (nch > 1) decays(1, g_tok_n, g_last_n);
        for (int c = 0; c < nch; ++c) {
            // H_{c-1} is complete (or, for c = 0, the first product has read H16 = H_init):
            // scale by e^{gL_c} for chunk c's update and publish its fp16 copy for chunk c+1
            if (!wait(T_C4, (uint32_t)c & 1)) break;
            fence_after_sync();
            {   // on the path to the next chunk's first products: the stores go out without
                // waiting one by one, one wait at the end
                const float el = __expf(g_last);
                const float2 e2 = make_float2(el, el);
#pragma unroll
                for (int q = 0; q < HC / 32; ++q) {
                    float t[32];
                    tmem_ld32(tbase + lane_off + kTH + half * HC + 32 * q, t);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 x = mul2(make_float2(t[2 * k], t[2 * k + 1]), e2);
                        t[2 * k] = x.x;
                        t[2 * k + 1] = x.y;
                    }
                    tmem_st32_nw(tbase + lane_off + kTH + half * HC + 32 * q, t);
                    if (c + 1 < nch) {
                        float h[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) h[k] = __uint_as_float(pack_h2(t[2 * k], t[2 * k + 1]));
                        tmem_st16_nw(tbase + lane_off + kTH16 + half * (HC / 2) + 16 * q, h);
                    }
                }
                tmem_wait_st();
            }
            // D1's Q half, Q H_{c-1} for this half's tokens (complete: C4 follows the first
            // products of chunk c); once read, the next chunk's first products may overwrite D1.
            // Read in the 16x256b layout (lanes g = lane / 4 and g + 8 of each 16-lane half,
            // token pairs 8i + tq, 8i + tq + 1), whose pairs stmatrix stores transposed.
            const uint32_t lq = tbase + ((uint32_t)(quad * 32) << 16);
            const uint32_t cq = (uint32_t)(64 + 32 * half);
            float qa[16], qb[16];   // lanes [0, 16) and [16, 32) of the warp's quarter
            tmem_ld16x256_x4x2(lq + kTD1 + cq, lq + (16u << 16) + kTD1 + cq, qa, qb);
            warp_arrive(T_H);
            __syncwarp();                 // the previous chunk's reads of the array are done
            arr[lane] = d.scale * __expf(g_tok);   // P' carries the scale already
            __syncwarp();
            // O^T = scale e^gam (Q H)^T + bottom half of D2^T for this half's 32 tokens
            if (!wait(T_C2, (uint32_t)c & 1)) break;
            fence_after_sync();
            float pa[16], pb[16];
            tmem_ld16x256_x4x2(lq + kTD2 + cq, lq + (16u << 16) + kTD2 + cq, pa, pb);
            warp_arrive(T_O);
            const int tq = 2 * (lane & 3), g8 = lane >> 2;
            // h[4i + m]: matrix m of token group i (m = 2 lane-half + (lane g or g + 8))
            uint32_t h[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 e = *reinterpret_cast<const float2 *>(arr + 8 * i + tq);
                const float2 x0 = fma2(e, make_float2(qa[4 * i], qa[4 * i + 1]), make_float2(pa[4 * i], pa[4 * i + 1]));
                const float2 x1 = fma2(e, make_float2(qa[4 * i + 2], qa[4 * i + 3]), make_float2(pa[4 * i + 2], pa[4 * i + 3]));
                const float2 y0 = fma2(e, make_float2(qb[4 * i], qb[4 * i + 1]), make_float2(pb[4 * i], pb[4 * i + 1]));
                const float2 y1 = fma2(e, make_float2(qb[4 * i + 2], qb[4 * i + 3]), make_float2(pb[4 * i + 2], pb[4 * i + 3]));
                h[4 * i] = pack_h2(x0.x, x0.y);
                h[4 * i + 1] = pack_h2(x1.x, x1.y);
                h[4 * i + 2] = pack_h2(y0.x, y0.y);
                h[4 * i + 3] = pack_h2(y1.x, y1.y);
            }
            const int64_t t0 = tok0(c);
            const int len = clen(c);
            if (EPI || len == kChunk) {
                // through the staging tile: a full chunk leaves with one tensor store per 64
                // columns; with the fused output step every chunk is staged
                if (storer) {
                    bulk_wait_read();                     // the previous store has read the tile
                    mbar_arrive(&bar[T_OFREE]);
                }
                if (!wait(T_OFREE, (uint32_t)nfree & 1)) break;
                ++nfree;
                // this thread addresses row lane % 8 (a token) of stored matrix m = lane / 8:
                // 8 dv columns from 32 quad + 16 (m / 2) + 8 (m % 2)
                const int m = lane >> 3, rr = lane & 7;
                const int dvl = 32 * quad + 16 * (m >> 1) + 8 * (m & 1);
                const uint32_t obox = smem_u32(sm + L::kO) + (uint32_t)(dvl >> 6) * kTileBytes;
                const uint32_t ochk = (uint32_t)(((dvl & 63) >> 3) ^ rr) << 4;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    stmatrix_x4_trans(obox + (uint32_t)(32 * half + 8 * i + rr) * 128 + ochk, h[4 * i], h[4 * i + 1],
                                      h[4 * i + 2], h[4 * i + 3]);
                if (EPI) {
                    // the gated RMSNorm over whole rows once every out warp's o is in the tile:
                    // 16 lanes per token, 8 consecutive dv each, the same arithmetic (and order
                    // of the sums) as the separate output step, in place in the tile
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[T_OFULL]);
                    if (!wait(T_OFULL, (uint32_t)c & 1) || !wait(T_GFULL, (uint32_t)c & 1)) break;
                    const int ot = (warp - kRowW) * 32 + lane;
                    const uint32_t cb = (uint32_t)(ot & 15);
#pragma unroll
                    for (int sg = 0; sg < 4; ++sg) {
                        const int r = (ot >> 4) + 16 * sg;
                        const uint32_t off = (cb >> 3) * kTileBytes + (uint32_t)r * 128 + (((cb & 7) ^ (uint32_t)(r & 7)) << 4);
                        float2 x[4];
                        Pairs<__half>::unpack(*reinterpret_cast<const uint4 *>(sm + L::kO + off), x);
                        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 4; ++i) ss2 = fma2(x[i], x[i], ss2);
                        float ss = ss2.x + ss2.y;
#pragma unroll
                        for (int sh = 8; sh >= 1; sh >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, sh);
                        if (r < len) out_finite = out_finite && isfinite(ss);
                        const float2 inv = splat2(rsqrtf(ss * (1.0f / (float)dv) + d.norm_eps));
                        const uint4 gu = *reinterpret_cast<const uint4 *>(sm + L::kG + off);
                        float2 gp[4], y[4];
                        uint4 pk;
                        if (bf16_act) {
                            Pairs<__nv_bfloat16>::unpack(gu, gp);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                y[i] = mul2(Pairs<__nv_bfloat16>::round(mul2(nw[i], mul2(x[i], inv))), silu2_fast(gp[i]));
                            pk = Pairs<__nv_bfloat16>::pack(y);
                        } else {
                            Pairs<__half>::unpack(gu, gp);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                y[i] = mul2(Pairs<__half>::round(mul2(nw[i], mul2(x[i], inv))), silu2_fast(gp[i]));
                            pk = Pairs<__half>::pack(y);
                        }
                        if (len == kChunk)
                            *reinterpret_cast<uint4 *>(sm + L::kO + off) = pk;
                        else if (r < len)
                            *reinterpret_cast<uint4 *>((unsigned char *)p.out +
                                                       ((t0 + r) * (int64_t)Hv * dv + (int64_t)j * dv + v0 + 8 * cb) * 2) = pk;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[T_GFREE]);   // this warp's gate reads are done
                }
                if (len == kChunk) {
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[T_OSTAGE]);
                    if (storer) {
                        if (!wait(T_OSTAGE, (uint32_t)nstage & 1)) break;
                        const CUtensorMap *om = EPI ? &maps.out : &maps.o;
                        tma_store_2d(om, j * dv + v0, (int)t0, sm + L::kO);
                        tma_store_2d(om, j * dv + v0 + 64, (int)t0, sm + L::kO + kTileBytes);
                        bulk_commit();
                    }
                    ++nstage;
                }
            } else {
                // the last, partial chunk of a sequence: the tile's other rows belong to the next
                __half *dst = o + (int64_t)j * dv + v0 + 32 * quad + g8;
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const __half2 hv = *reinterpret_cast<const __half2 *>(&h[4 * i + mm]);
                        const int dvo = 16 * (mm >> 1) + 8 * (mm & 1);
#pragma unroll
                        for (int e2 = 0; e2 < 2; ++e2) {
                            const int tok = 32 * half + 8 * i + tq + e2;
                            if (tok < len) dst[(t0 + tok) * (int64_t)Hv * dv + dvo] = e2 ? __high2half(hv) : __low2half(hv);
                        }
                    }
            }
            g_tok = g_tok_n;
            g_last = g_last_n;
            if (c + 2 < nch) decays(c + 2, g_tok_n, g_last_n);
        }
        if (storer) bulk_wait();   // the output stores are complete before the CTA leaves
        // a non-finite gated-delta-rule output (unless an earlier error was recorded)
        if (EPI && !out_finite) atomicCAS(p.status, GDN_OK, GDN_ERR_DEVICE_RANGE);
        if (p.hT && !s_err) {
            if (nch == 0) {
                store_final();
            } else if (wait(T_C4, (uint32_t)nch & 1)) {
                fence_after_sync();
                store_final();
            }
        }
    }
    __syncthreads();
    if (s_err) {
        // drain: this CTA's own copies and products, bounded, before the tensor memory is freed
        if (tid == kMmaW * 32) {
            atomicCAS(p.status, GDN_OK, GDN_ERR_DEVICE_TIMEOUT);
            mma_commit(&bar[T_DRAIN]);
            mbar_wait(&bar[T_DRAIN], 0);
        }
        if (tid == kTmaW * 32) {
            for (int c = tma_armed - NS < 0 ? 0 : tma_armed - NS; c < tma_armed; ++c)
                mbar_wait(&bar[T_FULL0 + c % NS], (uint32_t)(c / NS) & 1);
            for (int c = p_armed - kPSlots < 0 ? 0 : p_armed - kPSlots; c < p_armed; ++c)
                mbar_wait(&bar[T_PFULL0 + c % kPSlots], (uint32_t)(c / kPSlots) & 1);
            for (int c = v_armed - VS < 0 ? 0 : v_armed - VS; c < v_armed; ++c)
                mbar_wait(&bar[T_VFULL0 + c % VS], (uint32_t)(c / VS) & 1);
            if (EPI && g_armed > 0) mbar_wait(&bar[T_GFULL], (uint32_t)(g_armed - 1) & 1);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

int max_dyn_smem_tm() {
    int dev = 0, v = 232448;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return v;
}

template <int DK>
cudaError_t launch_tm(const Problem &p, cudaStream_t s, const unsigned char *prep_out, int64_t nslots_alloc,
                      int cbase, int cmax, bool pdl, unsigned nblocks) {
    const gdn_desc &d = p.d;
    TmMaps m;
    if (p.ntok > 0) {
        if (!encode_tile_map(&m.q_hi, p.q, (uint64_t)d.Hk * p.ntok, DK) ||
            !encode_tile_map(&m.k_hi, p.k, (uint64_t)d.Hk * p.ntok, DK) ||
            !encode_tile_map(&m.v, p.v, (uint64_t)d.Hv * p.ntok, d.dv) ||
            !encode_tile_map(&m.o, p.o, (uint64_t)p.ntok, (uint64_t)d.Hv * d.dv))
            return cudaErrorInvalidValue;
        if (p.fuse_epilogue) {
            // the gate view's rows are tokens (one sequence row, or batches back to back)
            const uint64_t grows = p.cu ? (uint64_t)p.ntok : (uint64_t)d.B * d.T;
            if (!encode_tile_map_pitch(&m.gate, p.gate, grows, (uint64_t)d.Hv * d.dv, (uint64_t)d.gate_stride_t * 2) ||
                !encode_tile_map(&m.out, p.out, (uint64_t)p.ntok, (uint64_t)d.Hv * d.dv))
                return cudaErrorInvalidValue;
        } else {
            memset(&m.gate, 0, sizeof(m.gate));
            memset(&m.out, 0, sizeof(m.out));
        }
    } else {
        memset(&m, 0, sizeof(m));   // no chunks: the kernel only copies the initial state
    }
    const int maxs = max_dyn_smem_tm();
    // all 512 TMEM columns: enough shared memory that a second CTA never shares the SM
    size_t smem = p.fuse_epilogue ? TmSmem<DK, true>::kTotal : TmSmem<DK, false>::kTotal;
    if (smem < (size_t)(maxs / 2 + 1024)) smem = (size_t)(maxs / 2 + 1024);
    if ((int)smem > maxs) return cudaErrorInvalidValue;
    auto kernel = p.fuse_epilogue ? (p.wait_immediate ? chain_tm_kernel<DK, true, true> : chain_tm_kernel<DK, false, true>)
                                  : (p.wait_immediate ? chain_tm_kernel<DK, true, false> : chain_tm_kernel<DK, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (nblocks == 0) return cudaSuccess;
    return launch_kernel(pdl, kernel, dim3(nblocks), dim3(kTmThreads), smem, s, m, p, d.dv / 128, nslots_alloc,
                         prep_out, cbase, cmax);
}

}  // namespace

bool chain_tm_supports(const gdn_desc &d) {
    return (d.dtype == GDN_BF16 || d.dtype == GDN_F16) && (d.dk == 64 || d.dk == 128) && d.dv >= 128 &&
           d.dv % 128 == 0;
}

int chain_tm_tiles(const gdn_desc &d) { return d.dv / 128; }

// The output step (gated RMSNorm over dv) fused into the transposed chain: one CTA
// holds a token's whole row when dv = 128; the gate must be a 16-bit view whose rows
// a tensor map can address (16-byte aligned base and row pitch, batches back to back).
// Not for the segmented schedule: the fused instance keeps one V slot (the gate tile
// takes the other), too shallow beside the prep segments (one 131072-token sequence:
// 5.1 -> 6.8 ms per step).
bool chain_tm_fuses_epilogue(const Problem &p) {
    const gdn_desc &d = p.d;
    if (!chain_tm_supports(d) || d.dv != 128 || p.ntok == 0 || !p.gate || !p.out || p.rec_o) return false;
    if (chunk_tc_segmented(p)) return false;
    if (d.gate_dtype != d.dtype || (d.norm_w_dtype != d.dtype && d.norm_w_dtype != GDN_F32)) return false;
    if ((uintptr_t)p.gate % 16 != 0 || (uintptr_t)p.out % 16 != 0 || (d.gate_stride_t * 2) % 16 != 0 ||
        d.gate_stride_t < (int64_t)d.Hv * d.dv)
        return false;
    return p.cu != nullptr || d.B == 1 || d.gate_stride_b == (int64_t)d.T * d.gate_stride_t;
}

cudaError_t launch_chain_tm(const Problem &p, cudaStream_t s, const unsigned char *prep_out, int64_t nslots_alloc,
                            int cbase, int cmax, bool pdl, unsigned nblocks) {
    return p.d.dk == 128 ? launch_tm<128>(p, s, prep_out, nslots_alloc, cbase, cmax, pdl, nblocks)
                         : launch_tm<64>(p, s, prep_out, nslots_alloc, cbase, cmax, pdl, nblocks);
}

}  // namespace gdn
