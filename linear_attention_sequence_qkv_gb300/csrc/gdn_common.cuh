// gdn_common.cuh -- shared device helpers of the GDN core-forward kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

namespace gdn {

constexpr int kChunk = 64;   // chunk length of the chunked gated delta rule
constexpr int kConvW = 4;    // short-conv taps

// ---------------------------------------------------------------- dtypes
template <typename T> struct Dt;
template <> struct Dt<float> {
    static __device__ __forceinline__ float to_f(float x) { return x; }
    static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Dt<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Dt<__half> {
    static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

template <typename T> __device__ __forceinline__ float to_f(T x) { return Dt<T>::to_f(x); }
template <typename T> __device__ __forceinline__ T from_f(float x) { return Dt<T>::from_f(x); }

// Storage type of the intermediates (q, k, v, o) for activation type T, and the
// type of the in-chunk cumulative decay (see gdn_internal.h).
template <typename T> struct Inter { using S = __half; using G = float; };
template <> struct Inter<float> { using S = float; using G = double; };

// round a float through the storage type T and back
template <typename T> __device__ __forceinline__ float round_through(float x) {
    return to_f<T>(from_f<T>(x));
}

// 16-byte vector of T: N elements
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    union {
        uint4 u;
        T e[N];
    };
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *out) {
    Vec16<T> v;
    v.u = u;
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) out[i] = to_f<T>(v.e[i]);
}

template <typename T>
__device__ __forceinline__ void load16_f(const T *p, float *out) {
    unpack16<T>(__ldg(reinterpret_cast<const uint4 *>(p)), out);
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float *in) {
    Vec16<T> v;
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) v.e[i] = from_f<T>(in[i]);
    return v.u;
}

template <typename T>
__device__ __forceinline__ void store16_f(T *p, const float *in) {
    *reinterpret_cast<uint4 *>(p) = pack16<T>(in);
}

// streaming store that does not keep the line in L1
template <typename T>
__device__ __forceinline__ void store16_f_cs(T *p, const float *in) {
    __stcs(reinterpret_cast<uint4 *>(p), pack16<T>(in));
}

__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// silu(x) = x * (1 + tanh(x/2)) / 2 with one hardware tanh (relative error
// ~2^-11): for values that are stored or consumed at 16-bit precision
__device__ __forceinline__ float silu_fast(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return 0.5f * x * (1.0f + t);
}
// the accurate form for fp32 results, the one-instruction form for 16-bit ones
template <typename T> __device__ __forceinline__ float silu_act(float x) {
    return sizeof(T) == 4 ? silu_f(x) : silu_fast(x);
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// softplus(x) = log(1 + e^x); above 20 the correction is below fp32 resolution
__device__ __forceinline__ float softplus_f(float x) {
    return x > 20.0f ? x : log1pf(expf(x));
}

// Address of token `tok` (flattened over batch rows of T tokens) in a [B,T,*] view.
__device__ __forceinline__ int64_t tok_offset(int64_t tok, int T, int64_t sb, int64_t st) {
    const int64_t b = tok / T;
    return b * sb + (tok - b * T) * st;
}

// Largest n in [0, N] with arr[n] <= x (arr non-decreasing, arr[0] <= x).
__device__ __forceinline__ int upper_index(const int32_t *arr, int N, int64_t x) {
    int lo = 0, hi = N;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((int64_t)arr[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Sequence n's chunk `m` located from a chunk slot. Returns false if the slot is
// past the last chunk. Without cu_seqlens, sequence n spans [n*T, (n+1)*T).
struct ChunkLoc {
    int n;           // sequence
    int64_t seq0;    // first token of the sequence
    int64_t seq1;    // one past its last token
    int64_t tok0;    // first token of the chunk
    int len;         // tokens in the chunk (1..64)
};

__device__ __forceinline__ bool locate_chunk(int64_t slot, const int32_t *cu, const int32_t *chunk_off,
                                             int N, int T, ChunkLoc &c) {
    if (cu == nullptr) {
        const int cps = (T + kChunk - 1) / kChunk;
        const int64_t n = slot / cps;
        if (n >= N) return false;
        const int m = (int)(slot - n * cps);
        c.n = (int)n;
        c.seq0 = n * (int64_t)T;
        c.seq1 = c.seq0 + T;
        c.tok0 = c.seq0 + (int64_t)m * kChunk;
    } else {
        if (slot >= chunk_off[N]) return false;
        const int n = upper_index(chunk_off, N, slot);
        c.n = n;
        c.seq0 = cu[n];
        c.seq1 = cu[n + 1];
        c.tok0 = c.seq0 + (slot - chunk_off[n]) * kChunk;
    }
    const int64_t rem = c.seq1 - c.tok0;
    c.len = rem < kChunk ? (int)rem : kChunk;
    return c.len > 0;
}

}  // namespace gdn
