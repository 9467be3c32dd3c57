// gdn_common.cuh -- shared device helpers of the GDN core-forward kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

namespace gdn {

// Programmatic dependent launch. A kernel launched with the programmatic
// stream-serialisation attribute may start while the kernel before it on the
// stream is still running; pdl_wait() returns once that kernel has completed
// and its writes are visible (at once when the kernel was launched plainly).
// pdl_trigger() lets the next such kernel launch as soon as every CTA of this
// one has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args &&...args) {
    if (!pdl) {
        kernel<<<grid, block, smem, s>>>(static_cast<Args &&>(args)...);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

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

// ------------------------------------------------------ packed fp32 pairs
// sm_100-class SMs run fp32 add / mul / fma on a register pair as one
// instruction; the streaming kernels keep their values as float2 pairs.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

// 16 bytes of T as Vec16<T>::N / 2 pairs
template <typename T> struct Pairs;
template <> struct Pairs<float> {
    static __device__ __forceinline__ void unpack(const uint4 &u, float2 *o) {
        o[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        o[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    static __device__ __forceinline__ uint4 pack(const float2 *in) {
        return make_uint4(__float_as_uint(in[0].x), __float_as_uint(in[0].y), __float_as_uint(in[1].x),
                          __float_as_uint(in[1].y));
    }
    static __device__ __forceinline__ float2 round(float2 x) { return x; }
};
template <> struct Pairs<__nv_bfloat16> {
    // a bf16 is the upper half of the fp32 with the same value
    static __device__ __forceinline__ float2 word(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t pack1(float2 x) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ void unpack(const uint4 &u, float2 *o) {
        o[0] = word(u.x); o[1] = word(u.y); o[2] = word(u.z); o[3] = word(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float2 *in) {
        return make_uint4(pack1(in[0]), pack1(in[1]), pack1(in[2]), pack1(in[3]));
    }
    static __device__ __forceinline__ float2 round(float2 x) { return word(pack1(x)); }
};
template <> struct Pairs<__half> {
    static __device__ __forceinline__ float2 word(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    static __device__ __forceinline__ uint32_t pack1(float2 x) {
        __half2 h = __float22half2_rn(x);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ void unpack(const uint4 &u, float2 *o) {
        o[0] = word(u.x); o[1] = word(u.y); o[2] = word(u.z); o[3] = word(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float2 *in) {
        return make_uint4(pack1(in[0]), pack1(in[1]), pack1(in[2]), pack1(in[3]));
    }
    static __device__ __forceinline__ float2 round(float2 x) { return word(pack1(x)); }
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu(x) = x / (1 + e^-x) on a pair, e^-x = 2^(-x log2 e) from the hardware
// base-2 exponential and the quotient from the hardware reciprocal (both a few
// ulp): for values kept at fp32 precision
__device__ __forceinline__ float2 silu2_acc(float2 x) {
    const float2 m = mul2(x, splat2(-1.4426950408889634f));
    const float2 d = add2(make_float2(ex2_approx(m.x), ex2_approx(m.y)), splat2(1.0f));
    return mul2(x, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}
// silu(x) = h + h tanh(h), h = x/2, with the hardware tanh (relative error
// ~2^-11): for values stored or consumed at 16-bit precision
__device__ __forceinline__ float2 silu2_fast(float2 x) {
    const float2 h = mul2(x, splat2(0.5f));
    return fma2(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
}
template <typename T> __device__ __forceinline__ float2 silu2_act(float2 x) {
    return sizeof(T) == 4 ? silu2_acc(x) : silu2_fast(x);
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
