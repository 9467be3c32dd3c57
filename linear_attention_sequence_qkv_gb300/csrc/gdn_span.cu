// gdn_span.cu -- composition of the affine state maps of consecutive spans of
// one sequence (the exchange step of the sequence-sharded core).
//
// Over a span of the sequence the chunked gated delta rule is affine in the
// span's initial state: H_end = A H_start + B (H = S^T, dk x dv), with A (dk x dk)
// the final state of the span run with v = 0 from the identity, and B the final
// state from zeros. Given every span's (A, B), the initial state of span s is
//     H_in[0] = h0,  H_in[s] = A[s-1] H_in[s-1] + B[s-1].
// One CTA per (v head, 32-column tile of dv) carries its H tile in shared memory
// through the spans (the spans are few: one per rank of the split).
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanCols = 32;

__global__ void __launch_bounds__(kScanThreads) span_scan_kernel(int spans, int Hv, int dk, int dv,
                                                                const float *__restrict__ A,
                                                                const float *__restrict__ B,
                                                                const float *__restrict__ h0,
                                                                float *__restrict__ H_in) {
    extern __shared__ float sm[];
    float *Hs = sm;                            // [dk][kScanCols] current state tile
    float *Hn = sm + dk * kScanCols;           // [dk][kScanCols] next
    const int j = blockIdx.x, c0 = blockIdx.y * kScanCols;
    const int ncol = min(kScanCols, dv - c0);
    const size_t st = (size_t)dk * dv, mt = (size_t)dk * dk;
    for (int idx = threadIdx.x; idx < dk * kScanCols; idx += kScanThreads) {
        const int r = idx / kScanCols, c = idx - r * kScanCols;
        Hs[idx] = (h0 && c < ncol) ? h0[(size_t)j * st + (size_t)r * dv + c0 + c] : 0.f;
    }
    __syncthreads();
    for (int s = 0; s < spans; ++s) {
        float *dst = H_in + ((size_t)s * Hv + j) * st;
        for (int idx = threadIdx.x; idx < dk * kScanCols; idx += kScanThreads) {
            const int r = idx / kScanCols, c = idx - r * kScanCols;
            if (c < ncol) dst[(size_t)r * dv + c0 + c] = Hs[idx];
        }
        if (s == spans - 1) break;
        // next = A H + B, one (row, column) per thread and step
        const float *As = A + ((size_t)s * Hv + j) * mt;
        const float *Bs = B + ((size_t)s * Hv + j) * st;
        for (int idx = threadIdx.x; idx < dk * kScanCols; idx += kScanThreads) {
            const int r = idx / kScanCols, c = idx - r * kScanCols;
            float v = c < ncol ? Bs[(size_t)r * dv + c0 + c] : 0.f;
            const float *ar = As + (size_t)r * dk;
            for (int m = 0; m < dk; ++m) v = fmaf(__ldg(ar + m), Hs[m * kScanCols + c], v);
            Hn[idx] = v;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < dk * kScanCols; idx += kScanThreads) Hs[idx] = Hn[idx];
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_span_scan(int spans, int Hv, int dk, int dv, const float *A, const float *B, const float *h0,
                             float *H_in, cudaStream_t s) {
    const size_t bytes = 2 * (size_t)dk * kScanCols * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(span_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    span_scan_kernel<<<dim3(Hv, (dv + kScanCols - 1) / kScanCols), kScanThreads, bytes, s>>>(spans, Hv, dk, dv, A, B,
                                                                                            h0, H_in);
    return cudaGetLastError();
}

}  // namespace gdn
