// gdn_static_ws.cu -- gdn_forward for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc or an allocating library routine:
// code that runs inside another framework's memory arena, plugins that are not
// handed an allocator, or hosts that forbid allocation once they are serving.
// For them this file keeps the forward's scratch in a fixed device array
// compiled into the library. Every GPU that loads the library holds the array
// (GDN_STATIC_WORKSPACE_BYTES) until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host it is only a
// stand-in symbol, not a device address. The device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made on the
// device, and again whenever the device's current context has changed since
// (after a cudaDeviceReset the module is loaded anew, possibly elsewhere).
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[GDN_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
struct Cached {
    void *ptr = nullptr;
    CUcontext ctx = nullptr;
};
Cached g_static_ws_ptr[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 ctx_fn() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuCtxGetCurrent_v4000) nullptr;
        return (PFN_cuCtxGetCurrent_v4000)f;
    }();
    return fn;
}

// Device address of g_static_ws on the current device (set up on first use and
// whenever the device's context is not the one the address was taken in).
int static_ws_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    // the same device again: initialises its primary context if needed and makes it
    // current on this thread, so that the driver reports the context in use
    if (cudaSetDevice(dev) != cudaSuccess) return GDN_ERR_CUDA;
    CUcontext ctx = nullptr;
    auto get_ctx = ctx_fn();
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    Cached &c = g_static_ws_ptr[dev];
    if (c.ptr == nullptr || c.ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return GDN_ERR_CUDA;
        c.ptr = p;
        c.ctx = ctx;
    }
    *out = c.ptr;
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_forward_static_ws(const gdn_desc *d, const void *q_raw, const void *k_raw,
                                     const void *v_raw, const void *a, const void *b,
                                     const void *gate, const void *conv_w, const float *A_log,
                                     const float *dt_bias, const void *norm_w,
                                     const int32_t *cu_seqlens, const float *initial_state,
                                     void *out, float *final_state, gdn_stream_t stream) {
    if (!d) return GDN_ERR_INVALID_ARG;
    size_t need = 0;
    int rc = gdn_workspace_bytes(d, &need);
    if (rc != GDN_OK) return rc;
    if (need > (size_t)GDN_STATIC_WORKSPACE_BYTES) return GDN_ERR_WORKSPACE;
    void *ws = nullptr;
    if ((rc = static_ws_address(&ws)) != GDN_OK) return rc;
    // Every region of the workspace (status word, chunk table, intermediates) is
    // written by this call before it is read, so the contents left by the last
    // call need no clearing.
    // one stream only: the segmented schedule of long sequences would create a
    // side stream on first use
    return gdn::forward_single_stream(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
                                      cu_seqlens, initial_state, out, final_state, ws,
                                      (size_t)GDN_STATIC_WORKSPACE_BYTES, (cudaStream_t)stream);
}

// The status word at the start of the fixed scratch: what gdn_device_status
// reads from a caller's workspace, for the calls above.
extern "C" int gdn_static_ws_device_status(int *status, gdn_stream_t stream) {
    if (!status) return GDN_ERR_INVALID_ARG;
    void *ws = nullptr;
    const int rc = static_ws_address(&ws);
    if (rc != GDN_OK) return rc;
    return gdn_device_status(ws, status, stream);
}
