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
// stand-in symbol, not a device address. The device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the first
// call made on the device.
#include <mutex>

#include "gdn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[GDN_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void *g_static_ws_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (set-up on first use).
int static_ws_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_static_ws_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return GDN_ERR_CUDA;
        g_static_ws_ptr[dev] = p;
    }
    *out = g_static_ws_ptr[dev];
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
