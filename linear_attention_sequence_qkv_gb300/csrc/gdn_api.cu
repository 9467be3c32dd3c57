// gdn_api.cu -- the C ABI (include/gdn.h): argument checks on metadata only,
// workspace layout and the kernel launches of the GDN core forward.
#include <atomic>
#include <stdint.h>
#include <string.h>

#include "gdn_internal.h"

using gdn::Layout;
using gdn::Problem;

namespace {

bool is_pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Checks every field of the descriptor. Returns GDN_OK or an error status.
int check_desc(const gdn_desc *d, bool packed) {
    if (!d) return GDN_ERR_INVALID_ARG;
    if (d->B < 1 || d->T < 0 || d->N < 1 || d->Hk < 1 || d->Hv < 1) return GDN_ERR_INVALID_ARG;
    if (packed ? d->B != 1 : d->N != d->B) return GDN_ERR_INVALID_ARG;
    if (d->dtype < GDN_F32 || d->dtype > GDN_F16) return GDN_ERR_UNSUPPORTED;
    if (d->gate_dtype != d->dtype && d->gate_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    if (d->norm_w_dtype != d->dtype && d->norm_w_dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    if (d->Hv % d->Hk != 0) return GDN_ERR_UNSUPPORTED;
    if (!is_pow2_in(d->dk, 16, 512) || !is_pow2_in(d->dv, 16, 512)) return GDN_ERR_UNSUPPORTED;
    if (d->conv_width != 4) return GDN_ERR_UNSUPPORTED;
    const int64_t strides[] = {d->q_stride_b, d->q_stride_t, d->k_stride_b, d->k_stride_t,
                               d->v_stride_b, d->v_stride_t, d->a_stride_b, d->a_stride_t,
                               d->b_stride_b, d->b_stride_t, d->gate_stride_b, d->gate_stride_t};
    for (int64_t s : strides)
        if (s < 0) return GDN_ERR_INVALID_ARG;
    const int64_t ch_qk = (int64_t)d->Hk * d->dk, ch_v = (int64_t)d->Hv * d->dv;
    if (d->T > 1 && (d->q_stride_t < ch_qk || d->k_stride_t < ch_qk || d->v_stride_t < ch_v ||
                     d->a_stride_t < d->Hv || d->b_stride_t < d->Hv || d->gate_stride_t < ch_v))
        return GDN_ERR_INVALID_ARG;
    // 16-byte vector access of q/k/v rows
    const int64_t es = (int64_t)gdn::act_size(d->dtype);
    const int64_t vs[] = {d->q_stride_b, d->q_stride_t, d->k_stride_b, d->k_stride_t,
                          d->v_stride_b, d->v_stride_t};
    for (int64_t s : vs)
        if ((s * es) % 16 != 0) return GDN_ERR_INVALID_ARG;
    if (!(d->l2_eps >= 0.f) || !(d->norm_eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if ((double)d->B * d->T * d->Hv * d->dv > 4.0e12) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

int check_ws(const gdn_desc *d, const void *ws, size_t bytes) {
    if (!ws || !aligned(ws, 256)) return GDN_ERR_WORKSPACE;
    if (bytes < gdn::make_layout(*d).total) return GDN_ERR_WORKSPACE;
    return GDN_OK;
}

std::atomic<int> g_wait_test_mode{0};

Problem base_problem(const gdn_desc *d, const int32_t *cu, void *ws) {
    Problem p;
    memset(&p, 0, sizeof(p));
    p.d = *d;
    p.wait_immediate = g_wait_test_mode.load();
    p.ntok = (int64_t)d->B * d->T;
    p.cu = cu;
    const Layout L = gdn::make_layout(*d);
    char *w = (char *)ws;
    p.status = (int32_t *)(w + L.status);
    p.chunk_off = (int32_t *)(w + L.chunk_off);
    p.q = w + L.q;
    p.k = w + L.k;
    p.v = w + L.v;
    p.beta = (float *)(w + L.beta);
    p.gamma = w + L.gamma;
    p.o = w + L.o;
    p.tpt = w + L.tpt;
    return p;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

int run_prologue(const Problem &p, cudaStream_t s) {
    if (p.cu != nullptr) {
        int rc = cuda_status(gdn::launch_seqlens_scan(p, s));
        if (rc != GDN_OK) return rc;
    }
    if (gdn::chunk_slots(p) == 0) {
        // nothing to compute; still publish an OK status for later stages
        return cuda_status(cudaMemsetAsync(p.status, 0, sizeof(int32_t), s));
    }
    return cuda_status(gdn::launch_prologue(p, s));
}

int run_chunk(const Problem &p, cudaStream_t s) {
    if (gdn::chunk_tc_supports(p.d)) {
        if (gdn::chunk_tc_segmented(p)) return cuda_status(gdn::launch_chunk_tc_segmented(p, s));
        return cuda_status(gdn::launch_chunk_tc(p, s));
    }
    return cuda_status(gdn::launch_chunk_simt(p, s));
}

int run_epilogue(const Problem &p, cudaStream_t s) {
    if (p.ntok == 0 || p.fuse_epilogue) return GDN_OK;
    return cuda_status(gdn::launch_epilogue(p, s));
}

}  // namespace

extern "C" {

int gdn_desc_init(gdn_desc *d, int B, int T, int packed, int Hk, int Hv, int dk, int dv,
                  int dtype) {
    if (!d) return GDN_ERR_INVALID_ARG;
    memset(d, 0, sizeof(*d));
    d->B = B;
    d->T = T;
    d->N = packed ? packed : B;
    d->Hk = Hk;
    d->Hv = Hv;
    d->dk = dk;
    d->dv = dv;
    d->conv_width = 4;
    d->dtype = dtype;
    d->gate_dtype = dtype;
    d->norm_w_dtype = dtype;
    const int64_t ch_qk = (int64_t)Hk * dk, ch_v = (int64_t)Hv * dv;
    d->q_stride_t = d->k_stride_t = ch_qk;
    d->q_stride_b = d->k_stride_b = ch_qk * T;
    d->v_stride_t = ch_v;
    d->v_stride_b = ch_v * T;
    d->a_stride_t = d->b_stride_t = Hv;
    d->a_stride_b = d->b_stride_b = (int64_t)Hv * T;
    d->gate_stride_t = ch_v;
    d->gate_stride_b = ch_v * T;
    d->l2_eps = 1e-6f;
    d->norm_eps = 1e-5f;
    d->scale = 1.0f;
    return check_desc(d, packed != 0);
}

int gdn_workspace_bytes(const gdn_desc *d, size_t *bytes) {
    if (!d || !bytes) return GDN_ERR_INVALID_ARG;
    *bytes = gdn::make_layout(*d).total;
    return GDN_OK;
}

int gdn_workspace_offsets(const gdn_desc *d, gdn_workspace_layout *out) {
    if (!d || !out) return GDN_ERR_INVALID_ARG;
    const Layout L = gdn::make_layout(*d);
    out->status = L.status;
    out->chunk_off = L.chunk_off;
    out->q = L.q;
    out->k = L.k;
    out->v = L.v;
    out->beta = L.beta;
    out->gamma = L.gamma;
    out->o = L.o;
    out->tpt = L.tpt;
    out->total = L.total;
    return GDN_OK;
}

int gdn_prologue(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                 const void *a, const void *b, const void *conv_w, const float *A_log,
                 const float *dt_bias, const int32_t *cu_seqlens, void *workspace,
                 size_t workspace_bytes, gdn_stream_t stream) {
    int rc = check_desc(d, cu_seqlens != nullptr);
    if (rc != GDN_OK) return rc;
    const bool tok = (int64_t)d->B * d->T > 0;   // token tensors may be empty (null)
    if ((tok && (!q_raw || !k_raw || !v_raw || !a || !b)) || !conv_w || !A_log || !dt_bias)
        return GDN_ERR_INVALID_ARG;
    if (!aligned(q_raw, 16) || !aligned(k_raw, 16) || !aligned(v_raw, 16) || !aligned(conv_w, 16))
        return GDN_ERR_INVALID_ARG;
    if ((rc = check_ws(d, workspace, workspace_bytes)) != GDN_OK) return rc;
    Problem p = base_problem(d, cu_seqlens, workspace);
    p.q_raw = q_raw;
    p.k_raw = k_raw;
    p.v_raw = v_raw;
    p.a = a;
    p.b = b;
    p.conv_w = conv_w;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    return run_prologue(p, (cudaStream_t)stream);
}

int gdn_chunk_rule(const gdn_desc *d, const int32_t *cu_seqlens, const float *initial_state,
                   float *final_state, void *workspace, size_t workspace_bytes,
                   gdn_stream_t stream) {
    int rc = check_desc(d, cu_seqlens != nullptr);
    if (rc != GDN_OK) return rc;
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return GDN_ERR_INVALID_ARG;
    if ((rc = check_ws(d, workspace, workspace_bytes)) != GDN_OK) return rc;
    Problem p = base_problem(d, cu_seqlens, workspace);
    p.h0 = initial_state;
    p.hT = final_state;
    return run_chunk(p, (cudaStream_t)stream);
}

int gdn_epilogue(const gdn_desc *d, const void *gate, const void *norm_w, void *out,
                 void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    // the epilogue works per token, so packing does not change it (B == 1 when packed)
    int rc = check_desc(d, d && d->N != d->B);
    if (rc != GDN_OK) return rc;
    const bool tok = (int64_t)d->B * d->T > 0;   // token tensors may be empty (null)
    if ((tok && (!gate || !out)) || !norm_w) return GDN_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(norm_w, 4)) return GDN_ERR_INVALID_ARG;
    if ((rc = check_ws(d, workspace, workspace_bytes)) != GDN_OK) return rc;
    Problem p = base_problem(d, nullptr, workspace);
    p.gate = gate;
    p.norm_w = norm_w;
    p.out = out;
    return run_epilogue(p, (cudaStream_t)stream);
}

}  // extern "C"

namespace {
int forward_impl(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                 const void *a, const void *b, const void *gate, const void *conv_w,
                 const float *A_log, const float *dt_bias, const void *norm_w,
                 const int32_t *cu_seqlens, const float *initial_state, void *out,
                 float *final_state, void *workspace, size_t workspace_bytes,
                 gdn_stream_t stream, bool single_stream, const void *conv_prefix = nullptr) {
    int rc = check_desc(d, cu_seqlens != nullptr);
    if (rc != GDN_OK) return rc;
    const bool tok = (int64_t)d->B * d->T > 0;   // token tensors may be empty (null)
    if ((tok && (!q_raw || !k_raw || !v_raw || !a || !b || !gate || !out)) || !conv_w || !A_log ||
        !dt_bias || !norm_w)
        return GDN_ERR_INVALID_ARG;
    if (!aligned(q_raw, 16) || !aligned(k_raw, 16) || !aligned(v_raw, 16) ||
        !aligned(conv_w, 16) || !aligned(out, 16) || !aligned(norm_w, 4))
        return GDN_ERR_INVALID_ARG;
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)) ||
        (conv_prefix && !aligned(conv_prefix, 16)))
        return GDN_ERR_INVALID_ARG;
    if ((rc = check_ws(d, workspace, workspace_bytes)) != GDN_OK) return rc;
    Problem p = base_problem(d, cu_seqlens, workspace);
    p.q_raw = q_raw;
    p.k_raw = k_raw;
    p.v_raw = v_raw;
    p.a = a;
    p.b = b;
    p.gate = gate;
    p.conv_w = conv_w;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.norm_w = norm_w;
    p.h0 = initial_state;
    p.hT = final_state;
    p.out = out;
    p.single_stream = single_stream;
    p.conv_prefix = conv_prefix;
    // prologue -> prep -> chain -> epilogue back to back on one stream (the
    // plain tensor-core chunk stage): each later kernel is a programmatic
    // dependent of the one before it
    p.pdl = !single_stream && p.ntok > 0 && gdn::chunk_tc_supports(*d) && !gdn::chunk_tc_segmented(p);
    p.fuse_epilogue = gdn::chain_tm_fuses_epilogue(p);
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = run_prologue(p, s)) != GDN_OK) return rc;
    if ((rc = run_chunk(p, s)) != GDN_OK) return rc;
    return run_epilogue(p, s);
}
}  // namespace

namespace gdn {
int forward_single_stream(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                          const void *a, const void *b, const void *gate, const void *conv_w,
                          const float *A_log, const float *dt_bias, const void *norm_w,
                          const int32_t *cu_seqlens, const float *initial_state, void *out,
                          float *final_state, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return forward_impl(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, cu_seqlens,
                        initial_state, out, final_state, workspace, workspace_bytes, (gdn_stream_t)stream, true);
}
}  // namespace gdn

extern "C" {

int gdn_forward(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                const void *a, const void *b, const void *gate, const void *conv_w,
                const float *A_log, const float *dt_bias, const void *norm_w,
                const int32_t *cu_seqlens, const float *initial_state, void *out,
                float *final_state, void *workspace, size_t workspace_bytes,
                gdn_stream_t stream) {
    return forward_impl(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, cu_seqlens,
                        initial_state, out, final_state, workspace, workspace_bytes, stream, false);
}

int gdn_forward_with_prefix(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                            const void *a, const void *b, const void *gate, const void *conv_w,
                            const float *A_log, const float *dt_bias, const void *norm_w,
                            const int32_t *cu_seqlens, const void *conv_prefix, const float *initial_state,
                            void *out, float *final_state, void *workspace, size_t workspace_bytes,
                            gdn_stream_t stream) {
    return forward_impl(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, cu_seqlens,
                        initial_state, out, final_state, workspace, workspace_bytes, stream, false, conv_prefix);
}

int gdn_span_scan(int spans, int Hv, int dk, int dv, const float *A, const float *B, const float *h0,
                  float *H_in, gdn_stream_t stream) {
    if (spans < 0 || Hv < 1 || !is_pow2_in(dk, 16, 512) || !is_pow2_in(dv, 16, 512)) return GDN_ERR_INVALID_ARG;
    if (spans == 0) return GDN_OK;
    if (!A || !B || !H_in) return GDN_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(H_in, 16) || (h0 && !aligned(h0, 16)))
        return GDN_ERR_INVALID_ARG;
    return cuda_status(gdn::launch_span_scan(spans, Hv, dk, dv, A, B, h0, H_in, (cudaStream_t)stream));
}

int gdn_decode_workspace_bytes(const gdn_desc *d, size_t *bytes) {
    if (!bytes) return GDN_ERR_INVALID_ARG;
    int rc = check_desc(d, false);
    if (rc != GDN_OK) return rc;
    if (d->T != 1) return GDN_ERR_INVALID_ARG;
    *bytes = gdn::make_decode_layout(*d).total;
    return GDN_OK;
}

int gdn_decode_step(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                    const void *a, const void *b, const void *gate, const void *conv_w,
                    const float *A_log, const float *dt_bias, const void *norm_w, void *conv_state,
                    float *state, void *out, void *workspace, size_t workspace_bytes,
                    gdn_stream_t stream) {
    int rc = check_desc(d, false);
    if (rc != GDN_OK) return rc;
    if (d->T != 1) return GDN_ERR_INVALID_ARG;
    if (!q_raw || !k_raw || !v_raw || !a || !b || !gate || !conv_w || !A_log || !dt_bias || !norm_w ||
        !conv_state || !state || !out)
        return GDN_ERR_INVALID_ARG;
    const size_t es = gdn::act_size(d->dtype);
    if (!aligned(q_raw, es) || !aligned(k_raw, es) || !aligned(v_raw, es) || !aligned(conv_w, es) ||
        !aligned(conv_state, es) || !aligned(state, 16) || !aligned(out, 16) || !aligned(norm_w, 4))
        return GDN_ERR_INVALID_ARG;
    const gdn::DecodeLayout L = gdn::make_decode_layout(*d);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return GDN_ERR_WORKSPACE;
    char *w = (char *)workspace;
    gdn::DecodeProblem p;
    memset(&p, 0, sizeof(p));
    p.d = *d;
    p.q_raw = q_raw;
    p.k_raw = k_raw;
    p.v_raw = v_raw;
    p.a = a;
    p.b = b;
    p.conv_w = conv_w;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.conv_state = conv_state;
    p.state = state;
    p.status = (int32_t *)(w + L.status);
    p.q = (float *)(w + L.q);
    p.k = (float *)(w + L.k);
    p.v = (float *)(w + L.v);
    p.beta = (float *)(w + L.beta);
    p.g = (float *)(w + L.g);
    p.o = w + L.o;
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = cuda_status(gdn::launch_decode(p, s))) != GDN_OK) return rc;
    // the forward's gated RMSNorm over the B new tokens
    Problem e;
    memset(&e, 0, sizeof(e));
    e.d = *d;
    e.ntok = d->B;
    e.gate = gate;
    e.norm_w = norm_w;
    e.out = out;
    e.status = p.status;
    e.o = p.o;
    return run_epilogue(e, s);
}

int gdn_device_status(const void *workspace, int *status, gdn_stream_t stream) {
    if (!workspace || !status) return GDN_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    *status = v;
    return GDN_OK;
}

int gdn_set_wait_test_mode(int immediate) {
    if (immediate != 0 && immediate != 1) return GDN_ERR_INVALID_ARG;
    g_wait_test_mode.store(immediate);
    return GDN_OK;
}

const char *gdn_status_string(int status) {
    switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID_ARG: return "invalid argument (null pointer, size, stride or alignment)";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration (dims, conv width, head ratio or dtype)";
    case GDN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case GDN_ERR_CUDA: return "CUDA launch or query failed";
    case GDN_ERR_DEVICE_SEQLENS: return "cu_seqlens malformed (device check)";
    case GDN_ERR_DEVICE_RANGE: return "non-finite intermediate (device check)";
    case GDN_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    default: return "unknown status";
    }
}

int gdn_chunk_kernel_kind(const gdn_desc *d) {
    if (!d) return GDN_ERR_INVALID_ARG;
    return gdn::chunk_tc_supports(*d) ? 1 : 0;
}

}  // extern "C"

extern "C" {

int gdn_backward_workspace_bytes(const gdn_desc *d, size_t *bytes) {
    if (!d || !bytes) return GDN_ERR_INVALID_ARG;
    *bytes = gdn::make_bwd_layout(*d).total;
    return GDN_OK;
}

int gdn_backward(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw, const void *a,
                 const void *b, const void *gate, const void *conv_w, const float *A_log, const float *dt_bias,
                 const void *norm_w, const int32_t *cu_seqlens, const float *initial_state,
                 const void *grad_out, const float *grad_final, void *dq_raw, void *dk_raw, void *dv_raw,
                 void *da, void *db, void *dgate, float *dconv_w, float *dA_log, float *ddt_bias,
                 float *dnorm_w, float *dinitial_state, void *workspace, size_t workspace_bytes,
                 gdn_stream_t stream) {
    int rc = check_desc(d, cu_seqlens != nullptr);
    if (rc != GDN_OK) return rc;
    const bool tok = (int64_t)d->B * d->T > 0;   // token tensors may be empty (null)
    if ((tok && (!q_raw || !k_raw || !v_raw || !a || !b || !gate || !grad_out || !dq_raw || !dk_raw ||
                 !dv_raw || !da || !db || !dgate)) ||
        !conv_w || !A_log || !dt_bias || !norm_w || !dconv_w || !dA_log || !ddt_bias || !dnorm_w)
        return GDN_ERR_INVALID_ARG;
    if (!aligned(q_raw, 16) || !aligned(k_raw, 16) || !aligned(v_raw, 16) || !aligned(conv_w, 16) ||
        !aligned(norm_w, 4) || !aligned(dq_raw, 16) || !aligned(dk_raw, 16) || !aligned(dv_raw, 16))
        return GDN_ERR_INVALID_ARG;
    if ((initial_state && !aligned(initial_state, 16)) || (grad_final && !aligned(grad_final, 16)) ||
        (dinitial_state && !aligned(dinitial_state, 16)))
        return GDN_ERR_INVALID_ARG;
    const gdn::BwdLayout L = gdn::make_bwd_layout(*d);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return GDN_ERR_WORKSPACE;
    Problem p = base_problem(d, cu_seqlens, workspace);
    p.q_raw = q_raw;
    p.k_raw = k_raw;
    p.v_raw = v_raw;
    p.a = a;
    p.b = b;
    p.gate = gate;
    p.conv_w = conv_w;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.norm_w = norm_w;
    p.h0 = initial_state;
    p.hT = nullptr;
    p.single_stream = true;
    char *w = (char *)workspace;
    cudaStream_t s = (cudaStream_t)stream;
    // the forward's prologue (q, k, v, beta and the in-chunk decay in the workspace)
    if ((rc = run_prologue(p, s)) != GDN_OK) return rc;
    gdn::BwdProblem bp;
    memset(&bp, 0, sizeof(bp));
    bp.f = p;
    bp.grad_out = grad_out;
    bp.grad_final = grad_final;
    bp.dq_raw = dq_raw;
    bp.dk_raw = dk_raw;
    bp.dv_raw = dv_raw;
    bp.da = da;
    bp.db = db;
    bp.dgate = dgate;
    bp.dconv_w = dconv_w;
    bp.dA_log = dA_log;
    bp.ddt_bias = ddt_bias;
    bp.dnorm_w = dnorm_w;
    bp.dinit = dinitial_state;
    bp.h0 = (float *)(w + L.h0);
    bp.mats = (float *)(w + L.mats);
    bp.vn = (float *)(w + L.vn);
    bp.dh1 = (float *)(w + L.dh1);
    bp.uq = (float *)(w + L.uq);
    bp.wv = (float *)(w + L.wv);
    bp.dO = (float *)(w + L.dO);
    bp.dR = (float *)(w + L.dR);
    bp.dq = (float *)(w + L.dq);
    bp.dk = (float *)(w + L.dk);
    bp.dbeta = (float *)(w + L.dbeta);
    bp.dgam = (float *)(w + L.dgam);
    bp.dz = (float *)(w + L.dz);
    bp.pa = (float *)(w + L.pa);
    bp.pnorm = (float *)(w + L.pnorm);
    bp.pconv = (float *)(w + L.pconv);
    bp.xbuf = (float *)(w + L.xbuf);
    bp.hdbuf = (float *)(w + L.hdbuf);
    return cuda_status(gdn::launch_backward(bp, s));
}

}  // extern "C"
