/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) layer core forward on GB300 (sm_103a).
 *
 * The core forward computes, per token t and v head h (GQA: v head h reads q/k
 * head h / (Hv/Hk)):
 *
 *   1. a width-4 causal depthwise convolution over the channel-concatenated
 *      [q_raw | k_raw | v_raw] projections followed by SiLU
 *      ("fused q/k/v short conv", flash-linear-attention PR #972, sections
 *      "Summary" and "Why"; "GDN Elementwise Fusion", option table, pre-GDR);
 *   2. per-head L2 normalisation of q and k, x * rsqrt(sum x^2 + 1e-6)
 *      ("perf(gated_delta_net): fold q/k L2-norm into the gated_delta_rule
 *      kernel", Megatron-LM PR #5396, section "Why");
 *   3. beta = sigmoid(b) and the decay g = -exp(A_log) * softplus(a + dt_bias)
 *      ("GDN Elementwise Fusion", option table: beta and decay preparation);
 *   4. the gated delta rule S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T)
 *      + beta_t v_t k_t^T, o_t = scale * S_t q_t, evaluated chunk by chunk
 *      (64 tokens, WY/UT form) with an fp32 state;
 *   5. y = RMSNorm(o) * SiLU(gate), the RMSNorm result materialised in the
 *      activation dtype before the fp32 gating multiply ("GDN Elementwise
 *      Fusion", post-GDR requirements and "Execution and numerical behavior").
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or synchronises (except gdn_device_status, which
 *    says so). Every call is asynchronous on `stream` (0 = legacy default).
 *  - Return value: GDN_OK (0) or a negative gdn_status. Argument checks read
 *    metadata only (no device synchronisation). On an error nothing is
 *    launched. There is no fallback path for unsupported inputs.
 *  - Element strides are in elements of the tensor's own dtype; the channel
 *    (last) dimension is always contiguous.
 *  - Device-side argument faults (a malformed cu_seqlens) cannot be seen by
 *    the host without a sync: the kernels then write a status word in the
 *    workspace and skip their work; read it with gdn_device_status().
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gdn_stream_t; /* == cudaStream_t */

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, bad stride or alignment */
    GDN_ERR_UNSUPPORTED = -2,  /* dk/dv not a power of two in [16, 512], conv_width != 4,
                                  Hv % Hk != 0, unsupported dtype combination */
    GDN_ERR_WORKSPACE = -3,    /* workspace missing, misaligned or smaller than
                                  gdn_workspace_bytes() */
    GDN_ERR_CUDA = -4,         /* a CUDA launch or query failed */
    GDN_ERR_DEVICE_SEQLENS = -5, /* (device status) cu_seqlens not 0-based, not
                                    non-decreasing or not ending at T */
    GDN_ERR_DEVICE_RANGE = -6,  /* (device status) a non-finite gated-delta-rule output
                                   reached step 5 (the separate output kernel, or the
                                   output step inside the chunk kernel): a non-finite
                                   input, or a value beyond the fp16 range of the
                                   intermediates */
    GDN_ERR_DEVICE_TIMEOUT = -7 /* (device status) a tensor-core kernel gave up waiting
                                   (about 1 s) for a copy or an MMA; results are invalid */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 } gdn_dtype;

/* Problem descriptor. Fill it with gdn_desc_init() and then override
 * strides/dtypes of views as needed. */
typedef struct {
    int32_t B, T;        /* batch rows, tokens per row; with cu_seqlens: B = 1 and
                            T = total packed tokens */
    int32_t N;           /* sequences: B without cu_seqlens, else cu_seqlens has N+1 entries */
    int32_t Hk, Hv;      /* q/k heads, v heads (Hv % Hk == 0) */
    int32_t dk, dv;      /* head dims: powers of two in [16, 512] */
    int32_t conv_width;  /* short-conv taps; must be 4 */
    int32_t dtype;       /* gdn_dtype of q_raw, k_raw, v_raw, a, b, conv_w and out */
    int32_t gate_dtype;  /* dtype, or GDN_F32 */
    int32_t norm_w_dtype;/* dtype, or GDN_F32 */
    int32_t reserved0;
    /* (batch, token) element strides; channel stride is 1 */
    int64_t q_stride_b, q_stride_t;
    int64_t k_stride_b, k_stride_t;
    int64_t v_stride_b, v_stride_t;
    int64_t a_stride_b, a_stride_t;
    int64_t b_stride_b, b_stride_t;
    int64_t gate_stride_b, gate_stride_t;
    float l2_eps;        /* q/k L2-norm eps, 1e-6 */
    float norm_eps;      /* output RMSNorm eps, 1e-5 */
    float scale;         /* q scale in o_t = scale * S_t q_t, 1 */
    int32_t reserved1;
} gdn_desc;

/* Fill *d for contiguous tensors: q_raw/k_raw [B,T,Hk*dk], v_raw [B,T,Hv*dv],
 * a/b [B,T,Hv], gate [B,T,Hv*dv], gate/norm_w in the act dtype,
 * l2_eps 1e-6, norm_eps 1e-5, scale 1, conv_width 4. N = B when packed == 0;
 * packed != 0 requires B == 1 and sets N = packed. Returns the validation
 * status of the filled descriptor. */
int gdn_desc_init(gdn_desc *d, int B, int T, int packed, int Hk, int Hv, int dk, int dv,
                  int dtype);

/* Bytes of scratch the forward needs for *d (intermediate q/k/v, beta, the
 * in-chunk cumulative decay, o, a status word and the chunk table). */
int gdn_workspace_bytes(const gdn_desc *d, size_t *bytes);

/* Offsets (bytes from the workspace base) of the intermediate tensors, for
 * inspection by tests and tools:
 *   q, k [Hk][Ntok][dk] after conv, SiLU and L2 norm: fp32 for fp32
 *   activations, else two fp16 planes (hi = fp16(x) at the offset, then
 *   lo = fp16(x - hi) right after the Hk*Ntok*dk hi elements); v [Hv][Ntok][dv]
 *   after conv and SiLU and o [Ntok][Hv][dv] (gated delta rule output): fp16 for
 *   bf16/fp16 activations, fp32 for fp32 activations; beta [Hv][Ntok] fp32;
 *   gamma [Hv][Ntok] = in-chunk inclusive cumulative sum of g, fp64 for fp32
 *   activations and fp32 otherwise; status: int32 device status word;
 *   chunk_off: int32 [N+1]; tpt: the tensor-core kernels' region (empty where
 *   they do not run): per (v head, chunk slot) 32 KB of prep tiles (the 128x64
 *   fp16 tile [T; P T], then X), and for one sequence (N = 1) after them the fp32
 *   state handed between the segments of its chain, [Hv][dk][dv]. */
typedef struct {
    size_t status, chunk_off, q, k, v, beta, gamma, o, tpt, total;
} gdn_workspace_layout;
int gdn_workspace_offsets(const gdn_desc *d, gdn_workspace_layout *layout);

/*
 * The whole core forward (steps 1-5 above) on `stream`.
 *   q_raw, k_raw   act dtype, [B,T,Hk*dk] at (q|k)_stride_(b|t); 16-byte aligned
 *                  base and strides
 *   v_raw          act dtype, [B,T,Hv*dv] at v_stride_(b|t); 16-byte aligned
 *   a, b           act dtype, [B,T,Hv] at (a|b)_stride_(b|t); any alignment
 *   gate           gate_dtype, [B,T,Hv*dv] at gate_stride_(b|t): may be a strided,
 *                  unaligned view into a wider projection buffer
 *   conv_w         act dtype, [2*Hk*dk + Hv*dv][4] contiguous, q|k|v channel
 *                  order, tap 3 multiplies the current token; 16-byte aligned
 *   A_log, dt_bias fp32 [Hv]
 *   norm_w         norm_w_dtype [dv] contiguous
 *   cu_seqlens     NULL, or int32 [N+1] packed-sequence offsets (then B == 1);
 *                  the conv halo and the state restart at every offset
 *   initial_state  NULL (zeros) or fp32 [N][Hv][dk][dv], the transposed state
 *                  S^T of every (sequence, v head); 16-byte aligned
 *   out            act dtype [B,T,Hv,dv] contiguous; 16-byte aligned
 *                  (token tensors and out may be NULL when B*T == 0)
 *   final_state    NULL (not written) or fp32 [N][Hv][dk][dv]; 16-byte aligned
 *   workspace      device scratch of >= gdn_workspace_bytes(), 256-byte aligned;
 *                  calls that share a workspace must not overlap on the GPU
 * Inputs are only read; initial_state and final_state may alias.
 * Ordering: the call's first kernel starts after everything queued on `stream`
 * before it, and work queued after the call starts after its last kernel. On
 * the tensor-core path without segments the later kernels of the call are
 * programmatic dependents of the kernel before them (their CTAs may become
 * resident early and wait on the device); a long single sequence runs part of
 * the chunk stage on a high-priority stream the library creates once per
 * device, joined back to `stream` by events.
 */
int gdn_forward(const gdn_desc *d,
                const void *q_raw, const void *k_raw, const void *v_raw,
                const void *a, const void *b, const void *gate,
                const void *conv_w, const float *A_log, const float *dt_bias,
                const void *norm_w, const int32_t *cu_seqlens,
                const float *initial_state, void *out, float *final_state,
                void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* The three stages of gdn_forward, callable one by one on the same workspace
 * (gdn_forward gives bit for bit the results of prologue, chunk_rule, epilogue in
 * this order). Where the transposed tensor-core chunk kernel holds a whole v-head
 * row (16-bit activations, dk 64 or 128, dv = 128), the gate and norm_w match the
 * activation dtype (norm_w may be fp32), the gate view has a 16-byte aligned base
 * and row pitch with its batch rows back to back, and the chunk stage is not cut
 * into segments (one long sequence), gdn_forward applies step 5 inside that kernel,
 * with the same arithmetic, and leaves o in the workspace unwritten.
 * gdn_prologue: steps 1-3 plus the in-chunk cumulative decay -> workspace q, k,
 *   v, beta, gamma (and the chunk table / status word when cu_seqlens is set).
 * gdn_chunk_rule: step 4 -> workspace o, final_state.
 * gdn_epilogue: step 5 -> out. */
int gdn_prologue(const gdn_desc *d, const void *q_raw, const void *k_raw,
                 const void *v_raw, const void *a, const void *b, const void *conv_w,
                 const float *A_log, const float *dt_bias, const int32_t *cu_seqlens,
                 void *workspace, size_t workspace_bytes, gdn_stream_t stream);
int gdn_chunk_rule(const gdn_desc *d, const int32_t *cu_seqlens,
                   const float *initial_state, float *final_state,
                   void *workspace, size_t workspace_bytes, gdn_stream_t stream);
int gdn_epilogue(const gdn_desc *d, const void *gate, const void *norm_w, void *out,
                 void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/* Wait for `stream`, then read the device status word of the last forward that
 * used `workspace` into *status (GDN_OK or a GDN_ERR_DEVICE_* code). This call
 * synchronises the stream. */
int gdn_device_status(const void *workspace, int *status, gdn_stream_t stream);

/* Static description of a status code. */
const char *gdn_status_string(int status);

/*
 * Test hook for the tensor-core kernels' bounded waits (GDN_ERR_DEVICE_TIMEOUT).
 * Every wait of those kernels on one of their own mbarriers gives up after about
 * a second; the CTA then records GDN_ERR_DEVICE_TIMEOUT, waits (again bounded) for
 * its own copies and products in flight, frees its tensor memory and returns.
 * With immediate = 1, calls made afterwards in this process launch these kernels
 * so that a main-loop wait which is not already complete gives up at once (a
 * non-blocking test instead of the timed wait), which drives that path on any
 * input without stalling the GPU; the drains keep their ~1 s limit. immediate = 0
 * restores the normal waits. The outputs of a call that timed out are
 * unspecified; the next call in the normal mode is unaffected. Not meant for
 * production use; there is no counterpart on the pages. Returns GDN_OK, or
 * GDN_ERR_INVALID_ARG for another value.
 */
int gdn_set_wait_test_mode(int immediate);

/*
 * gdn_forward without a caller-provided workspace, for callers that cannot
 * allocate device memory (code running inside another framework's memory
 * arena, plugins without an allocator, hosts that forbid allocation while
 * serving). The pages describe no such entry point; it has no counterpart there.
 *
 * The scratch is a fixed device array of GDN_STATIC_WORKSPACE_BYTES inside the
 * library; every GPU that loads the library holds it until the process exits.
 * Arguments and results are those of gdn_forward (same pointers, layouts and
 * status codes, without workspace and workspace_bytes).
 *  - Problems whose gdn_workspace_bytes() exceeds GDN_STATIC_WORKSPACE_BYTES are
 *    rejected with GDN_ERR_WORKSPACE before anything is launched.
 *  - The device is the current CUDA device; `stream` must belong to it. The
 *    first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 *    routine).
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents: calls that overlap on the GPU (different streams, or host
 *    threads racing on one device) race on it and must be serialised by the
 *    caller.
 *  - Device-side status (GDN_ERR_DEVICE_SEQLENS, GDN_ERR_DEVICE_RANGE,
 *    GDN_ERR_DEVICE_TIMEOUT) goes to the status word at the start of the
 *    array, as gdn_forward's goes to its workspace; read it with
 *    gdn_static_ws_device_status below.
 *  - The address is looked up again when the device's context changes (e.g.
 *    after cudaDeviceReset), so a reset between calls is safe.
 */
#define GDN_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)
int gdn_forward_static_ws(const gdn_desc *d,
                          const void *q_raw, const void *k_raw, const void *v_raw,
                          const void *a, const void *b, const void *gate,
                          const void *conv_w, const float *A_log, const float *dt_bias,
                          const void *norm_w, const int32_t *cu_seqlens,
                          const float *initial_state, void *out, float *final_state,
                          gdn_stream_t stream);

/* Wait for `stream`, then read the device status word of the last
 * gdn_forward_static_ws call on the current device into *status (GDN_OK or a
 * GDN_ERR_DEVICE_* code), like gdn_device_status for a caller's workspace. No
 * counterpart on the pages either. Synchronises the stream; allocates nothing.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG (null status) or GDN_ERR_CUDA. */
int gdn_static_ws_device_status(int *status, gdn_stream_t stream);

/* Which gated-delta-rule kernel serves *d: 0 = fp32 CUDA-core kernel,
 * 1 = tcgen05 tensor-core kernel (bf16/fp16). */
int gdn_chunk_kernel_kind(const gdn_desc *d);

/*
 * Decode: one new token for each of d->B sequences. The result is what
 * gdn_forward gives for one more token of each sequence (same definitions,
 * same readings): the width-4 causal conv takes the sequence's last three raw
 * inputs from a conv cache, then SiLU, the q/k L2 norm, beta and the decay, one
 * step of S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with
 * o_t = scale * S_t q_t from the carried state, and the gated RMSNorm. The pages
 * define the forward; a decode cache appears there only as the conv input that a
 * fused prefill conv has to leave out ("fused q/k/v short conv",
 * flash-linear-attention PR #972, "Risk / scope").
 *
 * d           d->T == 1, not packed (N == B), everything else as for gdn_forward;
 *             the token tensors are [B, 1, *] views (only the batch strides and
 *             the contiguous channels matter).
 * q_raw ... norm_w   as for gdn_forward, one token per sequence.
 * conv_state  act dtype [B][ch][3] contiguous, ch = 2*Hk*dk + Hv*dv in q|k|v
 *             order: per channel the raw inputs of the sequence's last three
 *             tokens, oldest first (zeros where the sequence has fewer). Read,
 *             then overwritten with the window advanced by this token. After a
 *             gdn_forward prefill it holds that call's last three raw tokens.
 * state       fp32 [B][Hv][dk][dv] (S^T per sequence and v head, the layout of
 *             gdn_forward's initial_state / final_state), 16-byte aligned; read
 *             and overwritten in place.
 * out         act dtype [B, 1, Hv, dv] contiguous, 16-byte aligned.
 * workspace   gdn_decode_workspace_bytes(d) bytes, 256-byte aligned; its first
 *             word is the device status (gdn_device_status).
 * Returns GDN_OK or a negative status as gdn_forward (GDN_ERR_INVALID_ARG for
 * d->T != 1 or a packed descriptor). conv_state, state, out and workspace must
 * not overlap each other or the inputs.
 */
int gdn_decode_workspace_bytes(const gdn_desc *d, size_t *bytes);
int gdn_decode_step(const gdn_desc *d,
                    const void *q_raw, const void *k_raw, const void *v_raw,
                    const void *a, const void *b, const void *gate,
                    const void *conv_w, const float *A_log, const float *dt_bias,
                    const void *norm_w, void *conv_state, float *state, void *out,
                    void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_forward for sequences that continue an earlier part (chunked prefill, or
 * one span of a sequence split across ranks): the width-4 causal conv reads the
 * raw inputs of the three tokens before each sequence from conv_prefix instead
 * of zeros ("fused q/k/v short conv", flash-linear-attention PR #972, "Summary":
 * a per-channel causal short conv over the projections; the earlier tokens are
 * the conv's left context). Everything else is gdn_forward's, with the state
 * carried in through initial_state.
 *
 * conv_prefix  act dtype [N][3][2*Hk*dk + Hv*dv] contiguous, 16-byte aligned:
 *              per sequence the raw q|k|v inputs (conv_w's channel order) of
 *              its three preceding tokens, oldest first; NULL = zeros (then
 *              this is gdn_forward).
 * Returns as gdn_forward (GDN_ERR_INVALID_ARG also for a misaligned prefix).
 */
int gdn_forward_with_prefix(const gdn_desc *d,
                            const void *q_raw, const void *k_raw, const void *v_raw,
                            const void *a, const void *b, const void *gate,
                            const void *conv_w, const float *A_log, const float *dt_bias,
                            const void *norm_w, const int32_t *cu_seqlens,
                            const void *conv_prefix, const float *initial_state,
                            void *out, float *final_state,
                            void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * The exchange step of the sequence-sharded core. Over a span of one sequence
 * the chunked gated delta rule (S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) +
 * beta_t v_t k_t^T, state H = S^T) is affine in the span's initial state:
 * H_end = A H_start + B, where B is the span's final state from zeros and A
 * (dk x dk) the span's final state with v = 0, dv = dk and the identity as
 * initial state (both by gdn_forward_with_prefix). Given every span's maps in
 * sequence order, this writes each span's initial state:
 *     H_in[0] = h0,  H_in[s] = A[s-1] H_in[s-1] + B[s-1].
 *
 * spans      number of spans (0: nothing to do).
 * A          fp32 [spans][Hv][dk][dk]; B fp32 [spans][Hv][dk][dv] (the last
 *            span's maps are not read); h0 fp32 [Hv][dk][dv] or NULL (zeros);
 * H_in       fp32 [spans][Hv][dk][dv], written.
 * All device pointers, 16-byte aligned. Returns GDN_OK, GDN_ERR_INVALID_ARG
 * (bad size, null or misaligned pointer) or GDN_ERR_CUDA. Asynchronous on
 * stream; H_in must not overlap A, B or h0.
 */
int gdn_span_scan(int spans, int Hv, int dk, int dv, const float *A, const float *B,
                  const float *h0, float *H_in, gdn_stream_t stream);

/*
 * Backward of the core: the gradients of
 *     L = sum(grad_out * out) + sum(grad_final * final_state)
 * with respect to every input of gdn_forward, first order. The pages define
 * the forward; training needs its first-order gradients ("GDN Elementwise
 * Fusion", Megatron Core developer guide, "Execution and numerical behavior":
 * the fused post-GDR kernels support first-order autograd; "fused q/k/v short
 * conv", flash-linear-attention PR #972, "Test plan": input and parameter
 * gradients of the fused path checked against the unfused one, and the
 * benchmark table timing forward + backward). Reading: the rounding of the
 * RMSNorm result to the activation dtype is taken as the identity (the
 * straight-through derivative of the rounded forward).
 *
 * The call recomputes the forward, storing each chunk's start state, and then
 * runs the reverse pass. What runs depends on the activation dtype:
 *  - fp32 activations: everything on CUDA cores in fp32 (the prologue, a
 *    state recompute, the reverse pass);
 *  - 2-byte activations with dk in {64, 128, 256} and dv a multiple of 64
 *    (gdn_chunk_kernel_kind() == 1): the forward's tcgen05 chunk stage (prep
 *    and chain) recomputes the states, the new values and the outputs in fp32;
 *    the dO' terms and the per-chunk dv contractions are tcgen05 products
 *    (split bf16 or fp16 operands, fp32 accumulators);
 *  - other 2-byte shapes: an fp32 CUDA-core state recompute; where dk and dv
 *    are multiples of 64 (dv <= 512) the outputs and the dO' terms are still
 *    tcgen05 products;
 *  - in every case the serial reverse chain, the per-chunk gradients' other
 *    terms and the elementwise backward run on CUDA cores in fp32.
 * Every sum has a fixed order: results are run-to-run identical.
 *
 * d, q_raw ... initial_state   exactly as for gdn_forward (same descriptor,
 *             strides, packing and alignment rules).
 * grad_out    act dtype [B*T][Hv][dv] contiguous (the gradient of out).
 * grad_final  fp32 [N][Hv][dk][dv] (S^T layout of final_state), or NULL = zeros.
 * dq_raw, dk_raw  act dtype, dense [B*T][Hk*dk]; dv_raw act dtype [B*T][Hv*dv];
 *             these three 16-byte aligned;
 * da, db      act dtype [B*T][Hv]; dgate gate dtype [B*T][Hv*dv] (all dense,
 *             whatever the strides of the inputs);
 * dconv_w     fp32 [2*Hk*dk+Hv*dv][4]; dA_log, ddt_bias fp32 [Hv];
 * dnorm_w     fp32 [dv]; dinitial_state fp32 [N][Hv][dk][dv] or NULL (skip).
 *             All outputs are written in full (not accumulated into).
 * workspace   gdn_backward_workspace_bytes(d) bytes, 256-byte aligned; it
 *             begins with gdn_forward's layout (status word first, so
 *             gdn_device_status reads it), followed by the backward's fp32
 *             regions: per token and v head about 2*dk*dv/64 + 3*dv + 2*dk + 196
 *             floats, plus 2*Hk*dk + Hv*dv floats per token (about 180 KB per
 *             token at 6 heads, dk 256, dv 512).
 * Returns GDN_OK, GDN_ERR_INVALID_ARG (null or misaligned pointer),
 * GDN_ERR_UNSUPPORTED (as gdn_forward), GDN_ERR_WORKSPACE or GDN_ERR_CUDA; a
 * malformed cu_seqlens sets GDN_ERR_DEVICE_SEQLENS in the workspace and the
 * kernels skip their work. Outputs must not overlap the inputs or workspace.
 */
int gdn_backward_workspace_bytes(const gdn_desc *d, size_t *bytes);
int gdn_backward(const gdn_desc *d,
                 const void *q_raw, const void *k_raw, const void *v_raw,
                 const void *a, const void *b, const void *gate,
                 const void *conv_w, const float *A_log, const float *dt_bias,
                 const void *norm_w, const int32_t *cu_seqlens,
                 const float *initial_state, const void *grad_out,
                 const float *grad_final, void *dq_raw, void *dk_raw, void *dv_raw,
                 void *da, void *db, void *dgate, float *dconv_w, float *dA_log,
                 float *ddt_bias, float *dnorm_w, float *dinitial_state,
                 void *workspace, size_t workspace_bytes, gdn_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H */
