// gdn_internal.h -- internal launch interfaces between the C ABI (gdn_api.cu)
// and the kernels. Not part of the public boundary (include/gdn.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Workspace regions (byte offsets); every region starts on a 256-byte boundary.
struct Layout {
    size_t status, chunk_off, q, k, v, beta, gamma, o, tpt, total;
};

// Chunk slots: an upper bound of the number of 64-token chunks over all
// sequences, ceil(ntok / 64) + N (each sequence adds at most one partial chunk).
inline int64_t chunk_slot_bound(const gdn_desc &d) {
    return ((int64_t)d.B * d.T + 63) / 64 + d.N;
}

// Bytes of the tensor-core kernels' [T; P T] tiles (0 where they do not run).
size_t chunk_tc_workspace(const gdn_desc &d);

inline size_t act_size(int dtype) { return dtype == GDN_F32 ? 4 : 2; }

// Intermediates. v (after the prologue) and o (after the chunk rule) are stored
// in fp16 for bf16 and fp16 activations (3 more mantissa bits than bf16 at the
// same size) and in fp32 for fp32 activations. The normalised q and k carry
// about fp32 precision (the q.k products of nearly orthogonal pairs cancel, and
// the output RMSNorm would amplify their rounding): fp32 for fp32 activations,
// otherwise two fp16 planes hi = fp16(x), lo = fp16(x - hi), so that the tensor
// cores can take both parts directly. The in-chunk cumulative decay is fp64 for
// fp32 activations (differences of large sums stay exact to fp32 precision) and
// fp32 otherwise.
inline size_t gamma_size(int dtype) { return dtype == GDN_F32 ? 8 : 4; }
inline size_t qk_size(int) { return 4; }   // fp32, or fp16 hi + fp16 lo

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t chunk_tc_workspace(const gdn_desc &d);

inline Layout make_layout(const gdn_desc &d) {
    const size_t s = act_size(d.dtype);
    const size_t ntok = (size_t)d.B * (size_t)d.T;
    Layout L;
    size_t off = 0;
    L.status = off;    off = align_up(off + 256, 256);
    L.chunk_off = off; off = align_up(off + 4 * ((size_t)d.N + 1), 256);
    L.q = off;         off = align_up(off + qk_size(d.dtype) * ntok * d.Hk * d.dk, 256);
    L.k = off;         off = align_up(off + qk_size(d.dtype) * ntok * d.Hk * d.dk, 256);
    L.v = off;         off = align_up(off + s * ntok * d.Hv * d.dv, 256);
    L.beta = off;      off = align_up(off + 4 * ntok * d.Hv, 256);
    L.gamma = off;     off = align_up(off + gamma_size(d.dtype) * ntok * d.Hv, 256);
    L.o = off;         off = align_up(off + s * ntok * d.Hv * d.dv, 256);
    L.tpt = off;       off = align_up(off + chunk_tc_workspace(d), 256);
    L.total = off;
    return L;
}

// Device pointers of one forward, resolved from the descriptor and workspace.
struct Problem {
    gdn_desc d;
    int64_t ntok;
    const void *q_raw, *k_raw, *v_raw, *a, *b, *gate, *conv_w, *norm_w;
    const float *A_log, *dt_bias;
    const int32_t *cu;            // null when not packed
    const float *h0;              // null: zeros
    float *hT;                    // null: not written
    void *out;
    int32_t *status, *chunk_off;
    void *q, *k, *v, *o;
    float *beta;
    void *gamma;                  // float, or double for fp32 activations
    void *tpt;                    // [T; P T] tiles of the tensor-core kernels
    bool single_stream;           // no side stream (the no-allocation entry point)
    // launch the chunk kernels and the epilogue as programmatic dependents of the
    // kernel before them on the stream (their CTAs become resident while that
    // kernel drains and wait for its completion on the device)
    bool pdl;
    // null in the forward. The backward's recompute through the tensor-core chunk
    // stage: the chain also stores the fp32 state at every chunk's start
    // ([slot][Hv][dk][dv]), the new values Vn and the outputs O in fp32
    // ([Hv][ntok][dv] each), and not the 16-bit o.
    float *rec_h0, *rec_vn, *rec_o;
    // null, or act dtype [N][3][2*Hk*dk + Hv*dv]: the raw q|k|v inputs of the three
    // tokens before each sequence (oldest first), read by the conv instead of zeros
    const void *conv_prefix;
    // 0: the tensor-core kernels' main-loop waits give up after about a second;
    // 1 (tests of the timeout path, gdn_set_wait_test_mode): a main-loop wait that is
    // not already complete gives up at once. Drains always use the ~1 s limit.
    int wait_immediate;
    // gdn_forward on the transposed chain with dv = 128: the chain applies the output
    // step (gated RMSNorm) itself and writes out; o in the workspace is not written
    bool fuse_epilogue;
};

// Upper bound on chunk slots: ceil(ntok/64) + N (each sequence adds at most one
// partial chunk), or the exact count without packing.
inline int64_t chunk_slots(const Problem &p) {
    if (p.cu == nullptr) return (int64_t)p.d.N * ((p.d.T + 63) / 64);
    return (p.ntok + 63) / 64 + p.d.N;
}

cudaError_t launch_seqlens_scan(const Problem &p, cudaStream_t s);
cudaError_t launch_prologue(const Problem &p, cudaStream_t s);
cudaError_t launch_chunk_simt(const Problem &p, cudaStream_t s);
cudaError_t launch_chunk_tc(const Problem &p, cudaStream_t s);
// a long single sequence: prep and chain in segments on two streams
bool chunk_tc_segmented(const Problem &p);
// the chunk stage with the recompute stores (p.rec_* set), one stream, no segments
cudaError_t launch_chunk_tc_rec(const Problem &p, cudaStream_t s);
cudaError_t launch_chunk_tc_segmented(const Problem &p, cudaStream_t s);
// gdn_forward on one stream only (used by gdn_forward_static_ws)
int forward_single_stream(const gdn_desc *d, const void *q_raw, const void *k_raw, const void *v_raw,
                          const void *a, const void *b, const void *gate, const void *conv_w,
                          const float *A_log, const float *dt_bias, const void *norm_w,
                          const int32_t *cu_seqlens, const float *initial_state, void *out,
                          float *final_state, void *workspace, size_t workspace_bytes, cudaStream_t stream);
bool chunk_tc_supports(const gdn_desc &d);
// the transposed chain (dk <= 128, 128-row dv tiles, operands in tensor memory;
// gdn_chain_tm.cu): chunks [cbase, cbase + cmax) of every sequence, nblocks =
// sequences x Hv x chain_tm_tiles CTAs
bool chain_tm_supports(const gdn_desc &d);
bool chain_tm_fuses_epilogue(const Problem &p);
int chain_tm_tiles(const gdn_desc &d);
cudaError_t launch_chain_tm(const Problem &p, cudaStream_t s, const unsigned char *prep_out, int64_t nslots_alloc,
                            int cbase, int cmax, bool pdl, unsigned nblocks);
cudaError_t launch_epilogue(const Problem &p, cudaStream_t s);
// H_in[s] = A[s-1] H_in[s-1] + B[s-1], H_in[0] = h0 (or zeros), per v head
cudaError_t launch_span_scan(int spans, int Hv, int dk, int dv, const float *A, const float *B, const float *h0,
                             float *H_in, cudaStream_t s);

// Backward: the forward's regions, then the backward's (all fp32), each on a
// 256-byte boundary. Slots are chunk slots (chunk_slot_bound), tokens the
// flattened B*T axis.
constexpr int kBwdEpiWarps = 4864;    // warps of the RMSNorm backward (152 SMs x 32)
constexpr int kBwdConvTokens = 256;   // tokens per block of the conv backward
struct BwdLayout {
    Layout f;                // the forward's regions (q, k, v, beta, gamma, o, ...)
    size_t h0;               // [slot][Hv][dk][dv]  state at each chunk's start
    size_t dh1;              // [slot][Hv][dk][dv]  gradient of the state at each chunk's end
    size_t uq;               // [slot][Hv][dk][dv]  Q^T diag(e^gam) dO' of each chunk
    size_t mats;             // [slot][Hv][3][64][64] T, decayed Q K^T, decayed K K^T
    size_t vn, dO, dR, wv;   // [Hv][ntok][dv]      new values; o, then scale * dL/do;
                             //                     dL/d(beta (v - e^g K H)); Pm^T dO'
    size_t dq, dk;           // [Hv][ntok][dk]      gradients of the normalised q, k per v head
    size_t dbeta, dgam;      // [Hv][ntok]          gradients of beta and of the per-token decay g
    size_t dz;               // [ntok][ch]          gradient of the pre-activation conv output
    size_t pa;               // [2][Hv][ntok]       per-token terms of ddt_bias and dA_log
    size_t pnorm;            // [kBwdEpiWarps][dv]  per-warp partial sums of dnorm_w
    size_t pconv;            // [blocks][ch][4]     per-block partial sums of dconv_w
    size_t xbuf;             // [slot][Hv][3][64][dk] dO' H0^T, dR0 H0^T, Vn dH1^T (tensor-core path)
    size_t hdbuf;            // [slot][Hv]          <H0, dH1> (tensor-core path)
    size_t total;
};
inline int64_t bwd_epi_warps(const gdn_desc &d) {
    const int64_t rows = (int64_t)d.B * d.T * d.Hv;
    return rows < kBwdEpiWarps ? (rows > 0 ? rows : 1) : kBwdEpiWarps;
}
inline int64_t bwd_conv_blocks(const gdn_desc &d) {
    const int64_t ntok = (int64_t)d.B * d.T;
    return ntok > 0 ? (ntok + kBwdConvTokens - 1) / kBwdConvTokens : 1;
}
inline BwdLayout make_bwd_layout(const gdn_desc &d) {
    BwdLayout L;
    L.f = make_layout(d);
    const size_t ntok = (size_t)d.B * (size_t)d.T, slots = (size_t)chunk_slot_bound(d);
    const size_t ch = 2 * (size_t)d.Hk * d.dk + (size_t)d.Hv * d.dv;
    const size_t st = (size_t)d.Hv * d.dk * d.dv * 4;
    size_t off = L.f.total;
    L.h0 = off;    off = align_up(off + slots * st, 256);
    L.dh1 = off;   off = align_up(off + slots * st, 256);
    L.uq = off;    off = align_up(off + slots * st, 256);
    L.mats = off;  off = align_up(off + slots * d.Hv * 3 * 64 * 64 * 4, 256);
    L.vn = off;    off = align_up(off + (size_t)d.Hv * ntok * d.dv * 4, 256);
    L.dO = off;    off = align_up(off + (size_t)d.Hv * ntok * d.dv * 4, 256);
    L.dR = off;    off = align_up(off + (size_t)d.Hv * ntok * d.dv * 4, 256);
    L.wv = off;    off = align_up(off + (size_t)d.Hv * ntok * d.dv * 4, 256);
    L.dq = off;    off = align_up(off + (size_t)d.Hv * ntok * d.dk * 4, 256);
    L.dk = off;    off = align_up(off + (size_t)d.Hv * ntok * d.dk * 4, 256);
    L.dbeta = off; off = align_up(off + (size_t)d.Hv * ntok * 4, 256);
    L.dgam = off;  off = align_up(off + (size_t)d.Hv * ntok * 4, 256);
    L.dz = off;    off = align_up(off + ntok * ch * 4, 256);
    L.pa = off;    off = align_up(off + 2 * (size_t)d.Hv * ntok * 4, 256);
    L.pnorm = off; off = align_up(off + (size_t)bwd_epi_warps(d) * d.dv * 4, 256);
    L.pconv = off; off = align_up(off + (size_t)bwd_conv_blocks(d) * ch * 4 * 4, 256);
    L.xbuf = off;  off = align_up(off + slots * d.Hv * 3 * 64 * (size_t)d.dk * 4, 256);
    L.hdbuf = off; off = align_up(off + slots * d.Hv * 4, 256);
    L.total = off;
    return L;
}
struct BwdProblem {
    Problem f;                          // the forward's inputs and workspace pointers
    const void *grad_out;               // act dtype [B*T][Hv][dv]
    const float *grad_final;            // [N][Hv][dk][dv] or null
    void *dq_raw, *dk_raw, *dv_raw;     // act dtype, dense [B*T][Hk*dk] / [B*T][Hv*dv]
    void *da, *db;                      // act dtype [B*T][Hv]
    void *dgate;                        // gate dtype [B*T][Hv*dv]
    float *dconv_w, *dA_log, *ddt_bias, *dnorm_w, *dinit;
    float *h0, *dh1, *uq, *mats, *vn, *dO, *dR, *wv, *dq, *dk, *dbeta, *dgam, *dz, *pa, *pnorm, *pconv;
    float *xbuf, *hdbuf;
};
cudaError_t launch_backward(const BwdProblem &p, cudaStream_t s);
// the per-chunk gradients' dv contractions on the tensor cores (gdn_backward_tc.cu)
bool chunk_x_tc_supports(const gdn_desc &d);
cudaError_t launch_chunk_x_tc(const BwdProblem &p, int64_t slots, cudaStream_t s);
// the outputs O on the tensor cores (gdn_backward_tc.cu)
bool out_tc_supports(const gdn_desc &d);
cudaError_t launch_out_tc(const BwdProblem &p, int64_t slots, cudaStream_t s);
// the dO' terms U, W on the tensor cores (gdn_backward_tc.cu)
bool dterms_tc_supports(const gdn_desc &d);
cudaError_t launch_dterms_tc(const BwdProblem &p, int64_t slots, cudaStream_t s);

// Decode (one token per sequence, d.T == 1): workspace regions, all fp32 but o.
struct DecodeLayout {
    size_t status, q, k, v, beta, g, o, total;
};
inline DecodeLayout make_decode_layout(const gdn_desc &d) {
    const size_t B = (size_t)d.B;
    DecodeLayout L;
    size_t off = 0;
    L.status = off; off = align_up(off + 256, 256);
    L.q = off;      off = align_up(off + 4 * B * d.Hk * d.dk, 256);   // [Hk][B][dk]
    L.k = off;      off = align_up(off + 4 * B * d.Hk * d.dk, 256);   // [Hk][B][dk]
    L.v = off;      off = align_up(off + 4 * B * d.Hv * d.dv, 256);   // [B][Hv*dv]
    L.beta = off;   off = align_up(off + 4 * B * d.Hv, 256);          // [B][Hv]
    L.g = off;      off = align_up(off + 4 * B * d.Hv, 256);          // [B][Hv]
    L.o = off;      off = align_up(off + act_size(d.dtype) * B * d.Hv * d.dv, 256);   // [B][Hv][dv], as o
    L.total = off;
    return L;
}
struct DecodeProblem {
    gdn_desc d;
    const void *q_raw, *k_raw, *v_raw, *a, *b, *conv_w;
    const float *A_log, *dt_bias;
    void *conv_state;
    float *state;
    int32_t *status;
    float *q, *k, *v, *beta, *g;
    void *o;
};
cudaError_t launch_decode(const DecodeProblem &p, cudaStream_t s);

}  // namespace gdn
