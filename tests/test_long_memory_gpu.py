"""GPU parity in the long-memory regime: the state carried from chunk to chunk
reaches the outputs.

With the workloads' decay recipe (A_log = log U[1, 16]) the decay over one
64-token chunk, exp(sum of g), is below 1e-2 nearly everywhere, so whatever a
kernel does with the state once a chunk has passed is numerically invisible.
These cases draw A_log = log U[0.001, 0.05] (``workloads.MILD``, the mild decay
the recurrence's closed-form pins use) and first assert that the draw really
keeps the carry alive (most full chunks decay by no more than 10x). They then
run every path that carries state through the C ABI against the oracle:

* the tensor-core chain at dk = 64, 128 and 256, hundreds of chunks, GQA, with
  and without an initial state;
* the segmented schedule of one long sequence (prep and chain segments, the
  state handed through the workspace);
* packed sequences with an initial state;
* the fp32 CUDA-core chunk kernel at dk = 512;
* the sequence-sharded path with four spans (span maps A far from zero);
* 64 decode steps after a prefill;
* the backward over six chunks (the carried state gradient);
* the long-context GQA configuration at its full 131072 tokens, two sampled
  v heads (fp32 carry over 2048 chunks).
"""
import numpy as np
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import context_parallel as cp
from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import (MILD, WORKLOADS, head_subproblem, make_cotangents,
                                                           make_inputs, replace, to_device)
from oracle import oracle as O
from tests._harness import check, check_grad, chunk_survival, oracle_backward, oracle_forward

pytestmark = pytest.mark.gpu


def mild(base, name, **kw):
    return replace(WORKLOADS[base], name=name, decay_range=MILD, **kw)


FORWARD = {
    # tensor-core chain, dk = 128, GQA 2 -> 4, two sequences of 257 chunks (ragged tail)
    "lm_tc_dk128_gqa": (mild("long_gqa_bf16", "lm_tc_dk128_gqa", B=2, T=256 * 64 + 19, Hk=2, Hv=4,
                             init_state_std=0.1), None),
    # tensor-core chain at the layer's head shape dk = 256, 200 chunks
    "lm_tc_dk256": (mild("layer_bf16", "lm_tc_dk256", B=2, T=200 * 64, Hk=1, Hv=2, dv=128), None),
    # fp16, dk = 64, 130 chunks, random initial state
    "lm_tc_dk64_fp16": (mild("ragged_fp16", "lm_tc_dk64_fp16", B=2, T=130 * 64 + 7, Hk=2, Hv=2, dv=64,
                             gate_extra=0), None),
    # one long sequence: the segmented schedule (300 chunks, GQA 2 -> 4)
    "lm_segmented": (mild("long_gqa_bf16", "lm_segmented", B=1, T=300 * 64 + 5, Hk=2, Hv=4,
                          init_state_std=0.1), None),
    # packed sequences with an initial state (long ones, a one-token one, an exact chunk)
    "lm_packed": (mild("varlen_bf16", "lm_packed", Hk=2, Hv=4, init_state_std=0.1, gate_extra=3),
                  [3000, 1, 700, 4100, 64, 2500]),
    # the fp32 CUDA-core chunk kernel at the widest key dimension
    "lm_fp32_dk512": (mild("tiny_fp32", "lm_fp32_dk512", B=1, T=10 * 64 + 3, Hk=1, Hv=2, dk=512, dv=64,
                           init_state_std=0.1), None),
    "lm_fp32_gqa": (mild("tiny_fp32", "lm_fp32_gqa", B=2, T=40 * 64, Hk=1, Hv=2, dk=64, dv=64,
                         init_state_std=0.1), None),
}


def run_forward(inp):
    di = to_device(inp, "cuda")
    bufs = gdn.forward(di)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    return bufs


@pytest.mark.parametrize("name", list(FORWARD))
def test_long_memory_forward(name):
    w, lengths = FORWARD[name]
    inp = make_inputs(w, lengths)
    surv = chunk_survival(inp)
    print(f"[long-memory] {name}: {surv:.2f} of full chunks keep >= 0.1 of the state")
    assert surv >= 0.5
    bufs = run_forward(inp)
    ref_out, ref_fin = oracle_forward(inp)
    check(bufs.out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} out")
    check(bufs.final_state.cpu().numpy(), ref_fin, w.dtype, f"{name} final_state")


def test_long_memory_segmented_staged_equals_forward():
    """The segmented schedule through the three stage calls equals gdn_forward bitwise."""
    w, _ = FORWARD["lm_segmented"]
    di = to_device(make_inputs(w), "cuda")
    a = gdn.forward(di)
    d = a.desc
    b = gdn.alloc(d, "cuda")
    gdn.gdn_prologue(d, di.q_raw, di.k_raw, di.v_raw, di.a, di.b, di.conv_w, di.A_log, di.dt_bias, None,
                     b.workspace, b.ws_bytes)
    gdn.gdn_chunk_rule(d, None, di.initial_state, b.final_state, b.workspace, b.ws_bytes)
    gdn.gdn_epilogue(d, di.gate, di.norm_w, b.out, b.workspace, b.ws_bytes)
    torch.cuda.synchronize()
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.final_state, b.final_state)


def test_long_memory_full_length_sampled_heads():
    """The long-context GQA configuration (131072 tokens, 16 -> 32 heads) with
    mild decay: two seeded v heads over the whole sequence (2048 chunks)."""
    w = mild("long_gqa_bf16", "lm_long_gqa_full")
    inp = make_inputs(w)
    g = torch.Generator().manual_seed(1234 + w.seed)
    heads = sorted(torch.randperm(w.Hv, generator=g)[:2].tolist())
    sub = head_subproblem(inp, heads)
    assert chunk_survival(sub) >= 0.5
    bufs = run_forward(inp)
    ref_out, ref_fin = oracle_forward(sub, threads=2)
    d = bufs.desc
    out = bufs.out.float().cpu().reshape(d.B * d.T, d.Hv, d.dv).numpy()[:, heads]
    check(out, ref_out, w.dtype, f"long_gqa mild heads {heads} out")
    check(bufs.final_state.cpu().numpy()[:, heads], ref_fin, w.dtype, f"long_gqa mild heads {heads} final_state")


def test_long_memory_spans():
    """Four spans of one sequence: each span's map A is far from zero, so the
    scan's A H_in term matters; outputs and final state against the oracle."""
    w = mild("long_gqa_bf16", "lm_spans", T=1500, Hk=2, Hv=4, init_state_std=0.1)
    inp = make_inputs(w)
    assert chunk_survival(inp) >= 0.5
    di = to_device(inp, "cuda")
    cuts = [0, 333, 700, 1100, 1500]
    ts = (di.q_raw, di.k_raw, di.v_raw, di.a, di.b, di.gate, di.conv_w, di.A_log, di.dt_bias, di.norm_w)
    # the map of the second span, from the library: |A| must not vanish
    s0, s1 = cuts[1], cuts[2]
    sl = lambda t: t[:, s0:s1].contiguous()
    pre = cp.tail_tokens(di.q_raw[:, :s0], di.k_raw[:, :s0], di.v_raw[:, :s0]).unsqueeze(0)
    A, _ = cp.span_maps(sl(di.q_raw), sl(di.k_raw), sl(di.v_raw), sl(di.a), sl(di.b), sl(di.gate), di.conv_w,
                        di.A_log, di.dt_bias, di.norm_w, pre, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv)
    torch.cuda.synchronize()
    amax = float(A.abs().amax())
    print(f"[long-memory] span map max |A| = {amax:.3e}")
    assert amax > 0.05
    out, fin = cp.emulate(*ts, cuts, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv, initial_state=di.initial_state)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_forward(inp)
    check(out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, "spans mild out")
    check(fin.cpu().numpy(), ref_fin, w.dtype, "spans mild final_state")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_long_memory_decode(dtype):
    """A GPU prefill of 64 tokens, then 64 GPU decode steps, each against the
    oracle forward over the same tokens (outputs of the decoded tokens and the
    final state)."""
    P, S = 64, 64
    base = "long_gqa_bf16" if dtype == "bf16" else "tiny_fp32"
    w = mild(base, f"lm_decode_{dtype}", B=4, T=P + S, Hk=2, Hv=4, init_state_std=0.1,
             **({"dk": 64, "dv": 64} if dtype == "fp32" else {}))
    inp = make_inputs(w)
    di = to_device(inp, "cuda")
    pre = gdn.desc_for(di.q_raw[:, :P], di.k_raw[:, :P], di.v_raw[:, :P], di.a[:, :P], di.b[:, :P],
                       di.gate[:, :P], di.norm_w, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv)
    bufs = gdn.alloc(pre, "cuda")
    gdn.gdn_forward(pre, di.q_raw[:, :P], di.k_raw[:, :P], di.v_raw[:, :P], di.a[:, :P], di.b[:, :P],
                    di.gate[:, :P], di.conv_w, di.A_log, di.dt_bias, di.norm_w, None, di.initial_state,
                    bufs.out, bufs.final_state, bufs.workspace, bufs.ws_bytes)
    state = bufs.final_state
    x = torch.cat([inp.q_raw, inp.k_raw, inp.v_raw], dim=2)
    cache = x[:, P - 3:P].permute(0, 2, 1).contiguous().cuda()
    tok = lambda t, y: y[:, t:t + 1]
    d = gdn.desc_for(tok(0, di.q_raw), tok(0, di.k_raw), tok(0, di.v_raw), tok(0, di.a), tok(0, di.b),
                     tok(0, di.gate), di.norm_w, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv)
    ws = torch.empty(gdn.gdn_decode_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    outs = []
    for t in range(P, P + S):
        out = torch.empty((w.B, 1, w.Hv, w.dv), dtype=di.q_raw.dtype, device="cuda")
        gdn.gdn_decode_step(d, tok(t, di.q_raw), tok(t, di.k_raw), tok(t, di.v_raw), tok(t, di.a), tok(t, di.b),
                            tok(t, di.gate), di.conv_w, di.A_log, di.dt_bias, di.norm_w, cache, state, out, ws,
                            ws.numel())
        outs.append(out)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(ws) == gdn.GDN_OK
    ref_out, ref_fin = oracle_forward(inp)
    ref = ref_out.reshape(w.B, P + S, w.Hv, w.dv)[:, P:]
    got = torch.cat(outs, dim=1).float().cpu().numpy()
    check(got, ref, w.dtype, f"decode mild {dtype} out")
    check(state.cpu().numpy(), ref_fin, w.dtype, f"decode mild {dtype} state")


BACKWARD = {
    # six chunks per sequence at the tensor-core shape, GQA, initial state
    "lm_bwd_bf16": (mild("long_gqa_bf16", "lm_bwd_bf16", B=2, T=6 * 64 + 10, Hk=1, Hv=2, dk=64, dv=64,
                         init_state_std=0.1), None),
    "lm_bwd_fp32": (mild("tiny_fp32", "lm_bwd_fp32", B=1, T=6 * 64, Hk=1, Hv=2, dk=32, dv=32,
                         init_state_std=0.1), None),
    "lm_bwd_packed_bf16": (mild("varlen_bf16", "lm_bwd_packed_bf16", Hk=1, Hv=2, dk=64, dv=64,
                                init_state_std=0.1), [400, 1, 70, 200]),
}
TOL = {"fp32": (1e-4, 1e-3), "bf16": (1e-2, 5e-2), "fp16": (1e-2, 5e-2)}
NAMES = ("dq_raw", "dk_raw", "dv_raw", "da", "db", "dgate", "dconv_w", "dA_log", "ddt_bias", "dnorm_w",
         "dinitial_state")


@pytest.mark.parametrize("name", list(BACKWARD))
def test_long_memory_backward(name):
    w, lengths = BACKWARD[name]
    inp = make_inputs(w, lengths)
    assert chunk_survival(inp) >= 0.5
    gout, gfin = make_cotangents(inp)
    di = to_device(inp, "cuda")
    grads = gdn.backward(di, gout.cuda(), gfin.cuda())
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(grads.workspace) == gdn.GDN_OK
    ref = oracle_backward(inp, gout, gfin)
    # the gradient of the initial state crosses every chunk: it must not vanish
    assert np.abs(ref["dinitial_state"]).max() > 1e-2
    for n in NAMES:
        got = getattr(grads, n).float().cpu().numpy()
        check_grad(got.reshape(ref[n].shape), ref[n], w.dtype, f"{name} {n}", TOL[w.dtype])
