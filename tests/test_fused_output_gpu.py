"""The output step fused into the transposed chunk kernel.

Where the transposed chain holds a token's whole v-head row (dv = 128) and the
gate is a 16-bit view a tensor map can address, gdn_forward applies the gated
RMSNorm ("GDN Elementwise Fusion", post-GDR requirements; "Execution and
numerical behavior": the RMSNorm result is rounded to the activation dtype before
the fp32 SiLU-gating product) inside the chain instead of in a separate kernel.
The fused step reads the o rows back in the separate kernel's layout and repeats
its arithmetic and order of sums, so gdn_forward must equal the three stage calls
(prologue, chunk rule, output step) bit for bit; one case is also checked against
the oracle. Cases: ragged packed sequences with an empty and a one-token sequence
and a strided gate; two batch rows; fp16 with fp32 norm weights; and a gate view
at an odd element offset, which the fused step does not take (the separate kernel
runs), to show that the fallback gives the same bits. Which path ran is observed,
not assumed: the fused step never writes the intermediate o of the workspace, so
a NaN pattern put there beforehand survives it and is overwritten by the separate
path. A non-finite output reports GDN_ERR_DEVICE_RANGE from the fused step as it
does from the separate kernel.
"""
from types import SimpleNamespace

import pytest
import torch

from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu

BASE = WORKLOADS["varlen_bf16"]
CASES = {
    "packed_bf16_dk128": (replace(BASE, name="fo_packed", Hk=2, Hv=4, n_packed=0, init_state_std=0.1),
                          [70, 1, 130, 0, 64, 200]),
    "batch2_bf16_dk128": (replace(BASE, name="fo_batch", B=2, T=300, Hk=2, Hv=2, n_packed=0), None),
    "fp16_dk64_normf32": (replace(BASE, name="fo_fp16", dtype="fp16", B=1, T=257, Hk=1, Hv=2, dk=64,
                                  n_packed=0, gate_extra=0), None),
}


def staged(di, d):
    b = gdn.alloc(d, "cuda")
    cu = di.cu_seqlens
    gdn.gdn_prologue(d, di.q_raw, di.k_raw, di.v_raw, di.a, di.b, di.conv_w, di.A_log, di.dt_bias, cu,
                     b.workspace, b.ws_bytes)
    gdn.gdn_chunk_rule(d, cu, di.initial_state, b.final_state, b.workspace, b.ws_bytes)
    gdn.gdn_epilogue(d, di.gate, di.norm_w, b.out, b.workspace, b.ws_bytes)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(b.workspace) == gdn.GDN_OK
    return b


def view(di, **kw):
    """An Inputs-like object with some tensors replaced (gdn.forward reads attributes)."""
    fields = dict(w=di.w, q_raw=di.q_raw, k_raw=di.k_raw, v_raw=di.v_raw, a=di.a, b=di.b, gate=di.gate,
                  conv_w=di.conv_w, A_log=di.A_log, dt_bias=di.dt_bias, norm_w=di.norm_w,
                  cu_seqlens=di.cu_seqlens, initial_state=di.initial_state)
    fields.update(kw)
    return SimpleNamespace(**fields)


SENTINEL = 0x7E7E   # an fp16 NaN pattern: no finite o has these bits


def forward_marked(di):
    """gdn.forward with the workspace's intermediate o filled with SENTINEL first;
    returns the buffers and whether o was left untouched (the fused step ran)."""
    a = gdn.alloc(gdn.make_desc(di), "cuda")
    o = a.ws_view("o").view(torch.int16)
    o.fill_(SENTINEL)
    gdn.forward(di, a)
    torch.cuda.synchronize()
    hits = int((o == SENTINEL).sum())
    assert hits in (0, o.numel()), "o partly written"
    return a, hits == o.numel()


def run_both(di, fused=True):
    a, untouched = forward_marked(di)
    assert untouched == fused
    assert gdn.gdn_device_status(a.workspace) == gdn.GDN_OK
    b = staged(di, a.desc)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    assert torch.equal(a.final_state, b.final_state)
    return a


@pytest.mark.parametrize("name", list(CASES))
def test_fused_output_equals_stage_calls(name):
    w, lengths = CASES[name]
    inp = make_inputs(w, lengths)
    di = to_device(inp, "cuda")
    if name == "fp16_dk64_normf32":
        di = view(di, norm_w=di.norm_w.float())
    a = run_both(di)
    if name == "packed_bf16_dk128":
        ref_out, ref_fin = oracle_forward(inp)
        check(a.out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} out")
        check(a.final_state.cpu().numpy(), ref_fin, w.dtype, f"{name} final_state")


def test_unaligned_gate_takes_the_separate_output_step():
    w, lengths = CASES["packed_bf16_dk128"]
    di = to_device(make_inputs(replace(w, gate_extra=64), lengths), "cuda")
    ch = w.Hv * w.dv
    odd = di.gate_buf[..., 1:1 + ch]            # 2-byte offset: no tensor map, no fusion
    assert odd.data_ptr() % 16 != 0
    run_both(view(di, gate=odd), fused=False)


def test_fused_step_reports_non_finite_output():
    # bf16 activations keep their intermediates in fp16: a conv output beyond the fp16
    # range becomes inf, and the fused step's row sums see it
    w = replace(BASE, name="fo_range", B=1, T=70, Hk=1, Hv=1, dk=64, n_packed=0)
    inp = make_inputs(w)
    inp.v_raw[0, 5, :] = 1e30
    di = to_device(inp, "cuda")
    a, untouched = forward_marked(di)
    assert untouched
    assert gdn.gdn_device_status(a.workspace) == gdn.GDN_ERR_DEVICE_RANGE
    # the next well-formed call on the same buffers clears it
    di.v_raw[0, 5, :] = 0.5
    gdn.forward(di, a)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(a.workspace) == gdn.GDN_OK
