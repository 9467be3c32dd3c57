"""GPU parity of the segmented chunk schedule of a long single sequence.

A single sequence of at least 256 chunks whose chain fills at most half of the
SMs is run in segments (the prep of the next segment beside the chain of the
current one, the state handed between segments through the workspace). These
cases take that schedule and are checked against the oracle like every other
forward: output and final state within the GDN tolerances.
"""
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu

CASES = {
    # 258 chunks (the last one ragged), random initial state
    "seg_bf16_ragged": replace(WORKLOADS["long_gqa_bf16"], name="seg_bf16_ragged", T=256 * 64 + 100,
                               Hk=1, Hv=2, dk=64, dv=64, init_state_std=0.1),
    # GQA 2 -> 4 heads, dk = 128, dv = 128, exactly 300 chunks
    "seg_gqa_bf16": replace(WORKLOADS["long_gqa_bf16"], name="seg_gqa_bf16", T=300 * 64, Hk=2, Hv=4),
}


def run(inp, staged):
    d = gdn.make_desc(inp)
    bufs = gdn.alloc(d, "cuda")
    if staged:
        gdn.gdn_prologue(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.conv_w, inp.A_log, inp.dt_bias,
                         None, bufs.workspace, bufs.ws_bytes)
        gdn.gdn_chunk_rule(d, None, inp.initial_state, bufs.final_state, bufs.workspace, bufs.ws_bytes)
        gdn.gdn_epilogue(d, inp.gate, inp.norm_w, bufs.out, bufs.workspace, bufs.ws_bytes)
    else:
        gdn.forward(inp, bufs)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    return bufs


@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_segmented_forward(name, staged):
    w = CASES[name]
    inp = make_inputs(w)
    bufs = run(to_device(inp, "cuda"), staged)
    ref_out, ref_fin = oracle_forward(inp)
    check(bufs.out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} out")
    check(bufs.final_state.cpu().numpy(), ref_fin, w.dtype, f"{name} final_state")


def test_segmented_is_deterministic():
    w = CASES["seg_bf16_ragged"]
    di = to_device(make_inputs(w), "cuda")
    a, b = run(di, False), run(di, False)
    assert torch.equal(a.out, b.out) and torch.equal(a.final_state, b.final_state)
