"""GPU parity of the backward (gdn_backward) against the oracle backward.

Each case draws seeded, already-rounded inputs and cotangents, runs the GPU
backward through the C ABI and compares every gradient with the fp64 oracle
(itself pinned by finite differences of the oracle forward). Tolerances are
relative to each gradient's own scale (relative L2 and max |d| / max |ref|):
fp32 activations (1e-4, 1e-3); bf16 / fp16 (1e-2, 5e-2), where the act-dtype
rounding of the gradient outputs alone contributes about 2e-3 relative L2
(bf16) and the forward's fp16 intermediates (v, o) a few 1e-4.
"""
import numpy as np
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import (WORKLOADS, make_cotangents, make_inputs, replace,
                                                           to_device)
from tests._harness import check_grad, oracle_backward

pytestmark = pytest.mark.gpu

TOL = {"fp32": (1e-4, 1e-3), "bf16": (1e-2, 5e-2), "fp16": (1e-2, 5e-2)}

CASES = {
    "tiny_fp32": (replace(WORKLOADS["tiny_fp32"], init_state_std=0.1), None),
    "ragged_fp16": (WORKLOADS["ragged_fp16"], None),
    # three chunks per sequence, the last one ragged, at the layer's head shape
    "layer_bf16_T160": (replace(WORKLOADS["layer_bf16"], T=160), None),
    # packed GQA 2 -> 4 heads with a one-token sequence and an exact chunk, strided gate
    "packed_gqa_bf16": (replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4, init_state_std=0.1),
                        [70, 1, 130, 64]),
    # narrow and wide head shapes (the 16- and 32-column reverse-chain tiles)
    "dk32_dv16_fp32": (replace(WORKLOADS["tiny_fp32"], Hk=1, Hv=2, dk=32, dv=16, T=130), None),
    "dk512_dv64_bf16": (replace(WORKLOADS["layer_bf16"], B=1, Hk=1, Hv=1, dk=512, dv=64, T=70,
                                init_state_std=0.1), None),
}

NAMES = ("dq_raw", "dk_raw", "dv_raw", "da", "db", "dgate", "dconv_w", "dA_log", "ddt_bias", "dnorm_w",
         "dinitial_state")


def run_case(name, final=True):
    w, lengths = CASES[name]
    inp = make_inputs(w, lengths)
    gout, gfin = make_cotangents(inp, final=final)
    di = to_device(inp, "cuda")
    grads = gdn.backward(di, gout.cuda(), None if gfin is None else gfin.cuda())
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(grads.workspace) == gdn.GDN_OK
    return w, inp, gout, gfin, grads


@pytest.mark.parametrize("name", list(CASES))
def test_backward_parity(name):
    w, inp, gout, gfin, grads = run_case(name)
    ref = oracle_backward(inp, gout, gfin)
    for n in NAMES:
        got = getattr(grads, n).float().cpu().numpy()
        check_grad(got.reshape(ref[n].shape), ref[n], w.dtype, f"{name} {n}", TOL[w.dtype])


def test_backward_without_final_gradient():
    w, inp, gout, gfin, grads = run_case("ragged_fp16", final=False)
    ref = oracle_backward(inp, gout, None)
    for n in NAMES:
        got = getattr(grads, n).float().cpu().numpy()
        check_grad(got.reshape(ref[n].shape), ref[n], w.dtype, f"no grad_final {n}", TOL[w.dtype])


def test_backward_is_deterministic():
    w, lengths = CASES["packed_gqa_bf16"]
    inp = make_inputs(w, lengths)
    gout, gfin = make_cotangents(inp)
    di = to_device(inp, "cuda")
    a = gdn.backward(di, gout.cuda(), gfin.cuda())
    b = gdn.backward(di, gout.cuda(), gfin.cuda())
    torch.cuda.synchronize()
    for n in NAMES:
        assert torch.equal(getattr(a, n), getattr(b, n)), n


def test_backward_reports_malformed_seqlens():
    """A decreasing cu_seqlens sets the device status; the kernels skip their work."""
    w, lengths = CASES["packed_gqa_bf16"]
    inp = make_inputs(w, lengths)
    gout, gfin = make_cotangents(inp)
    di = to_device(inp, "cuda")
    di.cu_seqlens[2] = di.cu_seqlens[1] - 1
    grads = gdn.backward(di, gout.cuda(), gfin.cuda())
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(grads.workspace) == gdn.GDN_ERR_DEVICE_SEQLENS
