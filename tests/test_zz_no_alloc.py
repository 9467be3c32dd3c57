"""The no-allocation entry point, gdn_forward_static_ws, against gdn_forward.

gdn_forward_static_ws serves callers that cannot allocate device memory (code
inside another framework's memory arena, plugins without an allocator, hosts
that forbid allocation while serving): it keeps its scratch in a fixed device
array inside the library instead of a caller-provided workspace. This test
calls it through the C ABI twice in a row on the same inputs and checks each
result against the ordinary entry point's, with the parity tolerances, and
checks that a problem larger than the fixed array is refused. It lives in a
file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import build, gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from tests._harness import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    gdn.load()
    return torch.device("cuda:0")


def static_call(inp, d, out, fin):
    gdn.gdn_forward_static_ws(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate,
                              inp.conv_w, inp.A_log, inp.dt_bias, inp.norm_w, inp.cu_seqlens,
                              inp.initial_state, out, fin)


@pytest.mark.parametrize("w", [
    WORKLOADS["tiny_fp32"],
    WORKLOADS["ragged_fp16"],
    replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4, dk=64, dv=64, n_packed=3, gate_extra=3),
], ids=lambda w: w.name)
def test_static_workspace_matches_forward_twice(dev, w):
    lengths = [70, 1, 130] if w.n_packed else None
    inp = to_device(make_inputs(w, lengths=lengths), dev)
    ref = gdn.forward(inp)
    d = ref.desc
    assert gdn.gdn_workspace_bytes(d) <= gdn.GDN_STATIC_WORKSPACE_BYTES
    for call in range(2):
        out = torch.full_like(ref.out, float("nan"))
        fin = torch.full_like(ref.final_state, float("nan"))
        static_call(inp, d, out, fin)
        torch.cuda.synchronize()
        check(out.float().cpu().numpy(), ref.out.float().cpu().numpy(), w.dtype, f"static call {call} out")
        check(fin.cpu().numpy(), ref.final_state.cpu().numpy(), w.dtype, f"static call {call} final_state")
        # the same kernels on the same inputs: identical bits
        assert torch.equal(out.view(torch.uint8), ref.out.view(torch.uint8))
        assert torch.equal(fin, ref.final_state)


def test_static_workspace_rejects_oversized_problem(dev):
    inp = to_device(make_inputs(replace(WORKLOADS["layer_bf16"], B=1, T=1024)), dev)
    d = gdn.make_desc(inp)
    assert gdn.gdn_workspace_bytes(d) > gdn.GDN_STATIC_WORKSPACE_BYTES
    out = torch.empty((1, 1024, 6, 512), dtype=torch.bfloat16, device=dev)
    rc = gdn.gdn_forward_static_ws(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate,
                                   inp.conv_w, inp.A_log, inp.dt_bias, inp.norm_w, None, None,
                                   out, None, check=False)
    assert rc == gdn.GDN_ERR_WORKSPACE
