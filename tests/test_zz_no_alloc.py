"""The no-allocation entry point, gdn_forward_static_ws, against gdn_forward.

gdn_forward_static_ws serves callers that cannot allocate device memory (code
inside another framework's memory arena, plugins without an allocator, hosts
that forbid allocation while serving): it keeps its scratch in a fixed device
array inside the library instead of a caller-provided workspace. The array is
shared by every call and keeps the last call's contents, so each checked call
here comes right after a different problem on the same array (another shape,
packing and initial state), and once after a call that failed on the device
(a malformed cu_seqlens). Every call goes through the C ABI; its result must
equal the ordinary entry point's bit for bit, its status word (read with
gdn_static_ws_device_status) must say GDN_OK, and for the small workloads the
output must also match the oracle within the parity tolerances. A problem
larger than the fixed array is refused. This file is collected last.
"""
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import build, gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    gdn.load()
    return torch.device("cuda:0")


def static_call(inp, d, out, fin, check_rc=True):
    return gdn.gdn_forward_static_ws(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate,
                                     inp.conv_w, inp.A_log, inp.dt_bias, inp.norm_w, inp.cu_seqlens,
                                     inp.initial_state, out, fin, check=check_rc)


CASES = {
    "tiny_fp32": (WORKLOADS["tiny_fp32"], None),
    "ragged_fp16": (WORKLOADS["ragged_fp16"], None),
    "packed_bf16": (replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4, dk=64, dv=64, n_packed=3, gate_extra=3,
                            init_state_std=0.1), [70, 1, 130]),
}
# a different problem run on the array before each checked call
OTHER = (replace(WORKLOADS["layer_bf16"], B=1, T=190, Hk=1, Hv=2, dk=128, dv=128, init_state_std=0.1), None)


def run_static(inp, d, like_out, like_fin):
    out = torch.full_like(like_out, float("nan"))
    fin = torch.full_like(like_fin, float("nan"))
    static_call(inp, d, out, fin)
    assert gdn.gdn_static_ws_device_status() == gdn.GDN_OK
    return out, fin


@pytest.mark.parametrize("name", list(CASES))
def test_static_workspace_matches_forward_twice(dev, name):
    w, lengths = CASES[name]
    inp_cpu = make_inputs(w, lengths=lengths)
    inp = to_device(inp_cpu, dev)
    ref = gdn.forward(inp)
    d = ref.desc
    assert gdn.gdn_workspace_bytes(d) <= gdn.GDN_STATIC_WORKSPACE_BYTES
    ow, ol = OTHER
    other = to_device(make_inputs(ow, ol), dev)
    other_ref = gdn.forward(other)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_forward(inp_cpu)
    for call in range(2):
        # another problem on the shared array first: its leftovers must not matter
        o2, f2 = run_static(other, other_ref.desc, other_ref.out, other_ref.final_state)
        torch.cuda.synchronize()
        assert torch.equal(o2.view(torch.uint8), other_ref.out.view(torch.uint8))
        out, fin = run_static(inp, d, ref.out, ref.final_state)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: identical bits
        assert torch.equal(out.view(torch.uint8), ref.out.view(torch.uint8))
        assert torch.equal(fin, ref.final_state)
        check(out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"static {name} call {call} out")
        check(fin.cpu().numpy(), ref_fin, w.dtype, f"static {name} call {call} final_state")


def test_static_workspace_after_device_error(dev):
    """A packed call with a malformed cu_seqlens reports GDN_ERR_DEVICE_SEQLENS
    through the static status word; the next well-formed call is unaffected."""
    w, lengths = CASES["packed_bf16"]
    inp = to_device(make_inputs(w, lengths=lengths), dev)
    ref = gdn.forward(inp)
    good = inp.cu_seqlens.clone()
    inp.cu_seqlens = torch.tensor([0, 70, 60, 201], dtype=torch.int32, device=dev)   # decreasing
    out = torch.empty_like(ref.out)
    fin = torch.empty_like(ref.final_state)
    static_call(inp, ref.desc, out, fin)
    assert gdn.gdn_static_ws_device_status() == gdn.GDN_ERR_DEVICE_SEQLENS
    inp.cu_seqlens = good
    out, fin = run_static(inp, ref.desc, ref.out, ref.final_state)
    torch.cuda.synchronize()
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
