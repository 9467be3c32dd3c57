"""GPU parity of the sequence-sharded core and of the prefixed forward.

* gdn_forward_with_prefix on packed sequences, each with its own conv prefix,
  against the oracle forward with the same prefix.
* The span path (context_parallel.emulate: per span the conv prefix, the maps
  A, B from two prefixed forwards, gdn_span_scan, the span's forward from its
  scanned initial state) against the oracle forward of the whole sequence:
  outputs and final state within the GDN tolerances.
"""
import numpy as np
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import context_parallel as cp
from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from oracle import oracle as O
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu

SPLITS = {
    # tensor-core chunk path (bf16, dk = dv = 128), GQA 2 -> 4, random initial state
    "gqa_bf16_4spans": (replace(WORKLOADS["long_gqa_bf16"], T=333, Hk=2, Hv=4, init_state_std=0.1),
                        [0, 64, 200, 260, 333]),
    "gqa_bf16_short_span": (replace(WORKLOADS["long_gqa_bf16"], T=333, Hk=2, Hv=4), [0, 3, 130, 333]),
    # fp32 CUDA-core chunk path
    "tiny_fp32_2spans": (replace(WORKLOADS["tiny_fp32"], T=200, init_state_std=0.1), [0, 100, 200]),
}


def tensors(di):
    return (di.q_raw, di.k_raw, di.v_raw, di.a, di.b, di.gate, di.conv_w, di.A_log, di.dt_bias, di.norm_w)


@pytest.mark.parametrize("name", list(SPLITS))
def test_span_path_equals_whole_sequence(name):
    w, cuts = SPLITS[name]
    inp = make_inputs(w)
    di = to_device(inp, "cuda")
    out, fin = cp.emulate(*tensors(di), cuts, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv,
                          initial_state=di.initial_state)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_forward(inp)
    check(out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} out")
    check(fin.cpu().numpy(), ref_fin, w.dtype, f"{name} final_state")


@pytest.mark.parametrize("name", ["varlen_prefix_bf16", "ragged_prefix_fp16"])
def test_prefixed_forward(name):
    if name == "varlen_prefix_bf16":
        w, lengths = replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4), [70, 1, 130, 64]
    else:
        w, lengths = WORKLOADS["ragged_fp16"], None
    inp = make_inputs(w, lengths)
    n = inp.n_seq
    ch = 2 * w.Hk * w.dk + w.Hv * w.dv
    g = torch.Generator().manual_seed(5)
    prefix = torch.randn((n, 3, ch), generator=g).to(inp.q_raw.dtype)
    di = to_device(inp, "cuda")
    d = gdn.make_desc(di)
    bufs = gdn.alloc(d, "cuda")
    gdn.gdn_forward_with_prefix(d, *tensors(di), di.cu_seqlens, prefix.cuda(), di.initial_state, bufs.out,
                                bufs.final_state, bufs.workspace, bufs.ws_bytes)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    ref_out, ref_fin = oracle_forward(inp, conv_prefix=prefix.float().numpy())
    check(bufs.out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} out")
    check(bufs.final_state.cpu().numpy(), ref_fin, w.dtype, f"{name} final_state")


def test_span_scan_composes_maps():
    """H_in[s] = A[s-1] H_in[s-1] + B[s-1] on random maps (fp32 on both sides)."""
    S, Hv, dk, dv = 5, 3, 32, 64
    g = torch.Generator().manual_seed(3)
    A = torch.randn((S, Hv, dk, dk), generator=g) / dk ** 0.5
    B = torch.randn((S, Hv, dk, dv), generator=g)
    h0 = torch.randn((Hv, dk, dv), generator=g)
    H = torch.empty((S, Hv, dk, dv), device="cuda")
    gdn.gdn_span_scan(S, Hv, dk, dv, A.cuda(), B.cuda(), h0.cuda(), H)
    torch.cuda.synchronize()
    ref = [h0.double()]
    for s in range(S - 1):
        ref.append(A[s].double() @ ref[-1] + B[s].double())
    np.testing.assert_allclose(H.cpu().double().numpy(), torch.stack(ref).numpy(), rtol=0, atol=1e-4)
