"""Guard bands around every buffer the forward writes.

out, final_state and the workspace are each placed inside a larger buffer whose
4 KiB bands on both sides hold a fixed byte pattern; after gdn_forward the
bands must be unchanged and the outputs must match the oracle. The cases are
the ones where an off-by-one store would land: ragged tails, packed sequences
(an empty one, a one-token one, an exact chunk), a single token, and both
tensor-core chain forms.
"""
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu

BAND = 4096
FILL = 0xA5

CASES = {
    "ragged_fp16": (WORKLOADS["ragged_fp16"], None),
    "packed_bf16_dk64": (replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4, dk=64, dv=128, gate_extra=3,
                                 init_state_std=0.1), [1, 64, 65, 0, 130, 3]),
    "packed_bf16_dk128": (replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4, gate_extra=0), [70, 1, 130, 64]),
    "one_token_fp32": (replace(WORKLOADS["tiny_fp32"], B=2, T=1, init_state_std=0.1), None),
    "one_token_bf16": (replace(WORKLOADS["layer_bf16"], B=3, T=1, Hk=1, Hv=2, dk=128, dv=128), None),
    "ragged_dk256": (replace(WORKLOADS["layer_bf16"], B=1, T=130, Hk=1, Hv=2, dv=128, init_state_std=0.1), None),
}


def guarded(nbytes, device):
    buf = torch.full((BAND + nbytes + BAND,), FILL, dtype=torch.uint8, device=device)
    return buf, buf[BAND:BAND + nbytes]


def bands_intact(buf, nbytes):
    lo, hi = buf[:BAND], buf[BAND + nbytes:]
    return bool((lo == FILL).all()) and bool((hi == FILL).all())


@pytest.mark.parametrize("name", list(CASES))
def test_guard_bands_untouched(name):
    w, lengths = CASES[name]
    inp = make_inputs(w, lengths)
    di = to_device(inp, "cuda")
    d = gdn.make_desc(di)
    act = di.q_raw.dtype
    n_tok = d.B * d.T
    out_bytes = n_tok * w.Hv * w.dv * torch.tensor([], dtype=act).element_size()
    fin_bytes = d.N * w.Hv * w.dk * w.dv * 4
    ws_bytes = gdn.gdn_workspace_bytes(d)
    ob, o_in = guarded(out_bytes, "cuda")
    fb, f_in = guarded(fin_bytes, "cuda")
    wb, w_in = guarded(ws_bytes, "cuda")
    out = o_in.view(act).view(d.B, d.T, w.Hv, w.dv)
    fin = f_in.view(torch.float32).view(d.N, w.Hv, w.dk, w.dv)
    for call in range(2):
        gdn.gdn_forward(d, di.q_raw, di.k_raw, di.v_raw, di.a, di.b, di.gate, di.conv_w, di.A_log, di.dt_bias,
                        di.norm_w, di.cu_seqlens, di.initial_state, out, fin, w_in, ws_bytes)
        torch.cuda.synchronize()
        assert gdn.gdn_device_status(w_in) == gdn.GDN_OK
        assert bands_intact(ob, out_bytes), f"{name}: a store landed next to out"
        assert bands_intact(fb, fin_bytes), f"{name}: a store landed next to final_state"
        assert bands_intact(wb, ws_bytes), f"{name}: a store landed next to the workspace"
    ref_out, ref_fin = oracle_forward(inp)
    check(out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} out")
    check(fin.cpu().numpy(), ref_fin, w.dtype, f"{name} final_state")
