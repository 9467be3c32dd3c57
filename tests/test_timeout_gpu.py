"""The bounded waits of the tensor-core kernels, driven on the GPU without a stall.

Every wait of the tensor-core chunk kernels (prep, both chain forms) on one of
their own mbarriers is bounded; on expiry the CTA records GDN_ERR_DEVICE_TIMEOUT,
drains its own copies and products (bounded), frees its tensor memory and
returns. gdn_set_wait_test_mode(1) makes a main-loop wait that is not already
complete give up at once (a non-blocking test), so the path runs on an ordinary
input. The test checks that the status word says so, and that the next call in
the normal mode, on the same workspace, returns GDN_OK and matches the oracle:
the context stays usable and nothing of the failed call leaks into the next.
"""
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu

CASES = {
    # dk = 256: the 64-column chain
    "chain64_dk256": replace(WORKLOADS["layer_bf16"], B=1, T=300, Hk=1, Hv=2, dv=128),
    # dk = 128: the transposed chain, GQA, packed sequences
    "chain_tm_dk128": (replace(WORKLOADS["varlen_bf16"], Hk=2, Hv=4, n_packed=3, gate_extra=0)),
}
LENGTHS = {"chain_tm_dk128": [200, 64, 130]}


@pytest.mark.parametrize("name", list(CASES))
def test_wait_timeout_reported_then_next_call_correct(name):
    w = CASES[name]
    inp = make_inputs(w, LENGTHS.get(name))
    di = to_device(inp, "cuda")
    bufs = gdn.forward(di)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    gdn.gdn_set_wait_test_mode(1)
    try:
        gdn.forward(di, bufs)
        status = gdn.gdn_device_status(bufs.workspace)
    finally:
        gdn.gdn_set_wait_test_mode(0)
    assert status == gdn.GDN_ERR_DEVICE_TIMEOUT
    bufs.out.fill_(float("nan"))
    bufs.final_state.fill_(float("nan"))
    gdn.forward(di, bufs)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    ref_out, ref_fin = oracle_forward(inp)
    check(bufs.out.float().cpu().numpy().reshape(ref_out.shape), ref_out, w.dtype, f"{name} after timeout out")
    check(bufs.final_state.cpu().numpy(), ref_fin, w.dtype, f"{name} after timeout final_state")
