"""GPU parity of the decode step (gdn_decode_step) against the oracle.

Each case runs a few decode steps on the GPU from the same seeded, already
rounded inputs as the oracle's decode chain (tests/test_oracle_decode.py pins
that chain to the forward): every step's output within the GDN tolerances, the
state after the last step likewise, and the conv cache bit-exact (it holds raw
inputs). A prefill case checks the GPU forward + one GPU decode step against the
oracle forward over one more token.
"""
import numpy as np
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import gdn
from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace, to_device
from oracle import oracle as O
from tests._harness import check, flat, oracle_forward

pytestmark = pytest.mark.gpu

STEPS = 4

CASES = {
    "layer_bf16": replace(WORKLOADS["layer_bf16"], T=STEPS, init_state_std=0.1),
    "gqa_bf16": replace(WORKLOADS["long_gqa_bf16"], B=8, T=STEPS, init_state_std=0.1),
    "tiny_fp32": replace(WORKLOADS["tiny_fp32"], B=3, T=STEPS, init_state_std=0.1),
    "ragged_fp16": replace(WORKLOADS["ragged_fp16"], T=STEPS),
    # 16 sequences: with dv = 16 a step has few outputs, and the relative L2 error
    # of a small sample is dominated by the odd bf16 rounding flip of the RMSNorm
    "dk512_dv16_bf16": replace(WORKLOADS["layer_bf16"], name="dk512_dv16_bf16", B=16, Hk=1, Hv=2, dk=512,
                               dv=16, T=STEPS, init_state_std=0.1),
    "dk16_dv512_fp16": replace(WORKLOADS["ragged_fp16"], name="dk16_dv512_fp16", Hk=2, Hv=4, dk=16, dv=512,
                               T=STEPS),
}


def raw_cache(inp, t_end):
    """Raw q|k|v inputs of tokens t_end-3 .. t_end-1 per channel, zero before 0: [B, ch, 3]."""
    x = torch.cat([inp.q_raw, inp.k_raw, inp.v_raw], dim=2)
    B, _, ch = x.shape
    cache = torch.zeros((B, ch, 3), dtype=x.dtype)
    for r in range(3):
        t = t_end - 3 + r
        if t >= 0:
            cache[:, :, r] = x[:, t]
    return cache


def token(t, x):
    return x[:, t:t + 1]


def oracle_step(inp, t, cache, state):
    w = inp.w
    return O.decode(q_raw=flat(inp.q_raw[:, t]), k_raw=flat(inp.k_raw[:, t]), v_raw=flat(inp.v_raw[:, t]),
                    a=flat(inp.a[:, t]), b=flat(inp.b[:, t]), gate=flat(inp.gate[:, t].contiguous()),
                    conv_w=inp.conv_w.float().numpy(), A_log=inp.A_log.numpy(), dt_bias=inp.dt_bias.numpy(),
                    norm_w=inp.norm_w.float().numpy(), conv_state=cache, state=state,
                    Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv, dtype=w.dtype)


def gpu_step(d, dev_inp, t, cache, state, out, ws):
    di = dev_inp
    gdn.gdn_decode_step(d, token(t, di.q_raw), token(t, di.k_raw), token(t, di.v_raw), token(t, di.a),
                        token(t, di.b), token(t, di.gate), di.conv_w, di.A_log, di.dt_bias, di.norm_w,
                        cache, state, out, ws, ws.numel())


def decode_desc(di):
    w = di.w
    return gdn.desc_for(token(0, di.q_raw), token(0, di.k_raw), token(0, di.v_raw), token(0, di.a),
                        token(0, di.b), token(0, di.gate), di.norm_w, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv)


@pytest.mark.parametrize("name", list(CASES))
def test_decode_steps(name):
    w = CASES[name]
    inp = make_inputs(w)
    di = to_device(inp, "cuda")
    act = di.q_raw.dtype
    B, ch = w.B, 2 * w.Hk * w.dk + w.Hv * w.dv
    d = decode_desc(di)
    ws = torch.empty(gdn.gdn_decode_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    init = inp.initial_state if inp.initial_state is not None else torch.zeros((B, w.Hv, w.dk, w.dv))
    state = init.clone().cuda().contiguous()
    cache = torch.zeros((B, ch, 3), dtype=act, device="cuda")
    out = torch.empty((B, 1, w.Hv, w.dv), dtype=act, device="cuda")
    o_cache = np.zeros((B, ch, 3), np.float32)
    o_state = init.double().numpy()
    for t in range(STEPS):
        gpu_step(d, di, t, cache, state, out, ws)
        ref, cs64, st64 = oracle_step(inp, t, o_cache, o_state)
        check(out.float().cpu().numpy().reshape(B, w.Hv, w.dv), ref, w.dtype, f"decode {name} step {t} out")
        o_cache, o_state = cs64.astype(np.float32), st64
    torch.cuda.synchronize()
    check(state.cpu().numpy(), o_state, w.dtype, f"decode {name} state")
    np.testing.assert_array_equal(cache.float().cpu().numpy(), o_cache)
    assert torch.equal(cache.cpu(), raw_cache(inp, STEPS))
    assert gdn.gdn_device_status(ws) == gdn.GDN_OK


@pytest.mark.parametrize("name,P", [("layer_bf16", 70), ("gqa_bf16", 2)])
def test_prefill_then_decode(name, P):
    """GPU forward over P tokens (final state), cache = its last raw tokens, one GPU
    decode step: equals the oracle forward over P + 1 tokens at the last token."""
    w = replace(CASES[name], T=P + 1)
    inp = make_inputs(w)
    di = to_device(inp, "cuda")
    pre = gdn.desc_for(di.q_raw[:, :P], di.k_raw[:, :P], di.v_raw[:, :P], di.a[:, :P], di.b[:, :P],
                       di.gate[:, :P], di.norm_w, Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv)
    bufs = gdn.alloc(pre, "cuda")
    gdn.gdn_forward(pre, di.q_raw[:, :P], di.k_raw[:, :P], di.v_raw[:, :P], di.a[:, :P], di.b[:, :P],
                    di.gate[:, :P], di.conv_w, di.A_log, di.dt_bias, di.norm_w, None, di.initial_state,
                    bufs.out, bufs.final_state, bufs.workspace, bufs.ws_bytes)
    state = bufs.final_state
    cache = raw_cache(inp, P).cuda()
    d = decode_desc(di)
    ws = torch.empty(gdn.gdn_decode_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    out = torch.empty((w.B, 1, w.Hv, w.dv), dtype=di.q_raw.dtype, device="cuda")
    gpu_step(d, di, P, cache, state, out, ws)
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle_forward(inp)
    ref_last = ref_out.reshape(w.B, P + 1, w.Hv, w.dv)[:, P]
    check(out.float().cpu().numpy().reshape(w.B, w.Hv, w.dv), ref_last, w.dtype, f"prefill+decode {name} out")
    check(state.cpu().numpy(), ref_fin, w.dtype, f"prefill+decode {name} state")
    assert torch.equal(cache.cpu(), raw_cache(inp, P + 1))


def test_decode_reports_nonfinite_output():
    """An infinite input reaches the output: the device status says so."""
    w = replace(CASES["tiny_fp32"], B=2)
    inp = make_inputs(w)
    inp.v_raw[1, 0, 5] = float("inf")
    di = to_device(inp, "cuda")
    d = decode_desc(di)
    ws = torch.empty(gdn.gdn_decode_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    ch = 2 * w.Hk * w.dk + w.Hv * w.dv
    cache = torch.zeros((w.B, ch, 3), dtype=torch.float32, device="cuda")
    state = torch.zeros((w.B, w.Hv, w.dk, w.dv), device="cuda")
    out = torch.empty((w.B, 1, w.Hv, w.dv), device="cuda")
    gpu_step(d, di, 0, cache, state, out, ws)
    assert gdn.gdn_device_status(ws) == gdn.GDN_ERR_DEVICE_RANGE
