"""Parity of the CUDA path (called through the C ABI) with the CPU oracle, on
the same seeded, already-rounded inputs.

Full workloads are compared element by element; the two largest are compared
on two seeded v heads over their full length (the oracle's cost grows with
heads x tokens x dk x dv). Tolerances: see ``_harness.check``."""
import numpy as np
import pytest
import torch

from linear_attention_sequence_qkv_gb300 import build, gdn
from linear_attention_sequence_qkv_gb300.workloads import (WORKLOADS, head_subproblem, make_inputs,
                                                           replace, to_device)
from oracle import oracle as O
from tests._harness import check, oracle_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    gdn.load()
    return torch.device("cuda:0")


def run_gpu(inp_cpu, dev, want_final_state=True):
    inp = to_device(inp_cpu, dev)
    bufs = gdn.forward(inp, want_final_state=want_final_state)
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    torch.cuda.synchronize()
    return bufs, inp


def host_out(bufs):
    d = bufs.desc
    return bufs.out.float().cpu().reshape(d.B * d.T, d.Hv, d.dv).numpy()


def compare_full(inp_cpu, bufs, what):
    ref_out, ref_fin = oracle_forward(inp_cpu)
    dt = inp_cpu.w.dtype
    check(host_out(bufs), ref_out, dt, f"{what} out")
    if bufs.final_state is not None:
        check(bufs.final_state.cpu().numpy(), ref_fin, dt, f"{what} final_state")


def sampled_heads(w, k=2):
    g = torch.Generator().manual_seed(1234 + w.seed)
    heads = sorted(torch.randperm(w.Hv, generator=g)[:k].tolist())
    return heads


def compare_heads(inp_cpu, bufs, heads, what):
    sub = head_subproblem(inp_cpu, heads)
    ref_out, ref_fin = oracle_forward(sub, threads=len(heads))
    out = host_out(bufs)[:, heads]
    fin = bufs.final_state.cpu().numpy()[:, heads]
    dt = inp_cpu.w.dtype
    check(out, ref_out, dt, f"{what} heads {heads} out")
    check(fin, ref_fin, dt, f"{what} heads {heads} final_state")


# ----------------------------------------------------------- workloads
@pytest.mark.parametrize("name", ["tiny_fp32", "layer_bf16", "ragged_fp16"])
def test_workload_full(dev, name):
    inp = make_inputs(WORKLOADS[name])
    bufs, _ = run_gpu(inp, dev)
    compare_full(inp, bufs, name)


@pytest.mark.parametrize("name", ["long_gqa_bf16", "varlen_bf16"])
def test_workload_sampled_heads(dev, name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    bufs, _ = run_gpu(inp, dev)
    compare_heads(inp, bufs, sampled_heads(w), name)


# ----------------------------------------------- small cases and edges
SMALL = {
    # several chunks, ragged tail, GQA, initial state
    "fp32_gqa_ragged": replace(WORKLOADS["tiny_fp32"], B=2, T=150, Hk=2, Hv=4, dk=32, dv=64,
                               init_state_std=0.1),
    "bf16_tiles": replace(WORKLOADS["layer_bf16"], B=1, T=300, Hk=2, Hv=4, dk=128, dv=128),
    "fp16_min_dims": replace(WORKLOADS["ragged_fp16"], B=3, T=77, Hk=1, Hv=2, dk=16, dv=16,
                             gate_extra=5),
    "bf16_max_dims": replace(WORKLOADS["layer_bf16"], B=1, T=70, Hk=1, Hv=1, dk=512, dv=512,
                             init_state_std=0.1),
    "fp32_wide_k": replace(WORKLOADS["tiny_fp32"], B=1, T=65, Hk=1, Hv=2, dk=512, dv=16),
    "fp32_single_token": replace(WORKLOADS["tiny_fp32"], B=2, T=1, init_state_std=0.1),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases(dev, name):
    inp = make_inputs(SMALL[name])
    bufs, _ = run_gpu(inp, dev)
    compare_full(inp, bufs, name)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_packed_ragged_lengths(dev, dtype):
    # lengths 1, 64, 65, an empty sequence, 130, 3; misaligned strided gate
    lengths = [1, 64, 65, 0, 130, 3]
    w = replace(WORKLOADS["varlen_bf16"], dtype=dtype, Hk=2, Hv=4, dk=64, dv=32,
                n_packed=len(lengths), gate_extra=3, init_state_std=0.1)
    inp = make_inputs(w, lengths=lengths)
    bufs, _ = run_gpu(inp, dev)
    compare_full(inp, bufs, f"packed_{dtype}")


def test_fp32_gate_and_norm_weight_with_bf16_activations(dev):
    w = replace(WORKLOADS["layer_bf16"], B=2, T=90, Hk=2, Hv=2, dk=64, dv=64, gate_extra=8)
    inp = make_inputs(w)
    inp.gate_buf = inp.gate_buf.float()
    inp.norm_w = inp.norm_w.float()
    bufs, _ = run_gpu(inp, dev)
    compare_full(inp, bufs, "fp32_gate")


def test_empty_sequence_batch(dev):
    w = replace(WORKLOADS["tiny_fp32"], B=2, T=0, init_state_std=0.1)
    inp = make_inputs(w)
    bufs, _ = run_gpu(inp, dev)
    assert bufs.out.numel() == 0
    assert torch.equal(bufs.final_state.cpu(), inp.initial_state)


def test_malformed_cu_seqlens_reports_device_status(dev):
    lengths = [10, 20, 30]
    w = replace(WORKLOADS["varlen_bf16"], Hk=1, Hv=1, dk=64, dv=64, n_packed=3, gate_extra=0)
    inp = to_device(make_inputs(w, lengths=lengths), dev)
    bufs = gdn.forward(inp)
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK
    bad = torch.tensor([0, 30, 10, 60], dtype=torch.int32, device=dev)   # not non-decreasing
    inp.cu_seqlens = bad
    gdn.forward(inp, bufs)
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_ERR_DEVICE_SEQLENS
    inp.cu_seqlens = torch.tensor([0, 10, 30, 59], dtype=torch.int32, device=dev)  # wrong total
    gdn.forward(inp, bufs)
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_ERR_DEVICE_SEQLENS
    torch.cuda.synchronize()


def test_run_to_run_bitwise_deterministic(dev):
    inp = to_device(make_inputs(replace(WORKLOADS["layer_bf16"], T=256)), dev)
    b1 = gdn.forward(inp)
    o1, f1 = b1.out.clone(), b1.final_state.clone()
    gdn.forward(inp, b1)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), b1.out.view(torch.int16))
    assert torch.equal(f1, b1.final_state)


STAGED_CASES = {
    "ragged_fp16": WORKLOADS["ragged_fp16"],
    # gdn_forward chains its four kernels by programmatic dependent launch; the
    # stage calls run them plainly: the results must not differ by a bit
    "layer_bf16": WORKLOADS["layer_bf16"],
    "packed_gqa_bf16": replace(WORKLOADS["varlen_bf16"], n_packed=6, max_len=700, seed=5),
}


@pytest.mark.parametrize("name", list(STAGED_CASES))
def test_stages_equal_forward_bitwise(dev, name):
    inp = to_device(make_inputs(STAGED_CASES[name]), dev)
    b1 = gdn.forward(inp)
    d = b1.desc
    b2 = gdn.alloc(d, dev)
    gdn.gdn_prologue(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.conv_w, inp.A_log,
                     inp.dt_bias, inp.cu_seqlens, b2.workspace, b2.ws_bytes)
    gdn.gdn_chunk_rule(d, inp.cu_seqlens, inp.initial_state, b2.final_state, b2.workspace, b2.ws_bytes)
    gdn.gdn_epilogue(d, inp.gate, inp.norm_w, b2.out, b2.workspace, b2.ws_bytes)
    torch.cuda.synchronize()
    assert torch.equal(b1.out.view(torch.int16), b2.out.view(torch.int16))
    assert torch.equal(b1.final_state, b2.final_state)


def test_non_finite_intermediate_reports_device_status(dev):
    # bf16 activations keep their intermediates in fp16: a conv output beyond the
    # fp16 range becomes inf and the epilogue reports it
    w = replace(WORKLOADS["layer_bf16"], B=1, T=70, Hk=1, Hv=1, dk=64, dv=64)
    inp = make_inputs(w)
    inp.v_raw[0, 5, :] = 1e30
    bufs, _ = None, None
    dinp = to_device(inp, dev)
    bufs = gdn.forward(dinp)
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_ERR_DEVICE_RANGE
    # the next well-formed call clears it
    dinp.v_raw[0, 5, :] = 0.5
    gdn.forward(dinp, bufs)
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK


@pytest.mark.parametrize("name", ["ragged_fp16", "tiny_fp32", "layer_bf16"])
def test_prologue_intermediates(dev, name):
    """q/k/v after conv, SiLU and L2 norm, beta and the in-chunk cumulative
    decay, read from the workspace, against the oracle's pinned steps."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    bufs, _ = run_gpu(inp, dev)
    s = inp.seq_starts()
    flat = lambda x: x.float().reshape(-1, x.shape[-1]).numpy()
    ch = w.Hk * w.dk
    cw = inp.conv_w.float().numpy()
    # intermediates are stored in fp16 for bf16/fp16 activations, fp32 for fp32
    rnd = torch.float32 if w.dtype == "fp32" else torch.float16
    as_act = lambda x: torch.from_numpy(x).to(rnd).double().numpy()
    q = O.l2norm(O.conv_silu(flat(inp.q_raw), cw[:ch], s), w.dk)
    k = O.l2norm(O.conv_silu(flat(inp.k_raw), cw[ch:2 * ch], s), w.dk)
    v = O.conv_silu(flat(inp.v_raw), cw[2 * ch:], s)
    tol = 1e-5 if w.dtype == "fp32" else 2.0 ** -9
    for name_, ref, hd, H in (("q", q, w.dk, w.Hk), ("k", k, w.dk, w.Hk), ("v", v, w.dv, w.Hv)):
        got = bufs.ws_view(name_).double().cpu().numpy()
        ref = ref.reshape(-1, H, hd).transpose(1, 0, 2)           # [H][ntok][d]
        if name_ == "v":                    # stored in the intermediate dtype
            err, bound = np.abs(got - as_act(ref)).max(), tol
        elif w.dtype == "fp32":
            err, bound = np.abs(got - ref).max(), 1e-5
        else:                               # fp16 hi + lo planes: about fp32 precision
            err, bound = np.abs(got[0] + got[1] - ref).max(), 2e-6
        print(f"[prologue] {name}: {name_} max abs {err:.3e}")
        assert err <= bound * max(1.0, np.abs(ref).max())
    beta, g = O.beta_decay(flat(inp.a), flat(inp.b), inp.A_log.numpy(), inp.dt_bias.numpy())
    gam = np.zeros_like(g)
    for s0, s1 in zip(s[:-1], s[1:]):
        for c0 in range(s0, s1, 64):
            gam[c0:min(c0 + 64, s1)] = np.cumsum(g[c0:min(c0 + 64, s1)], axis=0)
    gb = bufs.ws_view("beta").double().cpu().numpy().T
    gg = bufs.ws_view("gamma").double().cpu().numpy().T
    assert np.abs(gb - beta).max() <= 1e-6
    assert np.abs(gg - gam).max() <= 1e-5 * max(1.0, np.abs(gam).max())
