"""Pins of the oracle's whole core forward: its wiring of the pinned steps
(channel and weight offsets, GQA mapping, per-head indexing), causality,
state hand-off between calls, packed sequences and the chunked variant."""
import numpy as np
import pytest

from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, make_inputs, replace
from oracle import oracle as O


def flat(x):
    x = x.float()
    return x.reshape(-1, x.shape[-1]).numpy()


def run(inp, **kw):
    w = inp.w
    return O.forward(q_raw=flat(inp.q_raw), k_raw=flat(inp.k_raw), v_raw=flat(inp.v_raw),
                     a=flat(inp.a), b=flat(inp.b), gate=flat(inp.gate.contiguous()),
                     conv_w=inp.conv_w.float().numpy(), A_log=inp.A_log.numpy(),
                     dt_bias=inp.dt_bias.numpy(), norm_w=inp.norm_w.float().numpy(),
                     seq_start=inp.seq_starts(), Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv,
                     dtype=w.dtype,
                     initial_state=None if inp.initial_state is None else inp.initial_state.numpy(),
                     **kw)


SMALL = replace(WORKLOADS["ragged_fp16"], B=2, T=45, Hk=2, Hv=4, dk=8, dv=4,
                gate_extra=3, init_state_std=0.1)


def test_forward_is_the_composition_of_its_steps():
    inp = make_inputs(SMALL)
    w = inp.w
    out, fin = run(inp)
    s = inp.seq_starts()
    ch = w.Hk * w.dk
    cw = inp.conv_w.float().numpy()
    xq = O.conv_silu(flat(inp.q_raw), cw[:ch], s)
    xk = O.conv_silu(flat(inp.k_raw), cw[ch:2 * ch], s)
    xv = O.conv_silu(flat(inp.v_raw), cw[2 * ch:], s)
    q = O.l2norm(xq, w.dk)
    k = O.l2norm(xk, w.dk)
    beta, g = O.beta_decay(flat(inp.a), flat(inp.b), inp.A_log.numpy(), inp.dt_bias.numpy())
    gate = flat(inp.gate.contiguous())
    for h in range(w.Hv):
        hk = h // w.G
        o = np.zeros((s[-1], w.dv))
        for n in range(len(s) - 1):
            sl = slice(s[n], s[n + 1])
            ob, hT = O.delta_rule(q[sl, hk * w.dk:(hk + 1) * w.dk], k[sl, hk * w.dk:(hk + 1) * w.dk],
                                  xv[sl, h * w.dv:(h + 1) * w.dv], beta[sl, h], g[sl, h],
                                  h0=inp.initial_state[n, h].numpy().astype(np.float64))
            o[sl] = ob
            np.testing.assert_array_equal(fin[n, h], hT)
        y = O.gated_rmsnorm(o, gate[:, h * w.dv:(h + 1) * w.dv], inp.norm_w.float().numpy(),
                            dtype=w.dtype)
        np.testing.assert_array_equal(out[:, h], y)


def test_causal_prefix():
    w = replace(SMALL, B=1, T=128, init_state_std=0.0)
    inp = make_inputs(w)
    out, _ = run(inp)
    short = make_inputs(w)
    for name in ("q_raw", "k_raw", "v_raw", "a", "b", "gate_buf"):
        setattr(short, name, getattr(inp, name)[:, :100].contiguous())
    short.w = replace(w, T=100)
    out100, _ = run(short)
    np.testing.assert_array_equal(out100, out[:100])


def test_state_handoff_between_calls():
    # with an identity conv (one-hot current tap) the conv carries no memory, so
    # chaining final_state -> initial_state over two calls equals one call
    w = replace(SMALL, B=1, T=90, init_state_std=0.1)
    inp = make_inputs(w)
    cw = np.zeros(tuple(inp.conv_w.shape), np.float32)
    cw[:, 3] = 1.0
    import torch
    inp.conv_w = torch.from_numpy(cw)
    out, fin = run(inp)
    a = make_inputs(w)
    b = make_inputs(w)
    for part, sl in ((a, slice(0, 37)), (b, slice(37, 90))):
        for name in ("q_raw", "k_raw", "v_raw", "a", "b", "gate_buf"):
            setattr(part, name, getattr(inp, name)[:, sl].contiguous())
        part.conv_w = inp.conv_w
        part.w = replace(w, T=sl.stop - sl.start)
    out_a, fin_a = run(a)
    b.initial_state = torch.from_numpy(fin_a.astype(np.float32))
    out_b, fin_b = run(b)
    # fin_a passes through float32 between the calls
    np.testing.assert_allclose(out_a, out[:37], rtol=0, atol=0)
    np.testing.assert_allclose(out_b, out[37:], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(fin_b, fin, rtol=1e-6, atol=1e-7)


def test_packed_sequences_equal_separate_runs():
    lengths = [5, 1, 64, 70]
    w = replace(SMALL, B=1, T=0, n_packed=len(lengths), init_state_std=0.1)
    inp = make_inputs(w, lengths=lengths)
    out, fin = run(inp)
    s = inp.seq_starts()
    for n, L in enumerate(lengths):
        one = make_inputs(replace(w, T=L, n_packed=0))
        for name in ("q_raw", "k_raw", "v_raw", "a", "b", "gate_buf"):
            setattr(one, name, getattr(inp, name)[:, s[n]:s[n + 1]].contiguous())
        for name in ("conv_w", "A_log", "dt_bias", "norm_w"):
            setattr(one, name, getattr(inp, name))
        one.initial_state = inp.initial_state[n:n + 1]
        o1, f1 = run(one)
        np.testing.assert_array_equal(o1, out[s[n]:s[n + 1]])
        np.testing.assert_array_equal(f1[0], fin[n])


def test_empty_sequences_keep_their_initial_state():
    # a sequence without tokens applies no step of the recurrence: its final state is
    # its initial state, and the sequences around it are as if it were not there
    lengths = [0, 9, 0, 0, 70, 0]
    w = replace(SMALL, B=1, T=0, n_packed=len(lengths), init_state_std=0.1)
    inp = make_inputs(w, lengths=lengths)
    out, fin = run(inp)
    assert out.shape[0] == sum(lengths)
    h0 = inp.initial_state.numpy()
    for n, L in enumerate(lengths):
        if L == 0:
            np.testing.assert_array_equal(fin[n], h0[n])
    keep = [n for n, L in enumerate(lengths) if L > 0]
    dense = make_inputs(replace(w, n_packed=len(keep)), lengths=[lengths[n] for n in keep])
    for name in ("q_raw", "k_raw", "v_raw", "a", "b", "gate_buf", "conv_w", "A_log", "dt_bias", "norm_w"):
        setattr(dense, name, getattr(inp, name))
    dense.initial_state = inp.initial_state[keep]
    out2, fin2 = run(dense)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(fin[keep], fin2)


def test_gqa_equals_explicit_head_replication():
    import torch
    w = replace(SMALL, Hk=2, Hv=4)
    inp = make_inputs(w)
    out, fin = run(inp)
    rep = make_inputs(replace(w, Hk=4))
    G = 2
    B, T = inp.q_raw.shape[:2]
    for name in ("q_raw", "k_raw"):
        x = getattr(inp, name).reshape(B, T, 2, w.dk)
        setattr(rep, name, x.repeat_interleave(G, dim=2).reshape(B, T, 4 * w.dk))
    ch = 2 * w.dk
    cq = inp.conv_w[:ch].reshape(2, w.dk, 4).repeat_interleave(G, 0).reshape(-1, 4)
    ck = inp.conv_w[ch:2 * ch].reshape(2, w.dk, 4).repeat_interleave(G, 0).reshape(-1, 4)
    rep.conv_w = torch.cat([cq, ck, inp.conv_w[2 * ch:]], 0)
    for name in ("v_raw", "a", "b", "gate_buf", "A_log", "dt_bias", "norm_w", "initial_state"):
        setattr(rep, name, getattr(inp, name))
    out2, fin2 = run(rep)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(fin, fin2)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_forward_chunked_variant_matches_token_loop(dtype):
    w = replace(SMALL, dtype=dtype, T=150, dk=16, dv=8)
    inp = make_inputs(w)
    o1, f1 = run(inp)
    o2, f2 = run(inp, chunked=64)
    np.testing.assert_allclose(f2, f1, rtol=1e-9, atol=1e-12)
    # outputs agree except where the act-dtype rounding of the normed value
    # lands on the other side of a tie by ~1e-15
    close = np.isclose(o2, o1, rtol=1e-9, atol=1e-12)
    assert close.mean() > 0.999
