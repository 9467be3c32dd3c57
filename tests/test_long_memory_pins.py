"""Why the long-memory GPU cases exist: a mistake planted in the oracle's chunk
hand-off is caught by the mild-decay recipe and missed by the workloads'.

The forward is recomputed chunk by chunk from the oracle's pinned steps (conv +
SiLU, L2 norm, beta and decay, the token loop over one chunk at a time with
the state handed from chunk to chunk, the gated RMSNorm). Unchanged, that chain
equals the oracle forward. The planted mistake drops the decayed carry
exp(gamma_C) H_{c-1} from each chunk's state update (the chunk's own readout
still sees H_{c-1}), the kind of error a kernel's state pass could make. With
A_log = log U[1, 16] the decay over a chunk is below 1e-20, so the mistake
stays inside the bf16 tolerance; with the mild recipe it fails it.
"""
import numpy as np
import pytest

from linear_attention_sequence_qkv_gb300.workloads import MILD, WORKLOADS, make_inputs, replace
from oracle import oracle as O
from tests._harness import check, chunk_survival, flat, oracle_forward

C = 64


def chunked_forward(inp, drop_decayed_carry=False):
    w = inp.w
    s = inp.seq_starts()
    ch = w.Hk * w.dk
    cw = inp.conv_w.float().numpy()
    q = O.l2norm(O.conv_silu(flat(inp.q_raw), cw[:ch], s), w.dk)
    k = O.l2norm(O.conv_silu(flat(inp.k_raw), cw[ch:2 * ch], s), w.dk)
    v = O.conv_silu(flat(inp.v_raw), cw[2 * ch:], s)
    beta, g = O.beta_decay(flat(inp.a), flat(inp.b), inp.A_log.numpy(), inp.dt_bias.numpy())
    ntok = s[-1]
    o = np.zeros((ntok, w.Hv, w.dv))
    fin = np.zeros((len(s) - 1, w.Hv, w.dk, w.dv))
    G = w.Hv // w.Hk
    for n, (s0, s1) in enumerate(zip(s[:-1], s[1:])):
        for h in range(w.Hv):
            hk = h // G
            H = (inp.initial_state[n, h].double().numpy() if inp.initial_state is not None
                 else np.zeros((w.dk, w.dv)))
            for c0 in range(s0, s1, C):
                c1 = min(c0 + C, s1)
                qk = slice(hk * w.dk, (hk + 1) * w.dk)
                oc, H1 = O.delta_rule(q[c0:c1, qk], k[c0:c1, qk], v[c0:c1, h * w.dv:(h + 1) * w.dv],
                                      beta[c0:c1, h], g[c0:c1, h], h0=H)
                if drop_decayed_carry:
                    H1 = H1 - np.exp(g[c0:c1, h].sum()) * H
                o[c0:c1, h] = oc
                H = H1
            fin[n, h] = H
    gate = flat(inp.gate.contiguous())
    out = O.gated_rmsnorm(o.reshape(-1, w.dv), gate.reshape(-1, w.dv), inp.norm_w.float().numpy(),
                          dtype=w.dtype)
    return out.reshape(ntok, w.Hv, w.dv), fin


def case(decay_range):
    w = replace(WORKLOADS["layer_bf16"], B=2, T=8 * C + 11, Hk=1, Hv=2, dk=32, dv=32, init_state_std=0.1,
                decay_range=decay_range)
    return make_inputs(w)


@pytest.mark.parametrize("decay_range", [MILD, (1.0, 16.0)], ids=["mild", "workloads"])
def test_chunk_chain_equals_oracle_forward(decay_range):
    inp = case(decay_range)
    out, fin = chunked_forward(inp)
    ref_out, ref_fin = oracle_forward(inp)
    # the same steps in the same order up to the chunk hand-off: rounding-level agreement,
    # except where the RMSNorm's rounding to bf16 sits on a tie boundary
    assert np.abs(fin - ref_fin).max() < 1e-9
    assert np.mean(np.abs(out - ref_out) > 1e-9) < 1e-3


def test_mild_recipe_sees_the_dropped_carry():
    inp = case(MILD)
    assert chunk_survival(inp) >= 0.5
    ref_out, ref_fin = oracle_forward(inp)
    out, fin = chunked_forward(inp, drop_decayed_carry=True)
    with pytest.raises(AssertionError):
        check(fin, ref_fin, "bf16", "planted mistake final_state")
    with pytest.raises(AssertionError):
        check(out, ref_out, "bf16", "planted mistake out")


def test_workload_recipe_misses_the_dropped_carry():
    inp = case((1.0, 16.0))
    assert chunk_survival(inp) == 0.0
    ref_out, ref_fin = oracle_forward(inp)
    out, fin = chunked_forward(inp, drop_decayed_carry=True)
    check(fin, ref_fin, "bf16", "planted mistake (strong decay) final_state")
    check(out, ref_out, "bf16", "planted mistake (strong decay) out")
