"""Pins of the oracle backward (oracle/gdn_oracle_bwd.c) against the forward.

The pages define the forward only, so the backward is pinned by what the
mathematics fixes: the gradient of L = sum(grad_out * out) + sum(grad_final *
final_state) must equal the finite-difference derivative of the pinned oracle
forward (its real-valued form, act "fp64"), for every input element of a tiny
packed GQA problem and along random directions of a longer one whose
sequences cross the backward's 64-token checkpoints.

Inputs lie on a dyadic grid and the steps are powers of two, so every
perturbed input is exact in float32 and the 4-point central difference
(error O(h^4)) is limited only by double rounding.
"""
import numpy as np
import pytest

from oracle import oracle as O

H = 2.0 ** -15


def dyadic(rng, shape, std=1.0, q=64):
    return (np.round(rng.normal(0.0, std, size=shape) * q) / q).astype(np.float32)


def make_problem(seed, lens, Hk, Hv, dk, dv, init=True, gfin=True):
    rng = np.random.default_rng(seed)
    ntok = int(sum(lens))
    ch = 2 * Hk * dk + Hv * dv
    P = dict(q_raw=dyadic(rng, (ntok, Hk * dk)), k_raw=dyadic(rng, (ntok, Hk * dk)),
             v_raw=dyadic(rng, (ntok, Hv * dv)), a=dyadic(rng, (ntok, Hv)), b=dyadic(rng, (ntok, Hv)),
             gate=dyadic(rng, (ntok, Hv * dv)), conv_w=dyadic(rng, (ch, 4), 0.5),
             A_log=dyadic(rng, (Hv,), 0.5), dt_bias=dyadic(rng, (Hv,), 0.25),
             norm_w=(1.0 + dyadic(rng, (dv,), 0.25)).astype(np.float32))
    if init:
        P["initial_state"] = dyadic(rng, (len(lens), Hv, dk, dv), 0.5)
    G = dict(grad_out=dyadic(rng, (ntok, Hv, dv)),
             grad_final=dyadic(rng, (len(lens), Hv, dk, dv)) if gfin else None)
    meta = dict(seq_start=np.concatenate([[0], np.cumsum(lens)]), Hk=Hk, Hv=Hv, dk=dk, dv=dv, scale=0.75)
    return P, G, meta


def loss(P, G, meta):
    out, fin = O.forward(**P, **meta, dtype="fp64")
    L = float(np.sum(out * G["grad_out"].astype(np.float64)))
    if G["grad_final"] is not None:
        L += float(np.sum(fin * G["grad_final"].astype(np.float64)))
    return L


def fd(P, G, meta, name, direction):
    """4-point central difference of the loss along ``direction`` of input ``name``."""
    base = P[name]
    vals = {}
    for m in (-2, -1, 1, 2):
        Q = dict(P)
        Q[name] = (base.astype(np.float64) + m * H * direction).astype(np.float32)
        assert np.array_equal(Q[name].astype(np.float64), base.astype(np.float64) + m * H * direction)
        vals[m] = loss(Q, G, meta)
    return (8.0 * (vals[1] - vals[-1]) - (vals[2] - vals[-2])) / (12.0 * H)


GRAD_OF = dict(q_raw="dq_raw", k_raw="dk_raw", v_raw="dv_raw", a="da", b="db", gate="dgate",
               conv_w="dconv_w", A_log="dA_log", dt_bias="ddt_bias", norm_w="dnorm_w",
               initial_state="dinitial_state")


@pytest.mark.parametrize("init,gfin", [(True, True), (False, False)])
def test_backward_matches_elementwise_finite_differences(init, gfin):
    """Every element of every input: two packed sequences (3 and 5 tokens),
    GQA 1 -> 2 heads, dk = 3, dv = 2, scale 0.75."""
    P, G, meta = make_problem(1, [3, 5], 1, 2, 3, 2, init, gfin)
    grads = O.backward(**P, **G, **meta)
    worst = 0.0
    for name, gname in GRAD_OF.items():
        if name not in P:
            continue
        an = np.asarray(grads[gname]).reshape(-1)
        for idx in range(P[name].size):
            e = np.zeros(P[name].size)
            e[idx] = 1.0
            num = fd(P, G, meta, name, e.reshape(P[name].shape))
            err = abs(num - an[idx]) / (1.0 + abs(an[idx]))
            worst = max(worst, err)
            assert err < 1e-9, f"{gname}[{idx}]: backward {an[idx]!r} vs finite difference {num!r}"
    assert worst < 1e-9


def test_backward_directional_long_sequences():
    """Random directions of every input on sequences of 150 and 70 tokens
    (crossing the 64-token checkpoints), GQA 2 -> 4 heads, dk = 4, dv = 3."""
    P, G, meta = make_problem(2, [150, 70], 2, 4, 4, 3)
    grads = O.backward(**P, **G, **meta, threads=2)
    rng = np.random.default_rng(7)
    for name, gname in GRAD_OF.items():
        d = np.round(rng.normal(size=P[name].shape) * 4) / 4
        num = fd(P, G, meta, name, d)
        an = float(np.sum(np.asarray(grads[gname]) * d))
        assert abs(num - an) <= 1e-9 * (1.0 + abs(an)), f"{gname}: backward {an!r} vs finite difference {num!r}"


def test_backward_zero_cotangent_gives_zero_gradients():
    P, G, meta = make_problem(3, [9], 1, 1, 2, 2)
    G = dict(grad_out=np.zeros_like(G["grad_out"]), grad_final=None)
    grads = O.backward(**P, **G, **meta)
    for g in grads.values():
        assert not np.any(g)


def test_backward_state_only_cotangent():
    """With grad_out = 0 only the state path carries gradient: the gate and
    norm weight receive none, the initial state receives exp(sum g)-decayed
    terms (checked against the finite difference above), and v does."""
    P, G, meta = make_problem(4, [6], 1, 1, 2, 2)
    G = dict(grad_out=np.zeros_like(G["grad_out"]), grad_final=G["grad_final"])
    grads = O.backward(**P, **G, **meta)
    assert not np.any(grads["dgate"]) and not np.any(grads["dnorm_w"])
    assert np.any(grads["dv_raw"]) and np.any(grads["dinitial_state"])
    d = np.ones(P["v_raw"].shape)
    assert abs(fd(P, G, meta, "v_raw", d) - grads["dv_raw"].sum()) <= 1e-9 * (1 + abs(grads["dv_raw"].sum()))
