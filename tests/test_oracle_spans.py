"""Pins of the oracle's conv-prefix option and of the span (affine state map)
decomposition that the sequence-sharded core rests on.

* A sequence continued from an earlier part reads the earlier part's last
  three raw tokens in its conv. The oracle's `conv_prefix` option must equal
  the plain forward over [prefix; sequence] in which the prefix tokens leave
  the state untouched (b = -inf gives beta = 0, a = -inf gives g = 0): the
  outputs of the sequence's tokens and the final state agree.
* For each span of a sequence the chunk recurrence is affine in the span's
  initial state: H_end = A H_start + B, where B is the span's final state from
  a zero state and A the final state of the same span with v = 0, dv = dk and
  the identity as initial state. Composing the spans' maps gives each span's
  true initial state; the spans' forwards from those states reproduce the
  whole sequence's outputs and final state.
"""
import numpy as np
import pytest

from oracle import oracle as O


def rnd(rng, shape, std=1.0):
    return (rng.normal(0.0, std, size=shape)).astype(np.float32)


def problem(seed, T, Hk, Hv, dk, dv, init=True):
    rng = np.random.default_rng(seed)
    ch = 2 * Hk * dk + Hv * dv
    P = dict(q_raw=rnd(rng, (T, Hk * dk)), k_raw=rnd(rng, (T, Hk * dk)), v_raw=rnd(rng, (T, Hv * dv)),
             a=rnd(rng, (T, Hv)), b=rnd(rng, (T, Hv)), gate=rnd(rng, (T, Hv * dv)),
             conv_w=rnd(rng, (ch, 4), 0.25),
             A_log=np.log(rng.uniform(1.0, 4.0, size=Hv)).astype(np.float32),
             dt_bias=rnd(rng, (Hv,), 0.1), norm_w=(1.0 + rnd(rng, (dv,), 0.1)).astype(np.float32))
    init_state = rnd(rng, (1, Hv, dk, dv), 0.3) if init else None
    return P, init_state, dict(Hk=Hk, Hv=Hv, dk=dk, dv=dv)


def fwd(P, meta, T, init=None, prefix=None, dtype="fp64"):
    return O.forward(**P, **meta, seq_start=[0, T], dtype=dtype, initial_state=init, conv_prefix=prefix)


def span_inputs(P, t0, t1):
    return {k: (v[t0:t1] if v.ndim == 2 and v.shape[0] >= t1 and k not in ("conv_w",) else v)
            for k, v in P.items()}


def raw_prefix(P, t0):
    """[1, 3, ch]: the raw q|k|v inputs of tokens t0-3 .. t0-1 (zeros before 0)."""
    x = np.concatenate([P["q_raw"], P["k_raw"], P["v_raw"]], axis=1)
    pre = np.zeros((1, 3, x.shape[1]), np.float32)
    for r in range(3):
        t = t0 - 3 + r
        if t >= 0:
            pre[0, r] = x[t]
    return pre


@pytest.mark.parametrize("T", [5, 70])
def test_prefix_equals_frozen_prefix_tokens(T):
    P, init, meta = problem(1, T, 1, 2, 8, 4)
    rng = np.random.default_rng(9)
    ch = 2 * meta["Hk"] * meta["dk"] + meta["Hv"] * meta["dv"]
    pre = rnd(rng, (1, 3, ch))
    out_p, fin_p = fwd(P, meta, T, init, prefix=pre)
    # the same tokens after three real tokens that neither write (beta = 0) nor decay (g = 0)
    q_ch = meta["Hk"] * meta["dk"]
    cat = dict(P)
    cat["q_raw"] = np.concatenate([pre[0, :, :q_ch], P["q_raw"]])
    cat["k_raw"] = np.concatenate([pre[0, :, q_ch:2 * q_ch], P["k_raw"]])
    cat["v_raw"] = np.concatenate([pre[0, :, 2 * q_ch:], P["v_raw"]])
    frozen = np.full((3, meta["Hv"]), -np.inf, np.float32)
    cat["a"] = np.concatenate([frozen, P["a"]])
    cat["b"] = np.concatenate([frozen, P["b"]])
    cat["gate"] = np.concatenate([np.zeros((3, P["gate"].shape[1]), np.float32), P["gate"]])
    out_c, fin_c = fwd(cat, meta, T + 3, init)
    np.testing.assert_allclose(out_p, out_c[3:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(fin_p, fin_c, rtol=0, atol=1e-12)


def test_prefix_none_is_zero_prefix():
    P, init, meta = problem(2, 9, 1, 1, 4, 4)
    ch = 2 * 4 + 4
    a, fa = fwd(P, meta, 9, init)
    b, fb = fwd(P, meta, 9, init, prefix=np.zeros((1, 3, ch), np.float32))
    assert np.array_equal(a, b) and np.array_equal(fa, fb)


def span_maps(P, meta, t0, t1):
    """(A [Hv, dk, dk], B [Hv, dk, dv]) of span [t0, t1): H_end = A H_start + B."""
    Hk, Hv, dk, dv = meta["Hk"], meta["Hv"], meta["dk"], meta["dv"]
    S = span_inputs(P, t0, t1)
    T = t1 - t0
    pre = raw_prefix(P, t0) if t0 > 0 else None
    _, B = fwd(S, meta, T, None, prefix=pre)
    # A: v = 0 (raw inputs and prefix), dv' = dk, identity initial state
    Z = dict(S)
    Z["v_raw"] = np.zeros((T, Hv * dk), np.float32)
    Z["gate"] = np.zeros((T, Hv * dk), np.float32)
    Z["norm_w"] = np.ones(dk, np.float32)
    cw = P["conv_w"]
    Z["conv_w"] = np.concatenate([cw[:2 * Hk * dk], np.zeros((Hv * dk, 4), np.float32)])
    preA = None
    if pre is not None:
        preA = np.concatenate([pre[:, :, :2 * Hk * dk], np.zeros((1, 3, Hv * dk), np.float32)], axis=2)
    eye = np.broadcast_to(np.eye(dk, dtype=np.float32), (1, Hv, dk, dk)).copy()
    _, A = fwd(Z, dict(meta, dv=dk), T, eye, prefix=preA)
    return A[0], B[0]


@pytest.mark.parametrize("cuts", [[0, 64, 128, 200], [0, 1, 70, 133, 200], [0, 100, 200]])
def test_span_composition_equals_whole_sequence(cuts):
    T = cuts[-1]
    P, init, meta = problem(3, T, 2, 4, 8, 6)
    out_full, fin_full = fwd(P, meta, T, init)
    H = init[0].astype(np.float64)
    outs = []
    for t0, t1 in zip(cuts[:-1], cuts[1:]):
        A, B = span_maps(P, meta, t0, t1)
        S = span_inputs(P, t0, t1)
        pre = raw_prefix(P, t0) if t0 > 0 else None
        o, f = fwd(S, meta, t1 - t0, H[None].astype(np.float32), prefix=pre)
        # the span's final state from H is the affine map applied to H (to the
        # float32 rounding of H that the forward takes as its initial state)
        Hf = H.astype(np.float32).astype(np.float64)
        np.testing.assert_allclose(f[0], np.einsum("hij,hjk->hik", A, Hf) + B, rtol=0, atol=1e-10)
        outs.append(o)
        H = f[0]
    np.testing.assert_allclose(np.concatenate(outs), out_full, rtol=0, atol=2e-6)
    np.testing.assert_allclose(H, fin_full[0], rtol=0, atol=2e-6)
