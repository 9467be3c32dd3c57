"""Pins of the CPU oracle against facts fixed by the definitions and by
mathematics: closed forms, brute force on tiny inputs, invariants and special
cases that reduce to library routines. None of these re-types the oracle's own
loop; each is chosen so that a plausible slip (a dropped term, a flipped sign,
a transposed operand, an off-by-one tap) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def silu(x):
    return x * scipy.special.expit(x)


# ------------------------------------------------------------------ rounding
@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
def test_round_act_matches_torch_conversion(dtype, tdt):
    # For values that are exact in float32 the direct double rounding must equal
    # torch's float32 -> bf16/fp16 round-to-nearest-even conversion.
    g = torch.Generator().manual_seed(1)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 3)
    x = torch.cat([x, torch.tensor([65504.0, 65519.0, 65520.0, -65520.0, 1e-8, 3e-5, 6.1e-5])])
    want = x.to(tdt).to(torch.float64).numpy()
    got = np.array([O.round_act(float(v), dtype) for v in x.tolist()])
    np.testing.assert_array_equal(got, want)


def test_round_act_ties_and_double_inputs():
    # ties go to the even significand
    assert O.round_act(1 + 2**-8, "bf16") == 1.0
    assert O.round_act(1 + 3 * 2**-8, "bf16") == 1 + 2**-6
    assert O.round_act(1 + 2**-11, "fp16") == 1.0
    # a double just above a bf16 tie rounds up (rounding via float32 first would not)
    assert O.round_act(1 + 2**-8 + 2**-40, "bf16") == 1 + 2**-7
    assert O.round_act(65520.0, "fp16") == math.inf
    assert O.round_act(0.1, "fp32") == float(np.float32(0.1))


# ---------------------------------------------------------------------- conv
def test_conv_identity_and_shift_taps():
    rng = np.random.default_rng(0)
    T, C = 11, 5
    x = rng.standard_normal((T, C)).astype(np.float32)
    w = np.zeros((C, 4), np.float32)
    w[:, 3] = 1.0   # tap 3 multiplies the current token
    y = O.conv_silu(x, w, [0, T])
    np.testing.assert_allclose(y, silu(x.astype(np.float64)), rtol=1e-15)
    w[:] = 0.0
    w[:, 0] = 1.0   # tap 0 multiplies the token three steps back; zero halo
    y = O.conv_silu(x, w, [0, T])
    want = np.zeros((T, C))
    want[3:] = silu(x[:-3].astype(np.float64))
    np.testing.assert_allclose(y, want, rtol=1e-15)


def test_conv_matches_numpy_convolve_with_sequence_resets():
    rng = np.random.default_rng(1)
    starts = [0, 2, 9, 10, 23]   # sequences of length 2, 7, 1, 13
    C = 6
    x = rng.standard_normal((starts[-1], C)).astype(np.float32)
    w = rng.standard_normal((C, 4)).astype(np.float32)
    y = O.conv_silu(x, w, starts)
    want = np.zeros_like(y)
    for s0, s1 in zip(starts[:-1], starts[1:]):
        for c in range(C):
            full = np.convolve(x[s0:s1, c].astype(np.float64), w[c, ::-1].astype(np.float64))
            want[s0:s1, c] = silu(full[: s1 - s0])
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-15)


def test_concatenated_conv_equals_separate_convs_bitwise():
    # "fused q/k/v short conv": one depthwise conv over [q;k;v] channels equals
    # three convs because nothing mixes channels.
    rng = np.random.default_rng(2)
    T = 37
    xq, xk, xv = (rng.standard_normal((T, n)).astype(np.float32) for n in (8, 8, 16))
    wq, wk, wv = (rng.standard_normal((n, 4)).astype(np.float32) for n in (8, 8, 16))
    s = [0, 20, 37]
    cat = O.conv_silu(np.concatenate([xq, xk, xv], 1), np.concatenate([wq, wk, wv], 0), s)
    sep = np.concatenate([O.conv_silu(xq, wq, s), O.conv_silu(xk, wk, s),
                          O.conv_silu(xv, wv, s)], 1)
    assert np.array_equal(cat, sep)


# ------------------------------------------------------------------- l2 norm
def test_l2norm_closed_form_and_unit_norm():
    x = np.array([[3.0, 4.0]])
    y = O.l2norm(x, 2, eps=1e-6)
    np.testing.assert_allclose(y, [[3 / math.sqrt(25 + 1e-6), 4 / math.sqrt(25 + 1e-6)]],
                               rtol=1e-15)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 3 * 16))
    y = O.l2norm(x, 16, eps=1e-6).reshape(50, 3, 16)
    ss = (x.reshape(50, 3, 16) ** 2).sum(-1)
    np.testing.assert_allclose((y ** 2).sum(-1), ss / (ss + 1e-6), rtol=1e-13)


def test_l2norm_commutes_with_head_replication():
    # "fold q/k L2-norm...", section "Why": normalisation is per head, so GQA
    # replication before or after it gives the same result.
    rng = np.random.default_rng(4)
    x = rng.standard_normal((9, 2 * 8))
    rep = np.repeat(x.reshape(9, 2, 8), 3, axis=1).reshape(9, 6 * 8)
    a = np.repeat(O.l2norm(x, 8).reshape(9, 2, 8), 3, axis=1).reshape(9, 48)
    b = O.l2norm(rep, 8)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- beta, g
def test_beta_decay_closed_forms():
    a = np.array([[0.0, 3.0, -40.0, 40.0]], np.float32)
    b = np.array([[0.0, 2.0, -1.0, 5.0]], np.float32)
    A_log = np.array([0.0, math.log(4.0), 0.5, 1.0], np.float32)
    dt = np.array([0.0, -1.0, 0.0, 0.25], np.float32)
    beta, g = O.beta_decay(a, b, A_log, dt)
    np.testing.assert_allclose(beta[0], scipy.special.expit(b[0].astype(np.float64)), rtol=1e-15)
    assert beta[0, 0] == 0.5
    assert abs(g[0, 0] + math.log(2.0)) < 1e-15          # -e^0 * log(1 + e^0)
    want = -np.exp(A_log.astype(np.float64)) * np.logaddexp(0.0, (a[0] + dt).astype(np.float64))
    np.testing.assert_allclose(g[0], want, rtol=1e-14)
    assert g[0, 3] < 0 and abs(g[0, 3] / (-math.e * 40.25) - 1) < 1e-15


def test_golden_closed_forms():
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        kind = case["kind"]
        if kind == "silu_tap3":
            y = O.conv_silu(np.array([[case["x"]]], np.float32),
                            np.array([[0, 0, 0, 1]], np.float32), [0, 1])
            assert abs(y[0, 0] - case["want"]) < 1e-15
        elif kind == "beta_decay":
            beta, g = O.beta_decay(np.array([[case["a"]]], np.float32),
                                   np.array([[case["b"]]], np.float32),
                                   np.array([case["A_log"]], np.float32),
                                   np.array([case["dt_bias"]], np.float32))
            assert abs(beta[0, 0] - case["beta"]) < 1e-15
            assert abs(g[0, 0] - case["g"]) < 1e-15
        elif kind == "gated_rmsnorm_const":
            dv = case["dv"]
            o = np.full((1, dv), case["o"])
            y = O.gated_rmsnorm(o, np.full((1, dv), case["gate"], np.float32),
                                np.full(dv, case["norm_w"], np.float32), eps=case["eps"],
                                dtype="fp32")
            np.testing.assert_allclose(y[0], case["want"], rtol=1e-7)
        else:
            raise AssertionError(kind)


# ------------------------------------------------------------- delta rule
def _unit_rows(rng, T, d):
    x = rng.standard_normal((T, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def test_delta_rule_beta_zero_is_pure_decay():
    rng = np.random.default_rng(5)
    T, dk, dv = 13, 4, 3
    q = rng.standard_normal((T, dk))
    k = _unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    g = -rng.uniform(0.0, 0.2, T)
    h0 = rng.standard_normal((dk, dv))
    o, hT = O.delta_rule(q, k, v, np.zeros(T), g, h0=h0)
    gam = np.cumsum(g)
    for t in range(T):
        np.testing.assert_allclose(o[t], math.exp(gam[t]) * (h0.T @ q[t]), rtol=1e-13)
    np.testing.assert_allclose(hT, math.exp(gam[-1]) * h0, rtol=1e-13)


def test_state_layout_is_transposed_S():
    # initial state is stored as H = S^T [dk, dv]: with H = e_a e_b^T,
    # o = S q has a single non-zero entry o[b] = q[a]
    dk, dv = 5, 3
    h0 = np.zeros((dk, dv))
    h0[4, 1] = 1.0
    q = np.arange(1.0, dk + 1.0)[None, :]
    o, hT = O.delta_rule(q, np.eye(dk)[:1], np.zeros((1, dv)), [0.0], [0.0], h0=h0)
    np.testing.assert_array_equal(o[0], [0.0, 5.0, 0.0])
    np.testing.assert_array_equal(hT, h0)


def test_delta_rule_write_then_read_returns_value():
    # beta = 1, g = 0: S_t k_t = S_{t-1}(k_t - k_t) + v_t = v_t, so a query equal
    # to the key just written reads back exactly its value (o uses S_t).
    rng = np.random.default_rng(6)
    T, dk, dv = 20, 6, 4
    k = _unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    o, _ = O.delta_rule(k, k, v, np.ones(T), np.zeros(T), h0=rng.standard_normal((dk, dv)))
    np.testing.assert_allclose(o, v, rtol=1e-12, atol=1e-12)


def test_delta_rule_orthonormal_keys_retrieve_all_values():
    rng = np.random.default_rng(7)
    dk, dv, T = 8, 5, 6
    Q, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Q[:T]
    v = rng.standard_normal((T, dv))
    _, hT = O.delta_rule(np.zeros((T, dk)), k, v, np.ones(T), np.zeros(T))
    S = hT.T
    for i in range(T):
        np.testing.assert_allclose(S @ k[i], v[i], rtol=1e-12, atol=1e-13)
    # a direction orthogonal to every written key reads zero
    np.testing.assert_allclose(S @ Q[T], 0.0, atol=1e-13)


def test_delta_rule_scalar_geometric_closed_form():
    # dk = dv = 1, k = 1, constant beta, g, v: S_t = a S_{t-1} + c with
    # a = e^g (1 - beta), c = beta v, so S_t = a^t S_0 + c (1 - a^t) / (1 - a).
    T, beta, g, v, s0, qv = 17, 0.3, -0.2, 1.7, -0.4, 2.5
    a = math.exp(g) * (1 - beta)
    c = beta * v
    o, hT = O.delta_rule(np.full((T, 1), qv), np.ones((T, 1)), np.full((T, 1), v),
                         np.full(T, beta), np.full(T, g), h0=np.array([[s0]]))
    for t in range(1, T + 1):
        st = a**t * s0 + c * (1 - a**t) / (1 - a)
        assert abs(o[t - 1, 0] - qv * st) < 1e-13
    assert abs(hT[0, 0] - (a**T * s0 + c * (1 - a**T) / (1 - a))) < 1e-13


def test_delta_rule_brute_force_unrolled_products():
    # S_t = S_0 M_1...M_t + sum_u beta_u v_u k_u^T M_{u+1}...M_t with
    # M_u = e^{g_u} (I - beta_u k_u k_u^T), evaluated with explicit dk x dk
    # matrices (a different order of operations from the token loop).
    rng = np.random.default_rng(8)
    T, dk, dv = 6, 3, 2
    q = rng.standard_normal((T, dk))
    k = _unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    beta = rng.uniform(0.1, 0.9, T)
    g = -rng.uniform(0.0, 1.0, T)
    S0 = rng.standard_normal((dv, dk))
    o, hT = O.delta_rule(q, k, v, beta, g, h0=S0.T, scale=0.5)
    M = [math.exp(g[u]) * (np.eye(dk) - beta[u] * np.outer(k[u], k[u])) for u in range(T)]

    def prod(lo, hi):
        P = np.eye(dk)
        for u in range(lo, hi):
            P = P @ M[u]
        return P

    for t in range(T):
        St = S0 @ prod(0, t + 1)
        for u in range(t + 1):
            St = St + beta[u] * np.outer(v[u], k[u]) @ prod(u + 1, t + 1)
        np.testing.assert_allclose(o[t], 0.5 * St @ q[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT, St.T, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("C", [64, 16, 7, 1])
@pytest.mark.parametrize("decay", ["mild", "strong"])
def test_chunked_variant_equals_token_loop(C, decay):
    rng = np.random.default_rng(9)
    T, dk, dv = 150, 16, 8
    q = _unit_rows(rng, T, dk)
    k = _unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    beta = scipy.special.expit(rng.standard_normal(T))
    if decay == "mild":
        g = -rng.uniform(0.0, 0.1, T)
    else:  # the workload's scale: g ~ -A softplus(N(0,1)), A in [1, 16]
        g = -16.0 * np.logaddexp(0.0, rng.standard_normal(T))
    h0 = rng.standard_normal((dk, dv))
    o1, h1 = O.delta_rule(q, k, v, beta, g, h0=h0)
    o2, h2 = O.delta_rule(q, k, v, beta, g, h0=h0, chunk=C)
    np.testing.assert_allclose(o2, o1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(h2, h1, rtol=1e-10, atol=1e-12)


def test_delta_rule_scale_is_linear_in_output_only():
    rng = np.random.default_rng(10)
    T, dk, dv = 9, 4, 3
    args = (rng.standard_normal((T, dk)), _unit_rows(rng, T, dk), rng.standard_normal((T, dv)),
            rng.uniform(0, 1, T), -rng.uniform(0, 1, T))
    o1, h1 = O.delta_rule(*args)
    o2, h2 = O.delta_rule(*args, scale=0.125)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-15)
    np.testing.assert_array_equal(h1, h2)


# ----------------------------------------------------------- gated rmsnorm
def test_gated_rmsnorm_closed_forms():
    dv = 8
    o = np.full((1, dv), 0.5)
    nw = np.linspace(0.5, 1.5, dv).astype(np.float32)
    gate = np.full((1, dv), 1.0, np.float32)
    y = O.gated_rmsnorm(o, gate, nw, eps=1e-5, dtype="fp32")
    r = 0.5 / math.sqrt(0.25 + 1e-5)
    want = [float(np.float32(w * r)) * silu(1.0) for w in nw.astype(np.float64)]
    np.testing.assert_allclose(y[0], want, rtol=1e-15)
    # silu(0) = 0 zeroes the output whatever o is
    y = O.gated_rmsnorm(np.random.default_rng(0).standard_normal((3, dv)),
                        np.zeros((3, dv), np.float32), nw, dtype="bf16")
    assert np.all(y == 0.0)


def test_gated_rmsnorm_rounds_normed_value_to_act_dtype():
    # the RMSNorm result is materialised in the activation dtype before the
    # fp32 gating multiply ("GDN Elementwise Fusion", numerical behaviour)
    o = np.array([[1.0, 3.0]])           # mean(o^2) = 5
    nw = np.array([1.0, 1.0], np.float32)
    gate = np.array([[2.0, 2.0]], np.float32)
    y = O.gated_rmsnorm(o, gate, nw, eps=0.0, dtype="bf16")
    r = np.array([1 / math.sqrt(5), 3 / math.sqrt(5)])
    rb = torch.tensor(r, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert not np.array_equal(rb, r)
    np.testing.assert_allclose(y[0], rb * silu(2.0), rtol=1e-15)
