"""Pins of the oracle's decode step (CPU only).

A decode step is one more token of the forward recurrence, carried by a conv
cache (the raw inputs of the last width-1 tokens) and the state. So the
decode oracle is pinned to the forward oracle, itself pinned by closed forms
and brute force in test_oracle_pins.py:
  * decoding a sequence token by token from an empty cache reproduces the
    forward over the whole sequence, output by output, and its final state;
  * a forward over a prefix (prefill) followed by one decode step equals the
    forward over the prefix plus that token;
  * the cache that comes out is the raw inputs of the last tokens, exactly.
"""
import numpy as np
import pytest

from oracle import oracle as orc

W = 4


def problem(rng, N, T, Hk, Hv, dk, dv, init=True):
    ch = 2 * Hk * dk + Hv * dv
    f = lambda *s, sd=1.0: (rng.standard_normal(s) * sd).astype(np.float32)
    p = dict(
        q_raw=f(N, T, Hk * dk), k_raw=f(N, T, Hk * dk), v_raw=f(N, T, Hv * dv),
        a=f(N, T, Hv), b=f(N, T, Hv), gate=f(N, T, Hv * dv),
        conv_w=f(ch, W, sd=0.5), A_log=np.log(rng.uniform(1, 16, Hv)).astype(np.float32),
        dt_bias=f(Hv, sd=0.1), norm_w=(1 + f(dv, sd=0.1)).astype(np.float32),
        state=f(N, Hv, dk, dv, sd=0.1) if init else np.zeros((N, Hv, dk, dv), np.float32))
    return p


def forward(p, N, T, Hk, Hv, dk, dv, dtype):
    flat = lambda x: x.reshape(N * T, -1)
    return orc.forward(q_raw=flat(p["q_raw"]), k_raw=flat(p["k_raw"]), v_raw=flat(p["v_raw"]),
                       a=flat(p["a"]), b=flat(p["b"]), gate=flat(p["gate"]), conv_w=p["conv_w"],
                       A_log=p["A_log"], dt_bias=p["dt_bias"], norm_w=p["norm_w"],
                       seq_start=[n * T for n in range(N + 1)], Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                       dtype=dtype, initial_state=p["state"])


def step(p, t, cache, state, Hk, Hv, dk, dv, dtype):
    return orc.decode(q_raw=p["q_raw"][:, t], k_raw=p["k_raw"][:, t], v_raw=p["v_raw"][:, t],
                      a=p["a"][:, t], b=p["b"][:, t], gate=p["gate"][:, t], conv_w=p["conv_w"],
                      A_log=p["A_log"], dt_bias=p["dt_bias"], norm_w=p["norm_w"],
                      conv_state=cache, state=state, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype=dtype)


def raw_window(p, t_end, N, ch):
    """The raw inputs of tokens t_end-3 .. t_end-1 per channel, zero before 0."""
    x = np.concatenate([p["q_raw"], p["k_raw"], p["v_raw"]], axis=2)   # [N, T, ch]
    cache = np.zeros((N, ch, W - 1), np.float32)
    for r in range(W - 1):
        t = t_end - (W - 1) + r
        if t >= 0:
            cache[:, :, r] = x[:, t]
    return cache


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("Hk,Hv", [(2, 2), (2, 4)])
def test_decode_chain_equals_forward(dtype, Hk, Hv):
    rng = np.random.default_rng(7)
    N, T, dk, dv = 2, 9, 8, 16
    ch = 2 * Hk * dk + Hv * dv
    p = problem(rng, N, T, Hk, Hv, dk, dv)
    out_f, fin_f = forward(p, N, T, Hk, Hv, dk, dv, dtype)
    out_f = out_f.reshape(N, T, Hv, dv)
    cache = np.zeros((N, ch, W - 1), np.float32)
    state = p["state"]
    for t in range(T):
        out, cache64, state64 = step(p, t, cache, state, Hk, Hv, dk, dv, dtype)
        np.testing.assert_allclose(out, out_f[:, t], rtol=0, atol=1e-12)
        # the cache holds raw (already float32) values; the state stays in float64
        # in the forward, so carry the decode state at float64 precision too
        cache = cache64.astype(np.float32)
        np.testing.assert_array_equal(cache, raw_window(p, t + 1, N, ch))
        state = state64
    np.testing.assert_allclose(state, fin_f, rtol=0, atol=1e-12)


@pytest.mark.parametrize("T0", [1, 2, 5])
def test_prefill_then_decode(T0):
    rng = np.random.default_rng(11)
    N, Hk, Hv, dk, dv = 2, 1, 2, 16, 8
    ch = 2 * Hk * dk + Hv * dv
    p = problem(rng, N, T0 + 1, Hk, Hv, dk, dv)
    full_out, full_fin = forward(p, N, T0 + 1, Hk, Hv, dk, dv, "bf16")
    pre = {k: (v[:, :T0] if k in ("q_raw", "k_raw", "v_raw", "a", "b", "gate") else v) for k, v in p.items()}
    _, pre_fin = forward(pre, N, T0, Hk, Hv, dk, dv, "bf16")
    out, cache, state = step(p, T0, raw_window(p, T0, N, ch), pre_fin, Hk, Hv, dk, dv, "bf16")
    np.testing.assert_allclose(out, full_out.reshape(N, T0 + 1, Hv, dv)[:, T0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(state, full_fin, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(cache.astype(np.float32), raw_window(p, T0 + 1, N, ch))


def test_decode_with_zero_beta_only_decays():
    """b -> -inf gives beta = 0: the state only decays by exp(g) (closed form)."""
    rng = np.random.default_rng(3)
    N, Hk, Hv, dk, dv = 1, 1, 1, 4, 4
    ch = 2 * Hk * dk + Hv * dv
    p = problem(rng, N, 1, Hk, Hv, dk, dv)
    p["b"][:] = -200.0
    _, _, state = step(p, 0, np.zeros((N, ch, W - 1), np.float32), p["state"], Hk, Hv, dk, dv, "fp32")
    a, dtb, alog = float(p["a"][0, 0, 0]), float(p["dt_bias"][0]), float(p["A_log"][0])
    g = -np.exp(alog) * np.log1p(np.exp(a + dtb))
    np.testing.assert_allclose(state, np.exp(g) * p["state"].astype(np.float64), rtol=1e-12, atol=1e-15)
