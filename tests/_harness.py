"""Shared helpers of the GPU parity tests: oracle runs on the same seeded,
already-rounded inputs, and the tolerance checks."""
import numpy as np

from oracle import oracle as O


def flat(x):
    x = x.float()
    return x.reshape(-1, x.shape[-1]).numpy()


def oracle_forward(inp, threads=8, **kw):
    w = inp.w
    return O.forward(q_raw=flat(inp.q_raw), k_raw=flat(inp.k_raw), v_raw=flat(inp.v_raw),
                     a=flat(inp.a), b=flat(inp.b), gate=flat(inp.gate.contiguous()),
                     conv_w=inp.conv_w.float().numpy(), A_log=inp.A_log.numpy(),
                     dt_bias=inp.dt_bias.numpy(), norm_w=inp.norm_w.float().numpy(),
                     seq_start=inp.seq_starts(), Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv,
                     dtype=w.dtype,
                     initial_state=None if inp.initial_state is None else inp.initial_state.numpy(),
                     threads=threads, **kw)


def errors(got, ref):
    """(max |d| / max(1, |ref|), relative L2) of got against the oracle."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    scaled = float((d / np.maximum(1.0, np.abs(ref))).max()) if d.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return scaled, rel


# mantissa bits of the 2-byte activation dtypes
ULP_BITS = {"bf16": 7, "fp16": 10}


def ulp_act(x, dtype):
    """Spacing of the act dtype's numbers at |x| (normal range; the 3e-2 floor
    of the bound dominates long before the subnormals)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(ax)) - ULP_BITS[dtype])


def check(got, ref, dtype, what, kind=None):
    """Tolerances of the GDN core.

    fp32: max |d| <= 1e-4 max(1, |ref|).
    bf16/fp16: relative L2 <= 5e-3; every |d| <= 3e-2, except that an output
    in the act dtype may be off by up to three units in the last place of that
    dtype where that exceeds 3e-2 (|ref| >= 2 in bf16); the count of elements
    beyond 3e-2 is printed beside the raw max |d|. The three ulps: both sides round the RMSNorm result
    to the act dtype before the gating multiply, and two nearly equal values
    can round to neighbours; one ulp of the normalised value times SiLU(gate)
    is less than two ulps of the output. The kernel's own rounding of the
    output adds half an ulp (the oracle returns the unrounded product), and
    the arithmetic before the roundings the rest. A state (fp32 on both sides)
    gets the plain 3e-2. ``kind`` is "out" or "state"; by default it is read
    from ``what`` (a name ending in "state" is a state)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if kind is None:
        kind = "state" if what.rstrip().endswith("state") else "out"
    scaled, rel = errors(got, ref)
    d = np.abs(got - ref)
    raw = float(d.max()) if d.size else 0.0
    if dtype == "fp32":
        print(f"[parity] {what}: dtype={dtype} max_abs={raw:.3e} max_scaled={scaled:.3e} rel_l2={rel:.3e}")
        assert scaled <= 1e-4, f"{what}: max scaled error {scaled:.3e} > 1e-4"
        return
    if kind == "out":
        u = ulp_act(ref, dtype)
        bound = np.maximum(3e-2, 3.0 * u)
        ulps = float((d / u).max()) if d.size else 0.0
    else:
        bound = np.full(d.shape, 3e-2)
        ulps = float("nan")
    over = int((d > 3e-2).sum())
    worst = float((d / bound).max()) if d.size else 0.0
    print(f"[parity] {what}: dtype={dtype} max_abs={raw:.3e} max_ulps={ulps:.2f} "
          f"n_over_3e-2={over}/{d.size} max_scaled={scaled:.3e} rel_l2={rel:.3e} bound_use={worst:.3f}")
    assert worst <= 1.0, (f"{what}: max |d| {raw:.3e} exceeds max(3e-2, three {dtype} ulps) "
                          f"({worst:.3f} of the bound)")
    assert rel <= 5e-3, f"{what}: relative L2 error {rel:.3e} > 5e-3"


def oracle_backward(inp, grad_out, grad_final=None, threads=8):
    """The oracle's gradients for the same rounded inputs and cotangents."""
    w = inp.w
    return O.backward(q_raw=flat(inp.q_raw), k_raw=flat(inp.k_raw), v_raw=flat(inp.v_raw),
                      a=flat(inp.a), b=flat(inp.b), gate=flat(inp.gate.contiguous()),
                      conv_w=inp.conv_w.float().numpy(), A_log=inp.A_log.numpy(),
                      dt_bias=inp.dt_bias.numpy(), norm_w=inp.norm_w.float().numpy(),
                      seq_start=inp.seq_starts(), Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv,
                      grad_out=grad_out.float().reshape(-1, w.Hv, w.dv).numpy(),
                      grad_final=None if grad_final is None else grad_final.numpy(),
                      initial_state=None if inp.initial_state is None else inp.initial_state.numpy(),
                      threads=threads)


def check_grad(got, ref, dtype, what, tol):
    """Gradient tolerance, relative to the tensor's own scale: relative L2 and
    max |d| / max |ref| (gradients have no natural unit, so the forward's
    max(1, |ref|) floor would hide errors in small gradients)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))
    mx = float(np.abs(ref).max()) if ref.size else 0.0
    rmax = float(np.abs(got - ref).max() / mx) if mx > 0 else float(np.abs(got).max() if got.size else 0.0)
    print(f"[grad] {what}: dtype={dtype} rel_l2={rel:.3e} max_rel={rmax:.3e}")
    l2, mxt = tol
    assert rel <= l2, f"{what}: relative L2 error {rel:.3e} > {l2:.1e}"
    assert rmax <= mxt, f"{what}: max error {rmax:.3e} of max |ref| > {mxt:.1e}"


def chunk_survival(inp, C=64):
    """Fraction of full (sequence, v head, chunk) triples whose decay over the
    chunk, exp(sum of g), is at least 0.1: how much of the carried state still
    reaches the next chunk. Uses the oracle's pinned beta/decay step."""
    _, g = O.beta_decay(flat(inp.a), flat(inp.b), inp.A_log.numpy(), inp.dt_bias.numpy())
    s = inp.seq_starts()
    keep, tot = 0, 0
    for s0, s1 in zip(s[:-1], s[1:]):
        for c0 in range(s0, s1 - C + 1, C):
            e = np.exp(g[c0:c0 + C].sum(axis=0))
            keep += int((e >= 0.1).sum())
            tot += e.size
    return keep / tot if tot else 0.0
