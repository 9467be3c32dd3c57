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


def check(got, ref, dtype, what):
    """Tolerances of the GDN core: fp32 max|d| <= 1e-4 max(1,|ref|); bf16/fp16
    max|d| <= 3e-2 max(1,|ref|) and relative L2 <= 5e-3."""
    scaled, rel = errors(got, ref)
    print(f"[parity] {what}: dtype={dtype} max_scaled={scaled:.3e} rel_l2={rel:.3e}")
    if dtype == "fp32":
        assert scaled <= 1e-4, f"{what}: max scaled error {scaled:.3e} > 1e-4"
    else:
        assert scaled <= 3e-2, f"{what}: max scaled error {scaled:.3e} > 3e-2"
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
