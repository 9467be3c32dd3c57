"""Python binding of the CPU oracle (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The product path never
imports this module.

``build()`` compiles the plain C oracle with gcc (portable flags only, and
``-ffp-contract=off`` so results do not depend on whether the host fuses
multiply-adds). The heavy loops run in C; ``ctypes`` releases the GIL during
each call, so ``forward`` can spread v heads over host threads.
"""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_SRC_BWD = os.path.join(_HERE, "gdn_oracle_bwd.c")
_HDR = os.path.join(_HERE, "gdn_oracle.h")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

# "fp64": the RMSNorm result is not rounded (the real-valued forward)
ACT_CODES = {"fp32": 0, "bf16": 1, "fp16": 2, "fp64": 3}

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


class _Problem(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int), ("seq_start", _i64p),
        ("Hk", ctypes.c_int), ("Hv", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("conv_width", ctypes.c_int), ("act", ctypes.c_int),
        ("l2_eps", ctypes.c_double), ("norm_eps", ctypes.c_double), ("scale", ctypes.c_double),
        ("q_raw", _f32p), ("k_raw", _f32p), ("v_raw", _f32p), ("a", _f32p), ("b", _f32p),
        ("gate", _f32p), ("conv_w", _f32p), ("A_log", _f32p), ("dt_bias", _f32p),
        ("norm_w", _f32p), ("initial_state", _f32p),
        ("out", _f64p), ("final_state", _f64p),
        ("chunked", ctypes.c_int),
        ("conv_prefix", _f32p),
    ]


class _DecodeProblem(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("conv_width", ctypes.c_int), ("act", ctypes.c_int),
        ("l2_eps", ctypes.c_double), ("norm_eps", ctypes.c_double), ("scale", ctypes.c_double),
        ("q_raw", _f32p), ("k_raw", _f32p), ("v_raw", _f32p), ("a", _f32p), ("b", _f32p),
        ("gate", _f32p), ("conv_w", _f32p), ("A_log", _f32p), ("dt_bias", _f32p),
        ("norm_w", _f32p), ("conv_state", _f32p), ("state", _f64p),
        ("out", _f64p), ("conv_state_out", _f64p), ("state_out", _f64p),
    ]


class _BwdProblem(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int), ("seq_start", _i64p),
        ("Hk", ctypes.c_int), ("Hv", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("conv_width", ctypes.c_int),
        ("l2_eps", ctypes.c_double), ("norm_eps", ctypes.c_double), ("scale", ctypes.c_double),
        ("q_raw", _f32p), ("k_raw", _f32p), ("v_raw", _f32p), ("a", _f32p), ("b", _f32p),
        ("gate", _f32p), ("conv_w", _f32p), ("A_log", _f32p), ("dt_bias", _f32p),
        ("norm_w", _f32p), ("initial_state", _f32p), ("grad_out", _f32p), ("grad_final", _f32p),
        ("dq_raw", _f64p), ("dk_raw", _f64p), ("dv_raw", _f64p), ("da", _f64p), ("db", _f64p),
        ("dgate", _f64p), ("dconv_w", _f64p), ("dA_log", _f64p), ("dt_bias_grad", _f64p),
        ("dnorm_w", _f64p), ("dinitial_state", _f64p),
    ]


def build(force: bool = False) -> str:
    """Compile ``libgdn_oracle.so`` next to its source if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB) or
                 os.path.getmtime(_LIB) < max(os.path.getmtime(f) for f in (_SRC, _SRC_BWD, _HDR)))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                   "-fno-fast-math", "-o", tmp, _SRC, _SRC_BWD, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.gdn_oracle_round_act.restype = ctypes.c_double
        L.gdn_oracle_round_act.argtypes = [ctypes.c_double, ctypes.c_int]
        L.gdn_oracle_conv_silu.restype = None
        L.gdn_oracle_conv_silu.argtypes = [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int,
                                           _f32p, ctypes.c_int64, _f32p, _f64p]
        L.gdn_oracle_l2norm.restype = None
        L.gdn_oracle_l2norm.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_double, _f64p]
        L.gdn_oracle_beta_decay.restype = None
        L.gdn_oracle_beta_decay.argtypes = [ctypes.c_int64, ctypes.c_int, _f32p, _f32p,
                                            _f32p, _f32p, _f64p, _f64p]
        rule_args = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                     _f64p, ctypes.c_int64, _f64p, ctypes.c_int64, _f64p, ctypes.c_int64,
                     _f64p, _f64p, ctypes.c_int64, ctypes.c_double, _f64p,
                     _f64p, ctypes.c_int64, _f64p]
        L.gdn_oracle_delta_rule.restype = None
        L.gdn_oracle_delta_rule.argtypes = rule_args
        L.gdn_oracle_delta_rule_chunked.restype = None
        L.gdn_oracle_delta_rule_chunked.argtypes = rule_args[:3] + [ctypes.c_int] + rule_args[3:]
        L.gdn_oracle_gated_rmsnorm.restype = None
        L.gdn_oracle_gated_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int, _f64p, ctypes.c_int64,
                                               _f32p, ctypes.c_int64, _f32p, ctypes.c_double,
                                               ctypes.c_int, _f64p, ctypes.c_int64]
        L.gdn_oracle_forward.restype = ctypes.c_int
        L.gdn_oracle_forward.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int, ctypes.c_int]
        L.gdn_oracle_backward.restype = ctypes.c_int
        L.gdn_oracle_backward.argtypes = [ctypes.POINTER(_BwdProblem), ctypes.c_int, ctypes.c_int]
        L.gdn_oracle_decode.restype = ctypes.c_int
        L.gdn_oracle_decode.argtypes = [ctypes.POINTER(_DecodeProblem)]
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers
def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p32(a: Optional[np.ndarray]):
    return a.ctypes.data_as(_f32p) if a is not None else None


def _p64(a: Optional[np.ndarray]):
    return a.ctypes.data_as(_f64p) if a is not None else None


def round_act(x: float, dtype: str) -> float:
    return lib().gdn_oracle_round_act(float(x), ACT_CODES[dtype])


def conv_silu(x: np.ndarray, w: np.ndarray, seq_start: Sequence[int]) -> np.ndarray:
    """x [ntok, nch] (float32 values), w [nch, width] -> y [ntok, nch] float64."""
    x = _f32(x)
    w = _f32(w)
    ntok, nch = x.shape
    s = np.ascontiguousarray(np.asarray(seq_start, dtype=np.int64))
    y = np.zeros((ntok, nch), dtype=np.float64)
    lib().gdn_oracle_conv_silu(len(s) - 1, s.ctypes.data_as(_i64p), nch, w.shape[1],
                               _p32(x), nch, _p32(w), _p64(y))
    return y


def l2norm(x: np.ndarray, d: int, eps: float = 1e-6) -> np.ndarray:
    x = _f64(x).copy()
    nrows = x.shape[0]
    nheads = x.shape[1] // d
    lib().gdn_oracle_l2norm(nrows, nheads, d, eps, _p64(x))
    return x


def beta_decay(a, b, A_log, dt_bias):
    a = _f32(a)
    b = _f32(b)
    ntok, H = a.shape
    beta = np.zeros((ntok, H))
    g = np.zeros((ntok, H))
    lib().gdn_oracle_beta_decay(ntok, H, _p32(a), _p32(b), _p32(_f32(A_log)),
                                _p32(_f32(dt_bias)), _p64(beta), _p64(g))
    return beta, g


def delta_rule(q, k, v, beta, g, h0=None, scale=1.0, chunk: int = 0):
    """Single (sequence, head): q,k [T,dk], v [T,dv], beta,g [T]; h0 [dk,dv] (= S^T).
    Returns (o [T,dv], hT [dk,dv]). ``chunk`` > 0 selects the chunked variant."""
    q, k, v, beta, g = _f64(q), _f64(k), _f64(v), _f64(beta), _f64(g)
    T, dk = q.shape
    dv = v.shape[1]
    h0a = _f64(h0) if h0 is not None else None
    o = np.zeros((T, dv))
    hT = np.zeros((dk, dv))
    L = lib()
    if chunk > 0:
        L.gdn_oracle_delta_rule_chunked(T, dk, dv, chunk, _p64(q), dk, _p64(k), dk, _p64(v), dv,
                                        _p64(beta), _p64(g), 1, scale, _p64(h0a),
                                        _p64(o), dv, _p64(hT))
    else:
        L.gdn_oracle_delta_rule(T, dk, dv, _p64(q), dk, _p64(k), dk, _p64(v), dv,
                                _p64(beta), _p64(g), 1, scale, _p64(h0a), _p64(o), dv, _p64(hT))
    return o, hT


def gated_rmsnorm(o, gate, norm_w, eps=1e-5, dtype="fp32"):
    o = _f64(o)
    gate = _f32(gate)
    nrows, dv = o.shape
    y = np.zeros((nrows, dv))
    lib().gdn_oracle_gated_rmsnorm(nrows, dv, _p64(o), dv, _p32(gate), dv, _p32(_f32(norm_w)),
                                   eps, ACT_CODES[dtype], _p64(y), dv)
    return y


def forward(*, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
            seq_start, Hk, Hv, dk, dv, dtype, initial_state=None,
            l2_eps=1e-6, norm_eps=1e-5, scale=1.0, conv_width=4,
            heads: Optional[Sequence[int]] = None, threads: int = 1, chunked: int = 0,
            conv_prefix=None):
    """Whole core forward on flattened token arrays (float32 values):
    q_raw/k_raw [ntok, Hk*dk], v_raw [ntok, Hv*dv], a/b [ntok, Hv],
    gate [ntok, Hv*dv], conv_w [ch, width], A_log/dt_bias [Hv], norm_w [dv],
    initial_state [N, Hv, dk, dv] or None, conv_prefix [N, width-1, ch] (the raw
    inputs of the tokens before each sequence, oldest first) or None.
    Returns (out [ntok, Hv, dv] float64, final_state [N, Hv, dk, dv] float64);
    heads not in ``heads`` are left at zero."""
    arrs = dict(q_raw=_f32(q_raw), k_raw=_f32(k_raw), v_raw=_f32(v_raw), a=_f32(a), b=_f32(b),
                gate=_f32(gate), conv_w=_f32(conv_w), A_log=_f32(A_log),
                dt_bias=_f32(dt_bias), norm_w=_f32(norm_w))
    init = _f32(initial_state) if initial_state is not None else None
    pre = _f32(conv_prefix) if conv_prefix is not None else None
    s = np.ascontiguousarray(np.asarray(seq_start, dtype=np.int64))
    n_seq = len(s) - 1
    ntok = int(s[-1])
    out = np.zeros((ntok, Hv, dv))
    fin = np.zeros((n_seq, Hv, dk, dv))
    prob = _Problem(
        n_seq=n_seq, seq_start=s.ctypes.data_as(_i64p), Hk=Hk, Hv=Hv, dk=dk, dv=dv,
        conv_width=conv_width, act=ACT_CODES[dtype], l2_eps=l2_eps, norm_eps=norm_eps,
        scale=scale, **{k: _p32(v) for k, v in arrs.items()},
        initial_state=_p32(init), out=_p64(out), final_state=_p64(fin), chunked=int(chunked),
        conv_prefix=_p32(pre))
    heads = list(range(Hv)) if heads is None else list(heads)
    L = lib()

    def run(h):
        rc = L.gdn_oracle_forward(ctypes.byref(prob), h, h + 1)
        if rc != 0:
            raise RuntimeError(f"gdn_oracle_forward failed for head {h}")

    if threads <= 1 or len(heads) <= 1:
        for h in heads:
            run(h)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, heads))
    return out, fin


def decode(*, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
           conv_state, state, Hk, Hv, dk, dv, dtype,
           l2_eps=1e-6, norm_eps=1e-5, scale=1.0, conv_width=4):
    """One decode step (float32 values, one token per sequence):
    q_raw/k_raw [N, Hk*dk], v_raw [N, Hv*dv], a/b [N, Hv], gate [N, Hv*dv],
    conv_state [N, ch, width-1] (raw inputs of the last tokens, oldest first),
    state [N, Hv, dk, dv] (taken in float64). Returns (out [N, Hv, dv],
    conv_state_out, state_out), all float64."""
    arrs = dict(q_raw=_f32(q_raw), k_raw=_f32(k_raw), v_raw=_f32(v_raw), a=_f32(a), b=_f32(b),
                gate=_f32(gate), conv_w=_f32(conv_w), A_log=_f32(A_log),
                dt_bias=_f32(dt_bias), norm_w=_f32(norm_w), conv_state=_f32(conv_state))
    st = _f64(state)
    n = arrs["q_raw"].shape[0]
    ch = 2 * Hk * dk + Hv * dv
    out = np.zeros((n, Hv, dv))
    cso = np.zeros((n, ch, conv_width - 1))
    so = np.zeros((n, Hv, dk, dv))
    prob = _DecodeProblem(
        n_seq=n, Hk=Hk, Hv=Hv, dk=dk, dv=dv, conv_width=conv_width, act=ACT_CODES[dtype],
        l2_eps=l2_eps, norm_eps=norm_eps, scale=scale, **{k: _p32(v) for k, v in arrs.items()},
        state=_p64(st), out=_p64(out), conv_state_out=_p64(cso), state_out=_p64(so))
    if lib().gdn_oracle_decode(ctypes.byref(prob)) != 0:
        raise RuntimeError("gdn_oracle_decode failed")
    return out, cso, so


def backward(*, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w,
             seq_start, Hk, Hv, dk, dv, grad_out, grad_final=None, initial_state=None,
             l2_eps=1e-6, norm_eps=1e-5, scale=1.0, conv_width=4, threads: int = 1):
    """Gradients of sum(grad_out * out) + sum(grad_final * final_state) with
    respect to every input of ``forward`` (float32 values in the forward's
    shapes; grad_out [ntok, Hv, dv], grad_final [N, Hv, dk, dv] or None). The
    RMSNorm rounding is taken as the identity. Returns a dict of float64 arrays:
    dq_raw, dk_raw, dv_raw, da, db, dgate, dconv_w, dA_log, ddt_bias, dnorm_w,
    dinitial_state. ``threads`` spreads q/k heads over host threads."""
    arrs = dict(q_raw=_f32(q_raw), k_raw=_f32(k_raw), v_raw=_f32(v_raw), a=_f32(a), b=_f32(b),
                gate=_f32(gate), conv_w=_f32(conv_w), A_log=_f32(A_log),
                dt_bias=_f32(dt_bias), norm_w=_f32(norm_w), grad_out=_f32(grad_out))
    init = _f32(initial_state) if initial_state is not None else None
    gfin = _f32(grad_final) if grad_final is not None else None
    s = np.ascontiguousarray(np.asarray(seq_start, dtype=np.int64))
    n_seq = len(s) - 1
    ntok = int(s[-1])
    ch = 2 * Hk * dk + Hv * dv
    out = dict(dq_raw=np.zeros((ntok, Hk * dk)), dk_raw=np.zeros((ntok, Hk * dk)),
               dv_raw=np.zeros((ntok, Hv * dv)), da=np.zeros((ntok, Hv)), db=np.zeros((ntok, Hv)),
               dgate=np.zeros((ntok, Hv * dv)), dconv_w=np.zeros((ch, conv_width)),
               dA_log=np.zeros(Hv), ddt_bias=np.zeros(Hv), dnorm_w=np.zeros((Hv, dv)),
               dinitial_state=np.zeros((n_seq, Hv, dk, dv)))
    prob = _BwdProblem(
        n_seq=n_seq, seq_start=s.ctypes.data_as(_i64p), Hk=Hk, Hv=Hv, dk=dk, dv=dv,
        conv_width=conv_width, l2_eps=l2_eps, norm_eps=norm_eps, scale=scale,
        **{k: _p32(v) for k, v in arrs.items()}, initial_state=_p32(init), grad_final=_p32(gfin),
        dq_raw=_p64(out["dq_raw"]), dk_raw=_p64(out["dk_raw"]), dv_raw=_p64(out["dv_raw"]),
        da=_p64(out["da"]), db=_p64(out["db"]), dgate=_p64(out["dgate"]),
        dconv_w=_p64(out["dconv_w"]), dA_log=_p64(out["dA_log"]), dt_bias_grad=_p64(out["ddt_bias"]),
        dnorm_w=_p64(out["dnorm_w"]), dinitial_state=_p64(out["dinitial_state"]))
    L = lib()

    def run(hk):
        if L.gdn_oracle_backward(ctypes.byref(prob), hk, hk + 1) != 0:
            raise RuntimeError(f"gdn_oracle_backward failed for q/k head {hk}")

    if threads <= 1 or Hk <= 1:
        for hk in range(Hk):
            run(hk)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, range(Hk)))
    out["dnorm_w"] = out["dnorm_w"].sum(axis=0)
    return out
