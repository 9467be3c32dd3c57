"""Writes closed_forms.json: textbook values of the GDN core's elementwise
definitions at hand-picked inputs, evaluated with Python's math module (no call
into the oracle or the CUDA library).

Definitions (GDN core; "GDN Elementwise Fusion", option table):
  silu(x) = x / (1 + e^-x)                       (the conv's activation)
  beta    = sigmoid(b) = 1 / (1 + e^-b)
  g       = -exp(A_log) * log(1 + e^(a + dt_bias))
  y       = fp32(norm_w * o / sqrt(mean(o^2) + eps)) * silu(gate)
Inputs are chosen exactly representable in float32.
"""
import json
import math
import os
import struct


def f32(x):
    return struct.unpack("f", struct.pack("f", x))[0]


def silu(x):
    return x / (1.0 + math.exp(-x))


cases = [
    {"kind": "silu_tap3", "x": 2.0, "want": silu(2.0),
     "cite": "short conv with a one-hot current-token tap, then SiLU"},
    {"kind": "silu_tap3", "x": -0.5, "want": silu(-0.5), "cite": "same"},
    {"kind": "beta_decay", "a": 0.0, "b": 0.0, "A_log": 0.0, "dt_bias": 0.0,
     "beta": 0.5, "g": -math.log(2.0), "cite": "beta = sigmoid(b); g = -e^A_log softplus(a+dt_bias)"},
    {"kind": "beta_decay", "a": 1.0, "b": -1.0, "A_log": 0.5, "dt_bias": 0.0,
     "beta": 1.0 / (1.0 + math.e), "g": -math.exp(0.5) * math.log(1.0 + math.e), "cite": "same"},
    {"kind": "beta_decay", "a": -2.0, "b": 3.0, "A_log": 2.0, "dt_bias": 0.5,
     "beta": 1.0 / (1.0 + math.exp(-3.0)), "g": -math.exp(2.0) * math.log(1.0 + math.exp(-1.5)),
     "cite": "same"},
]
for o, nw, gate, eps in ((2.0, 1.5, -1.0, 1e-5), (0.25, 0.75, 3.0, 1e-5)):
    r = f32(nw * o / math.sqrt(o * o + eps))
    cases.append({"kind": "gated_rmsnorm_const", "dv": 4, "o": o, "norm_w": nw, "gate": gate,
                  "eps": eps, "want": r * silu(gate),
                  "cite": "RMSNorm of a constant row, weight, fp32 materialisation, SiLU gate"})

with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms.json"), "w") as f:
    json.dump({"source": "GDN core elementwise definitions, evaluated by make_closed_forms.py",
               "cases": cases}, f, indent=1)
