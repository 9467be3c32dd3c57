"""Seeded synthetic workloads for the Gated DeltaNet (GDN) layer core forward.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. The same generators feed the CUDA path (tests, benchmark,
smoke check) and the CPU oracle, so both see bit-identical, already-rounded
inputs.

Value recipe (all draws from a seeded ``torch.Generator`` on the CPU, in fp32,
then rounded once to the activation dtype):

* ``q_raw, k_raw, v_raw, a, b, gate`` ~ N(0, 1)
* ``conv_w`` ~ N(0, 0.25)  (0.25 read as the standard deviation)
* ``A_log`` = log U[1, 16]   (fp32, one per v head); a workload may set
  ``decay_range = (lo, hi)`` to draw ``A_log = log U[lo, hi]`` instead (the
  same uniform draw, mapped to another interval). ``MILD`` = (0.001, 0.05) is
  the long-memory recipe of the tests: with it the per-chunk decay
  ``exp(sum of g over 64 tokens)`` is about 0.05-0.95 instead of below 1e-90,
  so the state carried from chunk to chunk reaches the outputs.
* ``dt_bias`` ~ N(0, 0.1)    (fp32, one per v head; 0.1 read as std)
* ``norm_w`` = 1 + N(0, 0.1) (activation dtype)
* ``initial_state`` = 0, or N(0, 0.1) in fp32 where a workload asks for it
* packed sequences: lengths ~ U[1, 8192] integers, concatenated with int32
  ``cu_seqlens``; the gate is then a strided view into a wider projection
  buffer.

Shapes follow the projections of a GDN layer: q/k projections give
``Hk * dk`` channels per token, the v projection ``Hv * dv``, the a/b
projections ``Hv`` each, and the output gate ``Hv * dv`` (a view into a wider
buffer of ``Hv * dv + extra`` channels when ``gate_extra`` is set).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

ACT_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str              # activation dtype: "fp32" | "bf16" | "fp16"
    B: int                  # batch (1 when packed)
    T: int                  # tokens per batch row (total tokens when packed)
    Hk: int                 # q/k heads
    Hv: int                 # v heads (multiple of Hk)
    dk: int
    dv: int
    n_packed: int = 0       # >0: number of packed sequences (lengths U[1, max_len])
    max_len: int = 8192
    gate_extra: int = 0     # >0: gate is a view into [B, T, Hv*dv + gate_extra]
    init_state_std: float = 0.0
    seed: int = 0
    description: str = ""
    decay_range: tuple = (1.0, 16.0)   # A = exp(A_log) ~ U[lo, hi]

    @property
    def G(self) -> int:
        return self.Hv // self.Hk


# exp(A_log) range of the long-memory test recipe (see the module docstring)
MILD = (0.001, 0.05)

WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", "fp32", B=1, T=128, Hk=2, Hv=2, dk=64, dv=64,
        description="tiny fp32 core: B=1 T=128 2/2 heads dk=dv=64"),
    "layer_bf16": Workload(
        "layer_bf16", "bf16", B=2, T=2048, Hk=6, Hv=6, dk=256, dv=512,
        description="representative layer bf16: B=2 T=2048 hidden 2048 -> 6 heads dk=256 dv=512"),
    "ragged_fp16": Workload(
        "ragged_fp16", "fp16", B=2, T=100, Hk=6, Hv=6, dk=64, dv=128,
        gate_extra=64, init_state_std=0.1,
        description="ragged tail fp16: B=2 T=100 6 heads dk=64 dv=128, strided gate, random initial state"),
    "long_gqa_bf16": Workload(
        "long_gqa_bf16", "bf16", B=1, T=131072, Hk=16, Hv=32, dk=128, dv=128,
        description="long-context GQA bf16: B=1 T=131072 16->32 heads dk=dv=128"),
    "varlen_bf16": Workload(
        "varlen_bf16", "bf16", B=1, T=0, Hk=16, Hv=32, dk=128, dv=128,
        n_packed=64, max_len=8192, gate_extra=64,
        description="packed varlen bf16: 64 sequences U[1,8192] 16->32 heads dk=dv=128, strided gate"),
}


def replace(w: Workload, **kw) -> Workload:
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


@dataclass
class Inputs:
    """Host (CPU) tensors of one problem, already rounded to the act dtype."""
    w: Workload
    q_raw: torch.Tensor        # [B, T, Hk*dk] act
    k_raw: torch.Tensor        # [B, T, Hk*dk] act
    v_raw: torch.Tensor        # [B, T, Hv*dv] act
    a: torch.Tensor            # [B, T, Hv] act
    b: torch.Tensor            # [B, T, Hv] act
    gate_buf: torch.Tensor     # [B, T, Hv*dv + extra] act (gate = gate_buf[..., :Hv*dv])
    conv_w: torch.Tensor       # [2*Hk*dk + Hv*dv, 4] act
    A_log: torch.Tensor        # [Hv] fp32
    dt_bias: torch.Tensor      # [Hv] fp32
    norm_w: torch.Tensor       # [dv] act
    cu_seqlens: Optional[torch.Tensor]     # [N+1] int32 or None
    initial_state: Optional[torch.Tensor]  # [N, Hv, dk, dv] fp32 or None
    extras: dict = field(default_factory=dict)

    @property
    def gate(self) -> torch.Tensor:
        return self.gate_buf[..., : self.w.Hv * self.w.dv]

    @property
    def n_seq(self) -> int:
        return self.cu_seqlens.numel() - 1 if self.cu_seqlens is not None else self.w.B

    @property
    def n_tok(self) -> int:
        return self.q_raw.shape[0] * self.q_raw.shape[1]

    def seq_starts(self) -> list:
        """Token offsets [N+1] of every sequence in the flattened token order."""
        if self.cu_seqlens is not None:
            return [int(x) for x in self.cu_seqlens.tolist()]
        return [i * self.w.T for i in range(self.w.B + 1)]


def packed_lengths(w: Workload) -> list:
    g = torch.Generator().manual_seed(w.seed * 7919 + 17)
    return [int(x) for x in torch.randint(1, w.max_len + 1, (w.n_packed,), generator=g).tolist()]


def make_inputs(w: Workload, lengths: Optional[list] = None) -> Inputs:
    """Draw every input of workload ``w`` on the CPU from its seed."""
    act = ACT_DTYPES[w.dtype]
    g = torch.Generator().manual_seed(w.seed)

    def normal(shape, std=1.0, mean=0.0):
        return (torch.randn(shape, generator=g, dtype=torch.float32) * std + mean)

    cu = None
    B, T = w.B, w.T
    if w.n_packed or lengths is not None:
        if lengths is None:
            lengths = packed_lengths(w)
        offs = [0]
        for L in lengths:
            offs.append(offs[-1] + int(L))
        cu = torch.tensor(offs, dtype=torch.int32)
        B, T = 1, offs[-1]
    ch_qk = w.Hk * w.dk
    ch_v = w.Hv * w.dv
    q_raw = normal((B, T, ch_qk)).to(act)
    k_raw = normal((B, T, ch_qk)).to(act)
    v_raw = normal((B, T, ch_v)).to(act)
    a = normal((B, T, w.Hv)).to(act)
    b = normal((B, T, w.Hv)).to(act)
    gate_buf = normal((B, T, ch_v + w.gate_extra)).to(act)
    conv_w = normal((2 * ch_qk + ch_v, 4), std=0.25).to(act)
    lo, hi = (float(x) for x in w.decay_range)
    A_log = torch.log(torch.rand((w.Hv,), generator=g, dtype=torch.float32) * (hi - lo) + lo)
    dt_bias = normal((w.Hv,), std=0.1)
    norm_w = normal((w.dv,), std=0.1, mean=1.0).to(act)
    n_seq = (cu.numel() - 1) if cu is not None else B
    init = None
    if w.init_state_std > 0:
        init = normal((n_seq, w.Hv, w.dk, w.dv), std=w.init_state_std)
    return Inputs(w, q_raw, k_raw, v_raw, a, b, gate_buf, conv_w, A_log, dt_bias,
                  norm_w, cu, init)


def make_inputs_device(w: Workload, device, lengths: Optional[list] = None) -> Inputs:
    """Same recipe drawn directly on ``device`` (fast; values differ from the
    CPU draw). Used where only the distribution matters, e.g. for timing."""
    act = ACT_DTYPES[w.dtype]
    g = torch.Generator(device=device).manual_seed(w.seed)

    def normal(shape, std=1.0, mean=0.0):
        return torch.randn(shape, generator=g, dtype=torch.float32, device=device) * std + mean

    cu = None
    B, T = w.B, w.T
    if w.n_packed or lengths is not None:
        if lengths is None:
            lengths = packed_lengths(w)
        offs = [0]
        for L in lengths:
            offs.append(offs[-1] + int(L))
        cu = torch.tensor(offs, dtype=torch.int32, device=device)
        B, T = 1, offs[-1]
    ch_qk = w.Hk * w.dk
    ch_v = w.Hv * w.dv
    q_raw = normal((B, T, ch_qk)).to(act)
    k_raw = normal((B, T, ch_qk)).to(act)
    v_raw = normal((B, T, ch_v)).to(act)
    a = normal((B, T, w.Hv)).to(act)
    b = normal((B, T, w.Hv)).to(act)
    gate_buf = normal((B, T, ch_v + w.gate_extra)).to(act)
    conv_w = normal((2 * ch_qk + ch_v, 4), std=0.25).to(act)
    lo, hi = (float(x) for x in w.decay_range)
    A_log = torch.log(torch.rand((w.Hv,), generator=g, dtype=torch.float32, device=device) * (hi - lo) + lo)
    dt_bias = normal((w.Hv,), std=0.1)
    norm_w = normal((w.dv,), std=0.1, mean=1.0).to(act)
    n_seq = (cu.numel() - 1) if cu is not None else B
    init = None
    if w.init_state_std > 0:
        init = normal((n_seq, w.Hv, w.dk, w.dv), std=w.init_state_std)
    return Inputs(w, q_raw, k_raw, v_raw, a, b, gate_buf, conv_w, A_log, dt_bias,
                  norm_w, cu, init)


def to_device(inp: Inputs, device) -> Inputs:
    """Copy every tensor of ``inp`` to ``device`` (views are rebuilt, so the
    gate stays a strided view into its wider buffer)."""
    mv = lambda t: None if t is None else t.to(device)
    return Inputs(inp.w, mv(inp.q_raw), mv(inp.k_raw), mv(inp.v_raw), mv(inp.a), mv(inp.b),
                  mv(inp.gate_buf), mv(inp.conv_w), mv(inp.A_log), mv(inp.dt_bias),
                  mv(inp.norm_w), mv(inp.cu_seqlens), mv(inp.initial_state), dict(inp.extras))


def head_subproblem(inp: Inputs, heads: list) -> Inputs:
    """The same problem restricted to v heads ``heads``: each kept v head h
    brings its own copy of q/k head h // G, so the sub-problem has
    Hk = Hv = len(heads). Pure slicing; used to check sampled heads of large
    workloads."""
    w = inp.w
    G = w.G
    m = len(heads)
    qk_heads = [h // G for h in heads]
    dk, dv = w.dk, w.dv

    def take(t, width, idx):
        return torch.cat([t[..., i * width:(i + 1) * width] for i in idx], dim=-1).contiguous()

    ch_qk = w.Hk * dk
    cw = inp.conv_w
    conv_w = torch.cat([take(cw[:ch_qk].T, dk, qk_heads).T,
                        take(cw[ch_qk:2 * ch_qk].T, dk, qk_heads).T,
                        take(cw[2 * ch_qk:].T, dv, heads).T], dim=0).contiguous()
    return Inputs(replace(w, Hk=m, Hv=m, gate_extra=0),
                  take(inp.q_raw, dk, qk_heads), take(inp.k_raw, dk, qk_heads),
                  take(inp.v_raw, dv, heads), take(inp.a, 1, heads), take(inp.b, 1, heads),
                  take(inp.gate, dv, heads), conv_w, inp.A_log[heads].contiguous(),
                  inp.dt_bias[heads].contiguous(), inp.norm_w, inp.cu_seqlens,
                  None if inp.initial_state is None else inp.initial_state[:, heads].contiguous())


def make_cotangents(inp: Inputs, seed: int = 1, final: bool = True):
    """Seeded gradients of the outputs for the backward: grad_out ~ N(0, 1) in
    the act dtype [B, T, Hv, dv], grad_final ~ N(0, 1) fp32 [N, Hv, dk, dv]
    (or None)."""
    w = inp.w
    g = torch.Generator().manual_seed(seed * 104729 + w.seed)
    B, T = inp.q_raw.shape[0], inp.q_raw.shape[1]
    grad_out = torch.randn((B, T, w.Hv, w.dv), generator=g, dtype=torch.float32).to(ACT_DTYPES[w.dtype])
    grad_final = (torch.randn((inp.n_seq, w.Hv, w.dk, w.dv), generator=g, dtype=torch.float32)
                  if final else None)
    return grad_out, grad_final
