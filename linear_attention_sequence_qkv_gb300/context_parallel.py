"""Sequence-sharded (context-parallel) GDN core forward: one long sequence split
into consecutive spans, one per rank, joined by an affine state scan.

Over a span the chunked gated delta rule (S_t = exp(g_t) S_{t-1} (I - beta_t
k_t k_t^T) + beta_t v_t k_t^T, state H = S^T) is affine in the span's initial
state, H_end = A H_start + B. Each rank

1. takes the raw q|k|v inputs of the previous span's last three tokens as its
   conv prefix (exchanged between ranks: the width-4 causal conv needs them),
2. computes its span's maps with two calls of gdn_forward_with_prefix: B from
   a zero state; A with v = 0, dv = dk and the identity as initial state,
3. gathers every span's (A, B) (one all-gather: the path's only exchange),
4. composes them with gdn_span_scan into its own initial state, and
5. runs its span's forward from that state: its outputs, and (on the last
   rank) the sequence's final state.

The pages shard long context by moving heads instead (an all-to-all around the
local op, "GDN Elementwise Fusion", option table); the state scan above keeps
every head on every rank and exchanges only the dk x (dk + dv) maps per head.

Every step of the core runs in libgdn.so's kernels; this module allocates,
lays out the per-span inputs (zeros and identities for the map A) and calls
the collectives. ``emulate`` runs the same steps for all spans in one process
(collectives replaced by lists), which is how one GPU exercises the path.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import torch

from . import gdn

CONV_HALO = 3   # raw tokens of left context the width-4 conv needs


def raw_channels(q_raw: torch.Tensor, k_raw: torch.Tensor, v_raw: torch.Tensor) -> torch.Tensor:
    """[T, ch] raw inputs in conv_w's channel order (q | k | v) of a [1, T, *] span."""
    return torch.cat([q_raw[0], k_raw[0], v_raw[0]], dim=-1)


def tail_tokens(q_raw, k_raw, v_raw) -> torch.Tensor:
    """[3, ch]: the raw inputs of the span's last three tokens (the next span's conv prefix)."""
    x = raw_channels(q_raw, k_raw, v_raw)
    if x.shape[0] < CONV_HALO:
        raise ValueError("every span of a split sequence needs at least three tokens")
    return x[-CONV_HALO:].contiguous()


def exchange_tails(tail: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of every rank's tail; returns this rank's conv prefix [1, 3, ch]
    (the previous rank's tail, zeros on rank 0)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    tails = [torch.empty_like(tail) for _ in range(world)]
    dist.all_gather(tails, tail.contiguous(), group=group)
    pre = torch.zeros_like(tail) if rank == 0 else tails[rank - 1]
    return pre.unsqueeze(0).contiguous()


def gather_maps(A: torch.Tensor, B: torch.Tensor, group=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """All-gather of every span's maps in rank order: A [world, Hv, dk, dk], B [world, Hv, dk, dv]."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    As = [torch.empty_like(A) for _ in range(world)]
    Bs = [torch.empty_like(B) for _ in range(world)]
    dist.all_gather(As, A.contiguous(), group=group)
    dist.all_gather(Bs, B.contiguous(), group=group)
    return torch.stack(As).contiguous(), torch.stack(Bs).contiguous()


def _fwd(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, prefix, h0, Hk, Hv, dk, dv,
         stream=None):
    d = gdn.desc_for(q_raw, k_raw, v_raw, a, b, gate, norm_w, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    bufs = gdn.alloc(d, q_raw.device)
    gdn.gdn_forward_with_prefix(d, q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, None,
                                prefix, h0, bufs.out, bufs.final_state, bufs.workspace, bufs.ws_bytes, stream)
    return bufs


def span_maps(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, prefix, *, Hk, Hv, dk, dv,
              stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The span's affine state maps: A [Hv, dk, dk], B [Hv, dk, dv] (fp32)."""
    B = _fwd(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, prefix, None, Hk, Hv, dk, dv,
             stream).final_state
    T = q_raw.shape[1]
    dev, act = q_raw.device, q_raw.dtype
    ch_qk = Hk * dk
    v0 = torch.zeros((1, T, Hv * dk), dtype=act, device=dev)
    gate0 = torch.zeros((1, T, Hv * dk), dtype=gate.dtype, device=dev)
    w0 = torch.ones(dk, dtype=norm_w.dtype, device=dev)
    conv0 = torch.cat([conv_w[:2 * ch_qk], torch.zeros((Hv * dk, conv_w.shape[1]), dtype=conv_w.dtype,
                                                       device=dev)]).contiguous()
    pre0 = None
    if prefix is not None:
        pre0 = torch.cat([prefix[:, :, :2 * ch_qk],
                          torch.zeros((prefix.shape[0], CONV_HALO, Hv * dk), dtype=prefix.dtype, device=dev)],
                         dim=2).contiguous()
    eye = torch.eye(dk, dtype=torch.float32, device=dev).expand(1, Hv, dk, dk).contiguous()
    A = _fwd(q_raw, k_raw, v0, a, b, gate0, conv0, A_log, dt_bias, w0, pre0, eye, Hk, Hv, dk, dk,
             stream).final_state
    return A[0], B[0]


def span_initial_states(A_all: torch.Tensor, B_all: torch.Tensor, h0: Optional[torch.Tensor],
                        stream=None) -> torch.Tensor:
    """H_in [spans, Hv, dk, dv] from every span's maps (gdn_span_scan)."""
    S, Hv, dk, _ = A_all.shape
    dv = B_all.shape[-1]
    H_in = torch.empty((S, Hv, dk, dv), dtype=torch.float32, device=A_all.device)
    gdn.gdn_span_scan(S, Hv, dk, dv, A_all, B_all, None if h0 is None else h0.contiguous(), H_in, stream)
    return H_in


def context_parallel_forward(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, *, Hk, Hv, dk, dv,
                             initial_state: Optional[torch.Tensor] = None, group=None, stream=None):
    """This rank's span of one sequence ([1, T_r, *] tensors, spans in rank order,
    each at least three tokens). Returns (out [1, T_r, Hv, dv], final state
    [1, Hv, dk, dv] of the span: the sequence's final state on the last rank).
    initial_state: the sequence's initial state [1, Hv, dk, dv] (used on every
    rank's scan; only rank 0's span starts from it) or None."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    prefix = exchange_tails(tail_tokens(q_raw, k_raw, v_raw), group)
    if rank == 0:
        prefix = None
    A, B = span_maps(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, prefix, Hk=Hk, Hv=Hv,
                     dk=dk, dv=dv, stream=stream)
    A_all, B_all = gather_maps(A, B, group)
    H_in = span_initial_states(A_all, B_all, None if initial_state is None else initial_state[0], stream)
    bufs = _fwd(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, prefix,
                H_in[rank:rank + 1].contiguous(), Hk, Hv, dk, dv, stream)
    return bufs.out, bufs.final_state


def emulate(q_raw, k_raw, v_raw, a, b, gate, conv_w, A_log, dt_bias, norm_w, cuts: List[int], *, Hk, Hv, dk, dv,
            initial_state: Optional[torch.Tensor] = None, stream=None):
    """All spans [cuts[i], cuts[i+1]) of one [1, T, *] sequence in one process,
    with the same steps as context_parallel_forward (the collectives replaced by
    lists). Returns (out [1, T, Hv, dv], final state [1, Hv, dk, dv])."""
    spans = list(zip(cuts[:-1], cuts[1:]))

    def sl(x, t0, t1):
        return x[:, t0:t1]

    prefixes, maps = [], []
    for i, (t0, t1) in enumerate(spans):
        if t1 - t0 < CONV_HALO:
            raise ValueError("every span of a split sequence needs at least three tokens")
        prefix = None
        if i > 0:
            p0 = spans[i - 1][0]
            prefix = tail_tokens(sl(q_raw, p0, t0), sl(k_raw, p0, t0), sl(v_raw, p0, t0)).unsqueeze(0)
        prefixes.append(prefix)
        maps.append(span_maps(sl(q_raw, t0, t1), sl(k_raw, t0, t1), sl(v_raw, t0, t1), sl(a, t0, t1),
                              sl(b, t0, t1), sl(gate, t0, t1), conv_w, A_log, dt_bias, norm_w, prefix, Hk=Hk,
                              Hv=Hv, dk=dk, dv=dv, stream=stream))
    A_all = torch.stack([m[0] for m in maps]).contiguous()
    B_all = torch.stack([m[1] for m in maps]).contiguous()
    H_in = span_initial_states(A_all, B_all, None if initial_state is None else initial_state[0], stream)
    outs, fin = [], None
    for i, (t0, t1) in enumerate(spans):
        bufs = _fwd(sl(q_raw, t0, t1), sl(k_raw, t0, t1), sl(v_raw, t0, t1), sl(a, t0, t1), sl(b, t0, t1),
                    sl(gate, t0, t1), conv_w, A_log, dt_bias, norm_w, prefixes[i], H_in[i:i + 1].contiguous(), Hk,
                    Hv, dk, dv, stream)
        outs.append(bufs.out)
        fin = bufs.final_state
    return torch.cat(outs, dim=1), fin
