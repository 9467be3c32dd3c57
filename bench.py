#!/usr/bin/env python
"""Throughput of the Gated DeltaNet (GDN) layer core forward on GB300.

One step = one pass of the whole core forward (prologue, chunked gated delta
rule, gated RMSNorm epilogue) over one batch of synthetic input already
resident in HBM. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Timing: W untimed warm-up steps, then exactly K steps (one gdn_forward each,
CUDA events around the call) bracketed by a barrier and a device
synchronisation; L2 is flushed (a 512 MiB write, then a 256 MiB read that
leaves L2 clean) before every timed step, outside the events. Per-kernel
durations come from a second pass of K steps that runs the same work as the
three stage calls with CUDA events recorded on the launching stream between
them. For N > 1 every
rank runs its own replica (the path has no data exchange): value = tokens of
all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN core fwd tokens/s at 1 GB300 and % of roofline (HBM / BF16 MMA)"
CHUNK = 64

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from one
# ncu capture, keyed by kernel; each entry is only used while the kernel's
# source file still hashes to the recorded value.
# kernel -> (source file, sha256 of it, workload, bytes per launch)
# "chunk_rule" is the tensor-core chunk stage: chunk_prep_kernel + chunk_chain_kernel,
# one launch each per step; the figure is the sum of the two launches.
NCU_TRAFFIC: dict = {
    "chunk_rule": ("linear_attention_sequence_qkv_gb300/csrc/gdn_chunk_tc.cu",
                   "7e27d03e8366d5c7351d3b271ab0772303bf47da73b0f4f5293d30bab827f58c",
                   "layer_bf16", 115_082_240),
}


def sha256(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="layer_bf16")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other four workloads (reported under 'workloads')")
    ap.add_argument("--n-packed", type=int, default=0,
                    help="packed workloads: this many sequences instead of the workload's (smaller cases for "
                         "profiling)")
    ap.add_argument("--workload-steps", type=int, default=30,
                    help="timed steps for each of the other workloads (at most --steps)")
    ap.add_argument("--decode", action="store_true",
                    help="time the decode step (one token per sequence) instead of the forward")
    ap.add_argument("--decode-batch", type=int, default=256, help="sequences per decode step")
    ap.add_argument("--backward", action="store_true",
                    help="time forward + backward (gdn_forward then gdn_backward) per step")
    ap.add_argument("--spans", type=int, default=0,
                    help="time the sequence-sharded path with the sequence split into this many spans, "
                         "all on this GPU (the method's cost, not a multi-GPU time)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def algorithmic(w, ntok, n_seq, has_h0):
    """Bytes (and MMA flops) that each kernel must move (do), per launch."""
    s = 4 if w.dtype == "fp32" else 2
    ch = 2 * w.Hk * w.dk + w.Hv * w.dv
    state = n_seq * w.Hv * w.dk * w.dv * 4
    k1 = ntok * (2 * ch * s + 2 * w.Hv * s + 8 * w.Hv)
    k2 = ntok * (ch * s + 8 * w.Hv + w.Hv * w.dv * s) + state * (2 if has_h0 else 1)
    k3 = ntok * 3 * w.Hv * w.dv * s
    C = CHUNK
    k2_flops = ntok * w.Hv * (6 * C * w.dk + 4 * C * w.dv + 6 * w.dk * w.dv + (2.0 / 3.0) * C * C)
    return {"prologue": (k1, 0.0), "chunk_rule": (k2, k2_flops), "epilogue": (k3, 0.0)}


def roofline_entry(name, bytes_, flops, ms, pk, dtype):
    t = ms / 1e3
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    t_mma = flops / (pk["bf16_tflops"] * 1e12) if flops else 0.0
    if flops and t_mma >= t_hbm and dtype != "fp32":
        ach = flops / t / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "algorithmic_flops": flops,
                "algorithmic_bytes": bytes_, "ms": ms}
    ach = bytes_ / t / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"], "algorithmic_bytes": bytes_, "ms": ms}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100"]
        if gpu_id is not None:
            cmd.insert(1, f"--id={gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxs.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "samples": len(sms),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ reference arm
def oracle_sample(w):
    """Bounded sample of the workload for the CPU oracle: the first sequence,
    every v head (all of them for the small workloads)."""
    from linear_attention_sequence_qkv_gb300.workloads import head_subproblem, make_inputs, replace
    if w.n_packed:
        w1 = replace(w, n_packed=0, B=1, T=min(w.max_len, 2048))
    else:
        w1 = replace(w, B=1, T=min(w.T, 2048))
    inp = make_inputs(w1)
    heads = list(range(w1.Hv))
    if w1.Hv * w1.dk * w1.dv * w1.T > 6 * 256 * 512 * 2048:
        heads = heads[:2]
        inp = head_subproblem(inp, heads)
    return inp, w1, len(heads)


def run_oracle_once(inp, threads):
    from oracle import oracle as O
    w = inp.w
    flat = lambda x: x.float().reshape(-1, x.shape[-1]).numpy()
    args = dict(q_raw=flat(inp.q_raw), k_raw=flat(inp.k_raw), v_raw=flat(inp.v_raw), a=flat(inp.a),
                b=flat(inp.b), gate=flat(inp.gate.contiguous()), conv_w=inp.conv_w.float().numpy(),
                A_log=inp.A_log.numpy(), dt_bias=inp.dt_bias.numpy(), norm_w=inp.norm_w.float().numpy(),
                seq_start=inp.seq_starts(), Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv, dtype=w.dtype,
                initial_state=None if inp.initial_state is None else inp.initial_state.numpy(),
                threads=threads)
    t0 = time.perf_counter()
    O.forward(**args)
    return time.perf_counter() - t0


def cpu_baseline(w, cpu_seconds=12.0, max_runs=40):
    """The oracle on the sample, repeated until about ``cpu_seconds`` of CPU work
    (wall time x threads) are done; the median run gives the rate."""
    from oracle import oracle as O
    O.build()
    inp, w1, nheads = oracle_sample(w)
    threads = max(1, min(os.cpu_count() or 1, nheads))
    times = []
    while sum(times) * threads < cpu_seconds and len(times) < max_runs:
        times.append(run_oracle_once(inp, threads))
    dt = statistics.median(times)
    # tokens of the full workload per second: the sample covers nheads of w.Hv heads
    tps = w1.B * w1.T / dt * (nheads / w.Hv)
    return {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{w1.B * w1.T} tokens x {nheads}/{w.Hv} v heads of {w.name}, run {len(times)} "
                      f"times ({sum(times):.1f} s wall on {threads} threads; median {dt:.2f} s), "
                      f"scaled to all heads"}


def reference_arm(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle as O
    O.build()
    inp, w1, nheads = oracle_sample(w)
    threads = max(1, min(os.cpu_count() or 1, nheads))
    for _ in range(args.warmup):
        run_oracle_once(inp, threads)
    times = [run_oracle_once(inp, threads) for _ in range(args.steps)]
    tot = sum(times)
    tps = w1.B * w1.T * args.steps / tot * (nheads / w.Hv)
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample_tokens": w1.B * w1.T, "sample_heads": nheads,
                       "Hv": w.Hv, "dk": w.dk, "dv": w.dv},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{w1.B * w1.T} tokens x {nheads}/{w.Hv} v heads per step"},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our arm
# -------------------------------------------------------------- decode step
def decode_main(args, w):
    """One decode step per timed iteration: args.decode_batch sequences with the
    workload's head shape, each with a conv cache and a state resident in HBM."""
    import torch
    from linear_attention_sequence_qkv_gb300 import build, gdn
    from linear_attention_sequence_qkv_gb300.workloads import make_inputs_device, replace

    build.build()
    gdn.load()
    dev = torch.device("cuda", 0)
    B = args.decode_batch
    wd = replace(w, B=B, T=1, n_packed=0)
    inp = make_inputs_device(wd, dev)
    d = gdn.desc_for(inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.norm_w,
                     Hk=wd.Hk, Hv=wd.Hv, dk=wd.dk, dv=wd.dv)
    ws = torch.empty(gdn.gdn_decode_workspace_bytes(d), dtype=torch.uint8, device=dev)
    ch = 2 * wd.Hk * wd.dk + wd.Hv * wd.dv
    cache = torch.zeros((B, ch, 3), dtype=inp.q_raw.dtype, device=dev)
    state = torch.randn((B, wd.Hv, wd.dk, wd.dv), device=dev) * 0.1
    out = torch.empty((B, 1, wd.Hv, wd.dv), dtype=inp.q_raw.dtype, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        gdn.gdn_decode_step(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.conv_w,
                            inp.A_log, inp.dt_bias, inp.norm_w, cache, state, out, ws, ws.numel(), stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(ws) == gdn.GDN_OK
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = None if args.no_clocks else ClockSampler(None)
    torch.cuda.synchronize()
    for e in evs:
        flush.zero_()
        e[0].record()
        step()
        e[1].record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    s = 4 if wd.dtype == "fp32" else 2
    # algorithmic bytes of a step: the state read and written (fp32), the conv cache
    # read and written, the token's raw inputs, a, b, gate, and the output
    per_seq = (8 * wd.Hv * wd.dk * wd.dv + 2 * 3 * ch * s + ch * s + 2 * wd.Hv * s
               + 2 * wd.Hv * wd.dv * s)
    pk = peaks()
    ach = B * per_seq / (ms / 1e3) / 1e9
    line = {
        "metric": "GDN decode step tokens/s at 1 GB300 and % of HBM roofline", "value": B / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "bf16": "bf16", "fp16": "f16"}[wd.dtype], "data": "synthetic",
        "config": {"workload": f"decode_{w.name}", "sequences": B, "Hk": wd.Hk, "Hv": wd.Hv,
                   "dk": wd.dk, "dv": wd.dv, "l2": "flushed before every timed step (512 MiB write)"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / pk["hbm_gbs"], "algorithmic_bytes": B * per_seq, "traffic": None,
                     "kernel": "decode step (decode_prep + decode_state + epilogue)",
                     "peak_source": pk["source"]},
        "gpu_launches": 3 * args.steps, "gpu_launches_per_step": 3, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- forward + backward
def fp32_alu_peak_tflops():
    """FP32 FMA peak of the CUDA cores: 152 SMs x 128 FP32 lanes x 2 flops x the
    maximum SM clock (MEASURED_PEAKS.json's sm_max_mhz, else 2070 MHz)."""
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except (OSError, ValueError):
        pass
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def backward_flops(w, ntok):
    """Algorithmic flops of gdn_backward (its forward recompute included), per
    token and v head: 18 dk dv + 12 C dv + 12 C dk (C = 64): the recompute
    (K H0, Q H0, the state update; T R0, P Vn; K K^T, Q K^T), the reverse chain
    (Kd dH1, the two dH0 terms; P^T dO', T^T dVn) and the per-chunk gradients
    (dO' H0^T, dR0 H0^T, Vn dH1^T; dO' Vn^T, dR0 Vn^T; four 64x64 by 64xdk
    products)."""
    C = CHUNK
    return ntok * w.Hv * (18 * w.dk * w.dv + 12 * C * w.dv + 12 * C * w.dk)


def oracle_bwd_sample(w):
    from linear_attention_sequence_qkv_gb300.workloads import head_subproblem, make_inputs, replace
    if w.n_packed:
        w1 = replace(w, n_packed=0, B=1, T=min(w.max_len, 1024))
    else:
        w1 = replace(w, B=1, T=min(w.T, 1024))
    inp = make_inputs(w1)
    hk = list(range(w1.Hk))
    if w1.Hv * w1.dk * w1.dv * w1.T > 6 * 256 * 512 * 1024:
        hk = hk[:1]
        inp = head_subproblem(inp, list(range(w1.Hv // w1.Hk)))
    return inp, w1, len(hk) * (w1.Hv // w1.Hk)


def run_oracle_fwd_bwd(inp, threads):
    from linear_attention_sequence_qkv_gb300.workloads import make_cotangents
    from oracle import oracle as O
    w = inp.w
    flat = lambda x: x.float().reshape(-1, x.shape[-1]).numpy()
    gout, gfin = make_cotangents(inp)
    args = dict(q_raw=flat(inp.q_raw), k_raw=flat(inp.k_raw), v_raw=flat(inp.v_raw), a=flat(inp.a),
                b=flat(inp.b), gate=flat(inp.gate.contiguous()), conv_w=inp.conv_w.float().numpy(),
                A_log=inp.A_log.numpy(), dt_bias=inp.dt_bias.numpy(), norm_w=inp.norm_w.float().numpy(),
                seq_start=inp.seq_starts(), Hk=w.Hk, Hv=w.Hv, dk=w.dk, dv=w.dv,
                initial_state=None if inp.initial_state is None else inp.initial_state.numpy(),
                threads=threads)
    t0 = time.perf_counter()
    O.forward(**args, dtype=w.dtype)
    O.backward(**args, grad_out=gout.float().reshape(-1, w.Hv, w.dv).numpy(), grad_final=gfin.numpy())
    return time.perf_counter() - t0


def backward_main(args, w):
    """One step = gdn_forward + gdn_backward over the workload, inputs and
    cotangents resident in HBM."""
    import torch
    from linear_attention_sequence_qkv_gb300 import build, gdn
    from linear_attention_sequence_qkv_gb300.workloads import make_inputs_device

    cpu = None
    if not args.no_cpu_baseline:
        from oracle import oracle as O
        O.build()
        sinp, w1, nheads = oracle_bwd_sample(w)
        threads = max(1, min(os.cpu_count() or 1, sinp.w.Hk))   # the oracle spreads q/k heads
        dt = run_oracle_fwd_bwd(sinp, threads)
        cpu = {"value": w1.B * w1.T / dt * (nheads / w.Hv), "unit": "tokens/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{w1.B * w1.T} tokens x {nheads}/{w.Hv} v heads of {w.name}, oracle forward + "
                         f"backward, {dt:.2f} s wall, scaled to all heads"}
    build.build()
    gdn.load()
    dev = torch.device("cuda", 0)
    inp = make_inputs_device(w, dev)
    d = gdn.make_desc(inp)
    bufs = gdn.alloc(d, dev)
    grads = gdn.alloc_grads(d, dev)
    B, T = inp.q_raw.shape[0], inp.q_raw.shape[1]
    ntok = B * T
    g = torch.Generator(device=dev).manual_seed(1)
    gout = torch.randn((B, T, w.Hv, w.dv), generator=g, device=dev).to(inp.q_raw.dtype)
    gfin = torch.randn((d.N, w.Hv, w.dk, w.dv), generator=g, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record()
        gdn.forward(inp, bufs, stream)
        if ev:
            ev[1].record()
        gdn.backward(inp, gout, gfin, grads, stream)
        if ev:
            ev[2].record()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(grads.workspace) == gdn.GDN_OK
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = None if args.no_clocks else ClockSampler(None)
    torch.cuda.synchronize()
    for e in evs:
        flush.zero_()
        step(e)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms_f = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    ms_b = sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)
    ms = ms_f + ms_b
    pk_alu = fp32_alu_peak_tflops()
    fl = backward_flops(w, ntok)
    ach = fl / (ms_b / 1e3) / 1e12
    tc = gdn.gdn_chunk_kernel_kind(d) == 1
    # forward: prologue (+ scan), chunk stage, epilogue; backward: prologue (+ scan),
    # chunk matrices, the state recompute and outputs (on the tensor-core path the
    # forward's prep and chain with fp32 stores), RMSNorm backward, dO' terms,
    # reverse chain, (tensor-core dv contractions,) per-chunk gradients, prologue
    # and conv backward, four sums
    scan = 1 if inp.cu_seqlens is not None else 0
    bwd_tc = w.dtype != "fp32" and w.dk in (64, 128, 256) and w.dv % 64 == 0
    launches = (2 + scan + (2 if tc else 1)) + (1 + scan + 9 + (1 if bwd_tc else 0) + 4)

    e2e = None
    if not args.no_e2e:
        names = ["q_raw", "k_raw", "v_raw", "a", "b", "gate_buf", "conv_w", "A_log", "dt_bias", "norm_w"]
        if inp.cu_seqlens is not None:
            names.append("cu_seqlens")
        host = {nm: getattr(inp, nm).cpu().pin_memory() for nm in names}
        host["grad_out"] = gout.cpu().pin_memory()
        host["grad_final"] = gfin.cpu().pin_memory()
        dvc = {nm: torch.empty_like(t, device=dev) for nm, t in host.items()}
        outs = [bufs.out, grads.dq_raw, grads.dk_raw, grads.dv_raw, grads.da, grads.db, grads.dgate,
                grads.dconv_w, grads.dA_log, grads.ddt_bias, grads.dnorm_w, grads.dinitial_state]
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in outs_h)

        class Dev:
            pass
        di = Dev()
        for nm in names:
            setattr(di, nm, dvc[nm])
        di.gate = dvc["gate_buf"][..., : w.Hv * w.dv]
        di.cu_seqlens = dvc.get("cu_seqlens")
        di.initial_state = None
        di.w = w

        def e2e_step():
            for nm, t in host.items():
                dvc[nm].copy_(t, non_blocking=True)
            gdn.forward(di, bufs, stream)
            gdn.backward(di, dvc["grad_out"], dvc["grad_final"], grads, stream)
            for a_, b_ in zip(outs_h, outs):
                a_.copy_(b_, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        k = min(args.steps, 20)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(k):
            e2e_step()
        t1.record()
        torch.cuda.synchronize()
        ms_e2e = t0.elapsed_time(t1) / k
        e2e = {"value": ntok / (ms_e2e / 1e3), "unit": "tokens/s", "ms_per_step": ms_e2e, "steps": k,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "mode": "serial: pinned host inputs and cotangents copied in, forward + backward, "
                       "output and every gradient copied back, per step"}
    line = {
        "metric": "GDN core fwd+bwd tokens/s at 1 GB300", "value": ntok / (ms / 1e3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "bf16": "bf16", "fp16": "f16"}[w.dtype], "data": "synthetic",
        "config": {"workload": f"fwd_bwd_{w.name}", "B": d.B, "T": d.T, "N": d.N, "Hk": w.Hk, "Hv": w.Hv,
                   "dk": w.dk, "dv": w.dv, "tokens_per_step": ntok, "chunk": CHUNK,
                   "l2": "flushed before every timed step (512 MiB write)",
                   "fwd_ms": ms_f, "bwd_ms": ms_b, "bwd_arith": ("state recompute and outputs through the forward's tcgen05 chunk stage; dO' terms "
                                                  "and the per-chunk dv contractions on tcgen05; the rest fp32 CUDA cores"
                                                 if bwd_tc else "fp32 CUDA cores")},
        "roofline": {"bound": "alu", "achieved": ach, "peak": pk_alu, "unit": "TFLOP/s", "frac": ach / pk_alu,
                     "algorithmic_flops": fl, "ms": ms_b, "traffic": None,
                     "kernel": "gdn_backward (recompute, rms, chain, per-chunk, prologue, conv, sums)",
                     "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock"},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches * args.steps, "gpu_launches_per_step": launches, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- split sequence
def spans_main(args, w):
    """One step = the sequence-sharded forward of one sequence split into
    args.spans equal spans, every span's steps (conv prefix, maps A and B,
    span scan, span forward) run one after another on this GPU."""
    import torch
    from linear_attention_sequence_qkv_gb300 import build, context_parallel as cp, gdn
    from linear_attention_sequence_qkv_gb300.workloads import make_inputs_device, replace

    build.build()
    gdn.load()
    dev = torch.device("cuda", 0)
    wb = replace(w, B=1, n_packed=0, T=w.T if not w.n_packed else w.max_len)
    inp = make_inputs_device(wb, dev)
    T = inp.q_raw.shape[1]
    K = args.spans
    cuts = [round(i * T / K) for i in range(K + 1)]
    ts = (inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.conv_w, inp.A_log, inp.dt_bias, inp.norm_w)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        return cp.emulate(*ts, cuts, Hk=wb.Hk, Hv=wb.Hv, dk=wb.dk, dv=wb.dv, initial_state=inp.initial_state)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = None if args.no_clocks else ClockSampler(None)
    for e in evs:
        flush.zero_()
        e[0].record()
        step()
        e[1].record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    # the same sequence unsplit, for the ratio
    d = gdn.make_desc(inp)
    bufs = gdn.alloc(d, dev)
    for _ in range(3):
        gdn.forward(inp, bufs)
    torch.cuda.synchronize()
    evu = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e in evu:
        flush.zero_()
        e[0].record()
        gdn.forward(inp, bufs)
        e[1].record()
    torch.cuda.synchronize()
    ms_unsplit = sum(a.elapsed_time(b) for a, b in evu) / len(evu)
    line = {
        "metric": "GDN core fwd tokens/s, one sequence split into spans, all spans on 1 GB300",
        "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "bf16": "bf16", "fp16": "f16"}[wb.dtype], "data": "synthetic",
        "config": {"workload": f"spans{K}_{w.name}", "T": T, "spans": K, "Hk": wb.Hk, "Hv": wb.Hv, "dk": wb.dk,
                   "dv": wb.dv, "l2": "flushed before every timed step (512 MiB write)",
                   "unsplit_ms": ms_unsplit,
                   "per_span": "2 map forwards (B from zeros; A with v = 0, dv = dk, identity state) + the "
                               "span forward; one gdn_span_scan"},
        "gpu_launches_per_step": None, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# the five workloads the bench line reports (the first is the headline)
ALL_WORKLOADS = ("layer_bf16", "tiny_fp32", "ragged_fp16", "long_gqa_bf16", "varlen_bf16")


def arena(tensors, device, pin=False):
    """One byte buffer holding `tensors` back to back (256-byte aligned), and a view of
    each: a step's inputs (or outputs) then cross the host link as one copy."""
    import torch
    offs, o = [], 0
    for t in tensors:
        o = (o + 255) & ~255
        offs.append(o)
        o += t.numel() * t.element_size()
    buf = torch.empty(o, dtype=torch.uint8, device=device, pin_memory=pin)
    views = [buf[a: a + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for a, t in zip(offs, tensors)]
    return buf, views


def chunk_segments(w, d, inp, nsm):
    """Segments of the tensor-core chunk stage's schedule (1: not segmented): one
    long sequence whose chain CTAs fill at most half of the SMs is cut into up to 16."""
    nch = (d.T + CHUNK - 1) // CHUNK
    tm = w.dtype != "fp32" and w.dk in (64, 128) and w.dv % 128 == 0     # the transposed chain: 128-row dv tiles
    chain_ctas = w.Hv * (w.dv // 128 if tm else w.dv // 64)
    if inp.cu_seqlens is None and d.N == 1 and nch >= 256 and chain_ctas * 2 <= nsm:
        seg = max(-(-nch // 16), 64)
        return -(-nch // seg)
    return 1


def chunk_launch_count(gdn, d, w, inp, nsm):
    """Launches of the chunk stage per step: prep + chain on the tensor-core path
    (two per segment of a long single sequence), one kernel on the fp32 path."""
    if gdn.gdn_chunk_kernel_kind(d) != 1:
        return 1
    return 2 * chunk_segments(w, d, inp, nsm)


def fused_output_step(gdn, d, w, inp, nsm):
    """Whether gdn_forward applies the output step inside the transposed chain (dv = 128,
    a 16-byte-aligned gate view, not the segmented schedule): then it launches no
    separate output kernel."""
    if gdn.gdn_chunk_kernel_kind(d) != 1 or w.dtype == "fp32" or w.dk not in (64, 128) or w.dv != 128:
        return False
    if chunk_launch_count(gdn, d, w, inp, nsm) != 2:
        return False
    g = inp.gate
    return g.data_ptr() % 16 == 0 and (g.stride(1) * g.element_size()) % 16 == 0


def measure_workload(w, steps, warmup, dev, world, barrier, gpu_id, with_clocks, torch, gdn, make_inputs_device):
    """Time one workload: ``steps`` gdn_forward calls (CUDA events around each,
    L2 flushed before each), then the same count as the three stage calls with
    events between them (the per-kernel breakdown). Returns the measurements and
    the device buffers (the headline's end-to-end pass reuses them)."""
    inp = make_inputs_device(w, dev)
    d = gdn.make_desc(inp)
    bufs = gdn.alloc(d, dev)
    ntok = d.B * d.T
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MiB

    def flush_l2():
        # write more than L2 (129 MB), then read another 256 MiB so that L2 is
        # left holding clean lines: the timed kernels then pay no write-back of
        # the flush's dirty lines
        flush.zero_()
        flush_rd.sum()
    stream = torch.cuda.current_stream()

    def fwd_step(ev=None):
        # one gdn_forward: the public call (its kernels back to back on the
        # stream, each a programmatic dependent of the one before)
        if ev:
            ev[0].record()
        gdn.gdn_forward(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.gate, inp.conv_w, inp.A_log,
                        inp.dt_bias, inp.norm_w, inp.cu_seqlens, inp.initial_state, bufs.out, bufs.final_state,
                        bufs.workspace, bufs.ws_bytes, stream)
        if ev:
            ev[1].record()

    def step(ev=None):
        # the same work as three stage calls with events between them (the
        # per-kernel breakdown; no overlap across the stage boundaries)
        if ev:
            ev[0].record()
        gdn.gdn_prologue(d, inp.q_raw, inp.k_raw, inp.v_raw, inp.a, inp.b, inp.conv_w, inp.A_log,
                         inp.dt_bias, inp.cu_seqlens, bufs.workspace, bufs.ws_bytes, stream)
        if ev:
            ev[1].record()
        gdn.gdn_chunk_rule(d, inp.cu_seqlens, inp.initial_state, bufs.final_state, bufs.workspace,
                           bufs.ws_bytes, stream)
        if ev:
            ev[2].record()
        gdn.gdn_epilogue(d, inp.gate, inp.norm_w, bufs.out, bufs.workspace, bufs.ws_bytes, stream)
        if ev:
            ev[3].record()

    for _ in range(warmup):
        flush_l2()
        fwd_step()
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK

    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    sampler = ClockSampler(gpu_id) if with_clocks else None
    torch.cuda.synchronize()
    barrier()
    for i in range(steps):          # the timed steps: gdn_forward
        flush_l2()
        fwd_step(evf[i])
    torch.cuda.synchronize()
    barrier()
    for i in range(steps):          # the per-kernel breakdown: the three stages
        flush_l2()
        step(evs[i])
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop() if sampler else None
    assert gdn.gdn_device_status(bufs.workspace) == gdn.GDN_OK

    per = {"prologue": [], "chunk_rule": [], "epilogue": [], "staged": []}
    for e in evs:
        per["prologue"].append(e[0].elapsed_time(e[1]))
        per["chunk_rule"].append(e[1].elapsed_time(e[2]))
        per["epilogue"].append(e[2].elapsed_time(e[3]))
        per["staged"].append(e[0].elapsed_time(e[3]))
    times = [a.elapsed_time(b) for a, b in evf]
    ms_mean = sum(times) / len(times)
    ms_median = statistics.median(times)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms_mean, ms_median], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_mean, ms_median = float(t[0].item()), float(t[1].item())

    pk = peaks()
    alg = algorithmic(w, ntok, d.N, inp.initial_state is not None)
    kernels = {}
    for name in ("prologue", "chunk_rule", "epilogue"):
        ms = sum(per[name]) / len(per[name])
        kernels[name] = roofline_entry(name, alg[name][0], alg[name][1], ms, pk, w.dtype)
        kernels[name]["ms_median"] = statistics.median(per[name])
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    fused = fused_output_step(gdn, d, w, inp, nsm)
    launches = (1 + (1 if inp.cu_seqlens is not None else 0) + chunk_launch_count(gdn, d, w, inp, nsm) +
                (0 if fused else 1))
    res = {"ms_per_step": ms_mean, "ms_per_step_median": ms_median, "fused_output_step": fused,
           "value": ntok * world / (ms_mean / 1e3), "tokens_per_step": ntok,
           "staged_ms_per_step": sum(per["staged"]) / len(per["staged"]), "kernels": kernels,
           "gpu_launches_per_step": launches, "steps": steps, "warmup": warmup, "clocks": clocks,
           "chunk_kernel": "tcgen05" if gdn.gdn_chunk_kernel_kind(d) == 1 else "cuda-core fp32",
           "shape": {"B": d.B, "T": d.T, "N": d.N, "Hk": w.Hk, "Hv": w.Hv, "dk": w.dk, "dv": w.dv,
                     "dtype": w.dtype}}
    return res, inp, d, bufs, pk, flush_l2, stream


def main():
    args = parse()
    from linear_attention_sequence_qkv_gb300.workloads import WORKLOADS, replace
    w = WORKLOADS[args.workload]
    if args.n_packed and w.n_packed:
        w = replace(w, name=f"{w.name}_n{args.n_packed}", n_packed=args.n_packed)
    if args.impl == "reference":
        reference_arm(args, w)
        return
    if args.decode:
        decode_main(args, w)
        return
    if args.backward:
        backward_main(args, w)
        return
    if args.spans:
        spans_main(args, w)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    # CPU baseline first (host threads only; before any GPU work)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    from linear_attention_sequence_qkv_gb300 import build, gdn
    from linear_attention_sequence_qkv_gb300.workloads import make_inputs_device

    build.build()
    gdn.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    res, inp, d, bufs, pk, flush_l2, stream = measure_workload(
        w, args.steps, args.warmup, dev, world, barrier, gpu_id, not args.no_clocks, torch, gdn,
        make_inputs_device)
    ntok = d.B * d.T
    kernels = res["kernels"]
    tc = res["chunk_kernel"] == "tcgen05"
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    roof = dict(kernels[dom])
    roof["kernel"] = dom
    if dom == "chunk_rule":
        tm = w.dtype != "fp32" and w.dk in (64, 128) and w.dv % 128 == 0
        roof["launches"] = (["chunk_prep_kernel", "chain_tm_kernel" if tm else "chunk_chain_kernel"] if tc
                            else ["chunk_simt_kernel"])
    tr = NCU_TRAFFIC.get(dom)
    roof["traffic"] = None
    if tr is not None:
        src, digest, wl, nbytes = tr
        if wl == w.name and os.path.exists(os.path.join(ROOT, src)) and sha256(os.path.join(ROOT, src)) == digest:
            roof["traffic"] = nbytes
    roof["peak_source"] = pk["source"]

    # end to end through the C ABI with host buffers: pinned H2D of every input,
    # the forward, D2H of the output and the final state, all inside the events.
    # The step's inputs sit in one pinned host arena and cross the host link as one
    # copy; out and final_state share one device arena and come back as one copy
    # (the link moves one large copy at ~210 GB/s and a dozen smaller ones at ~180).
    e2e = None
    if not args.no_e2e:
        names = ["q_raw", "k_raw", "v_raw", "a", "b", "gate_buf", "conv_w", "A_log", "dt_bias", "norm_w"]
        if inp.cu_seqlens is not None:
            names.append("cu_seqlens")
        if inp.initial_state is not None:
            names.append("initial_state")
        srcs = [getattr(inp, nm) for nm in names]
        h_in, hv = arena(srcs, "cpu", pin=True)
        for v, t in zip(hv, srcs):
            v.copy_(t)
        h_out, _ = arena([bufs.out, bufs.final_state], "cpu", pin=True)
        h2d = h_in.numel()
        d2h = h_out.numel()
        ksteps = min(args.steps, 100)
        ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(ksteps)]

        def dev_buffers():
            d_in, views = arena(srcs, dev)
            d_out, (o_, f_) = arena([bufs.out, bufs.final_state], dev)
            return d_in, dict(zip(names, views)), d_out, o_, f_

        def forward_on(b_, o_, f_):
            gdn.gdn_forward(d, b_["q_raw"], b_["k_raw"], b_["v_raw"], b_["a"], b_["b"],
                            b_["gate_buf"][..., : w.Hv * w.dv], b_["conv_w"], b_["A_log"], b_["dt_bias"],
                            b_["norm_w"], b_.get("cu_seqlens"), b_.get("initial_state"), o_, f_,
                            bufs.workspace, bufs.ws_bytes, stream)

        bset = [dev_buffers(), dev_buffers()]

        def e2e_step(e):
            d_in, b_, d_out, o_, f_ = bset[0]
            e[0].record()
            d_in.copy_(h_in, non_blocking=True)
            forward_on(b_, o_, f_)
            h_out.copy_(d_out, non_blocking=True)
            e[1].record()

        for _ in range(3):
            e2e_step(ev2[0])
        torch.cuda.synchronize()
        barrier()
        for i in range(ksteps):
            flush_l2()
            e2e_step(ev2[i])
        torch.cuda.synchronize()
        barrier()
        ms_e2e = sum(a.elapsed_time(b) for a, b in ev2) / ksteps
        if world > 1:
            t = torch.tensor([ms_e2e], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms_e2e = float(t.item())
        serial = {"value": ntok * world / (ms_e2e / 1e3), "ms_per_step": ms_e2e, "steps": ksteps,
                  "l2": "flushed before every step"}

        # Pipelined: the copy of step i+1 overlaps the kernels of step i and the
        # read-back of step i-1 (a copy-in stream, the compute stream, a read-back
        # stream; inputs and outputs double-buffered on the device). Every step still
        # copies its inputs from pinned host memory and reads its output and final
        # state back.
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer k copied
        ev_used = [torch.cuda.Event() for _ in range(2)]   # kernels done with buffer k
        ev_read = [torch.cuda.Event() for _ in range(2)]   # outputs k copied back

        def pipe_step(i):
            k = i % 2
            d_in, b_, d_out, o_, f_ = bset[k]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_used[k])
                d_in.copy_(h_in, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i >= 2:
                stream.wait_event(ev_read[k])
            forward_on(b_, o_, f_)
            ev_used[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_used[k])
                h_out.copy_(d_out, non_blocking=True)
                ev_read[k].record(s_out)

        for i in range(4):
            pipe_step(i)
        torch.cuda.synchronize()
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        s_in.wait_event(t0)
        for i in range(ksteps):
            pipe_step(i + 4)
        t1.record(s_out)   # after the last read-back
        torch.cuda.synchronize()
        barrier()
        ms_pipe = t0.elapsed_time(t1) / ksteps
        if world > 1:
            t = torch.tensor([ms_pipe], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms_pipe = float(t.item())
        e2e = {"value": ntok * world / (ms_pipe / 1e3), "unit": "tokens/s", "ms_per_step": ms_pipe,
               "steps": ksteps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "mode": "pipelined: each step's host-to-device copy overlaps the previous step's "
                       "kernels and read-back (a copy-in stream, the compute stream, a read-back "
                       "stream; double-buffered device inputs, outputs and final states); the "
                       "step's inputs are one pinned host arena copied in one piece, out and "
                       "final_state one device arena read back in one piece; timed from the "
                       "first copy to the last read-back",
               "serial": serial}
        # the outputs that crossed the link are the forward's
        o_chk = h_out[: bufs.out.numel() * bufs.out.element_size()].view(bufs.out.dtype).view(bufs.out.shape)
        e2e["readback_matches_device"] = bool(torch.equal(o_chk.to(dev), bset[(ksteps + 3) % 2][3]))
    del bufs, inp

    # the other workloads, each measured the same way in this run (one GPU only)
    workloads = {}
    if world == 1 and not args.no_workloads:
        for name in ALL_WORKLOADS:
            wk = WORKLOADS[name]
            if name == w.name:
                r = dict(res)
            else:
                r, _i, _d, _b, _p, _f, _s = measure_workload(
                    wk, min(args.steps, args.workload_steps), min(args.warmup, 5), dev, world, barrier, gpu_id,
                    not args.no_clocks, torch, gdn, make_inputs_device)
                del _i, _b
                torch.cuda.empty_cache()
            r = {k: v for k, v in r.items() if k != "value"} | {"tokens_per_s": r["value"]}
            workloads[name] = r

    line = {
        "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "ms_per_step_median": res["ms_per_step_median"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "bf16": "bf16", "fp16": "f16"}[w.dtype], "data": "synthetic",
        "config": {"workload": w.name, "B": d.B, "T": d.T, "N": d.N, "Hk": w.Hk, "Hv": w.Hv,
                   "dk": w.dk, "dv": w.dv, "tokens_per_step": ntok, "chunk": CHUNK,
                   "l2": "flushed before every timed step (512 MiB write, then 256 MiB read)",
                   "parallelism": f"replicas x{world}",
                   "chunk_kernel": res["chunk_kernel"],
                   "timing": "value: one gdn_forward per step, CUDA events around the call, mean over the "
                             "steps (ms_per_step_median beside it); kernels: the same work as gdn_prologue / "
                             "gdn_chunk_rule / gdn_epilogue with events between them, a second pass of the "
                             "same step count (where a workload's fused_output_step is true, gdn_forward runs the "
                             "output step inside the chunk kernel instead of the separate output kernel the "
                             "stage calls time)",
                   "staged_ms_per_step": res["staged_ms_per_step"]},
        "roofline": roof,
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": res["gpu_launches_per_step"] * args.steps,
        "gpu_launches_per_step": res["gpu_launches_per_step"],
        "clocks": res["clocks"],
        "workloads": workloads,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
