#!/usr/bin/env python
"""Benchmark of the Memory Caching forward on GB300.

One step = one full forward (segment states, online reads, gates, cached
readout, y) over one batch of synthetic input already resident in HBM.
Default workload: long-context MC-GRM, B=1 H=16 L=65536 d=128 seg_len=1024
(N=64), bf16 inputs, fp32 states.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) shard nothing: each
rank runs its own copy of the workload (independent (batch, head) problems,
no collective on the data path) and the value is all ranks' tokens over the
slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mc_inputs  # noqa: E402
from mc_inputs import GRM, RESIDUAL, SSC  # noqa: E402

METRIC = "tokens/sec MC-GRM forward (L=64K,d=128,N=64) on 1 GB300; % bf16 TC peak"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
SMS = 152
FP32_LANES_PER_SM = 128
SM_MAX_GHZ = 2.07


# ----------------------------------------------------------------------------- algorithmic work

def segment_counts(w):
    """Per-token (s_t = 1-based segment number, n_t = cached segments read)."""
    C, L = w.seg_len, w.L
    s = [t // C + 1 for t in range(L)]
    if w.mode == RESIDUAL:
        n = [0] * L  # linear memory: the cached sum collapses into one fixed memory
    elif w.mode == SSC:
        n = [min(w.topk, st - 1) for st in s]
    else:
        n = [st - 1 for st in s]
    return s, n


def factorised_reads(w):
    """Per head, sum over tokens of the earlier tokens the factorised readout must read:
    y_t = sum_j g_{t,seg(j)} v_j (k_j . q_t) over j <= t in the memories token t reads
    (every earlier token for GRM / Soup / Mean and for Residual's plain causal sum; for
    SSC its own segment's tokens up to t and the topk selected segments)."""
    C, L = w.seg_len, w.L
    if w.mode != SSC:
        return L * (L + 1) // 2
    tot = 0
    for t in range(L):
        s = t // C
        tot += min(w.topk, s) * C + (t - s * C + 1)
    return tot


def algorithmic_flops(w):
    """Per step, all heads.  State form (the segment-state and readout kernels): online
    write + read (4 d^2 per token), cached reads (2 d^2 per token and cached segment read),
    gate scores (2 d per token and score).  Factorised form (the piece-state, gate and
    factorised readout kernels): the cached states written (2 d^2 per token), 4 d per token
    and earlier token read (k_j . q_t, then v_j times it), the same gate scores.  The
    method's work ("total") is the smaller of the two; each kernel is credited with its
    own form's share."""
    s, n = segment_counts(w)
    d = w.d
    bh = w.B * w.H
    per_head_online = w.L * 4 * d * d
    per_head_cached = 2 * d * d * sum(n)
    per_head_gate = 0 if w.mode in (RESIDUAL, mc_inputs.MEAN) else 2 * d * sum(s)
    state_form = per_head_online + per_head_cached + per_head_gate
    fact_read = 4 * d * factorised_reads(w)
    fact_form = w.L * 2 * d * d + fact_read + per_head_gate
    return {"total": bh * min(state_form, fact_form),
            "state_form": bh * state_form, "factorised_form": bh * fact_form,
            "online": bh * per_head_online,
            "state": bh * per_head_online // 2,
            "readout": bh * (per_head_online // 2 + per_head_cached + per_head_gate),
            "seg_state_tc": bh * per_head_online // 2,
            "readout_tc": bh * (per_head_online // 2 + per_head_cached + per_head_gate),
            "seg_piece_tc": bh * w.L * 2 * d * d,
            "gates_tc": bh * per_head_gate,
            "readout_fact_tc": bh * fact_read}


def algorithmic_bytes(w):
    elt = 2 if w.dtype == "bf16" else 4
    bh = w.B * w.H
    n_in = 4 if w.mode != RESIDUAL else 3
    return bh * (w.L * w.d * elt * (n_in + 1) + w.N * w.d * w.d * 4)


def kernel_bytes(w):
    """Algorithmic bytes per launch of each tensor-core kernel, given the split of the
    step between them: what each must read and write at least.  The segment-state
    kernels read k, v (and u for the routed aggregations) and write the fp32 states;
    the state-form readout reads q, k, v (u), every cached state once as a bf16 operand,
    and writes y; the gate kernel reads u and writes the bf16 gates; the factorised
    readout reads q, k, v and the gates and writes y.  Scratch images that only pass
    between the kernels are not counted."""
    elt = 2 if w.dtype == "bf16" else 4
    bh = w.B * w.H
    row = w.L * w.d * elt
    routed = w.mode not in (RESIDUAL, mc_inputs.MEAN)
    # u is read for the tokens after the first segment only: those before have one memory,
    # whose gate is 1 whatever the score
    urow = (w.L - min(w.seg_len, w.L)) * w.d * elt if routed else 0
    st32 = w.N * w.d * w.d * 4
    s, _ = segment_counts(w)
    gate_bytes = 2 * (sum(s)) if routed else 0  # bf16 gates, one per token and memory it reads
    return {"seg_state_tc": bh * (2 * row + urow + st32),
            "readout_tc": bh * (4 * row + urow + st32 // 2),
            "seg_piece_tc": bh * ((3 if routed else 2) * row + st32),
            "gates_tc": bh * (row + gate_bytes),
            "readout_fact_tc": bh * (4 * row + gate_bytes)}


def workload_bound(w, peaks):
    """'tensor' when the algorithmic flops at the bf16 peak take longer than the algorithmic
    bytes at the HBM peak, else 'hbm'."""
    t_tc = algorithmic_flops(w)["total"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = algorithmic_bytes(w) / (peaks["hbm_gbs"] * 1e9)
    return "tensor" if t_tc >= t_hbm else "hbm"


def metric_name(w):
    if w == mc_inputs.LONG_GRM:
        return METRIC
    return f"tokens/sec MC-{mc_inputs.MODE_NAMES[w.mode].upper()} forward ({w.name}) on 1 GB300"


# ----------------------------------------------------------------------------- peaks and clocks

_CSRC = "memory_caching_linear_gb300/csrc/"
# the sources each tensor-core kernel is built from: the state-form path, and the general path
KERNEL_SOURCES = tuple(_CSRC + f for f in ("k_tc.cu", "k_tc64.cu", "tc_state_form.cuh", "sm100.cuh",
                                           "tc_common.cuh", "tensormap.cuh", "mc_internal.cuh"))
GEN_KERNEL_SOURCES = tuple(_CSRC + f for f in ("k_gen.cu", "sm100.cuh", "tc_common.cuh", "tensormap.cuh",
                                               "mc_internal.cuh"))
GEN_KERNELS = ("seg_piece_tc", "gates_tc", "readout_fact_tc")


def kernel_source_hash(kernel: str = "readout_tc") -> str:
    """sha256 over the sources `kernel` is built from, in a fixed order."""
    h = hashlib.sha256()
    for rel in (GEN_KERNEL_SOURCES if kernel in GEN_KERNELS else KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu summary
    profiles/<kernel>_<workload>.md, or None when there is none or the kernel's sources
    changed after the counters were taken (the summary records their hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-").strip()
        if ":" in line:
            key, _, val = line.partition(":")
            fields[key.strip().strip("`")] = val.strip().strip("`")
    try:
        if fields.get("kernel_source_sha256") != kernel_source_hash(kernel):
            return None
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError, OSError):
        return None


L2_BYTES = 129 * 10**6
FLUSH_BYTES = 256 * 2**20  # written between timed steps when the inputs would stay in L2


def l2_note(inputs_bytes):
    """How the timed steps treat the L2 for inputs of this size (see timed_steps)."""
    gib = inputs_bytes / 2**30
    if inputs_bytes > 2 * L2_BYTES:
        return f"inputs {gib:.2f} GiB > L2 129 MB, not flushed"
    return f"inputs {gib:.3f} GiB fit in L2: 256 MiB written before every timed step (not timed)"


def forward_inputs_bytes(w):
    """Bytes of q, k, v, u of a forward workload."""
    return 4 * w.B * w.H * w.L * w.d * (2 if w.dtype == "bf16" else 4)


def forward_config(w, world, note):
    """The `config` object of a forward workload's JSON line (both arms)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "seg_len": w.seg_len, "N": w.N,
            "agg": mc_inputs.MODE_NAMES[w.mode], "topk": w.topk, "input_dtype": w.dtype, "l2": note,
            "parallelism": f"replicas x{world} (independent (batch, head) problems)"}


def timed_steps(step, steps, inputs_bytes):
    """Run `steps` calls of step() and return (ms, l2 note).  Inputs larger than twice the
    L2 run back to back between two events on the current stream; smaller ones get a
    256 MiB write before every call (the L2 holds none of the inputs when a call starts)
    and events around each call, whose times are summed."""
    import torch
    stream = torch.cuda.current_stream()
    if inputs_bytes > 2 * L2_BYTES:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1), l2_note(inputs_bytes)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=torch.device("cuda", torch.cuda.current_device()))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(evs):
        flush.fill_(i & 0xFF)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs), l2_note(inputs_bytes)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return self
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return self

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, dist=None) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * steps * world / (max_ms / 1e3)


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(w, budget_s: float, steps_hint: int = 1):
    """Time the fp64 oracle, as it stands, on a bounded sample of workload w:
    heads 0..P-1 (P = host cores, capped at B*H), and S segments spread evenly
    over the sequence (S chosen to fit the time budget), full d and L.  Returns
    (tokens/s, cores, description)."""
    import numpy as np
    import oracle
    cores = os.cpu_count() or 1
    bh = min(cores, w.B * w.H)
    q, k, v, u = mc_inputs.make_inputs(1, bh, w.L, w.d, w.seed, w.dtype)
    q, k, v, u = (t.float().numpy() for t in (q, k, v, u))
    sw = tuple(t.numpy() for t in mc_inputs.make_swla_scalars(1, bh, w.L, w.seed)) if w.swla else None
    picks = [w.N // 2] if w.N < 4 else [int((i + 0.5) * w.N / 4) for i in range(4)]
    # probe with one segment, then size the sample to the budget
    mask = np.zeros(w.N, bool)
    mask[picks[0]] = True
    t0 = time.perf_counter()
    oracle.forward(q, k, v, u, w.seg_len, w.mode, w.topk, seg_mask=mask, nthreads=cores, swla=sw)
    t_one = time.perf_counter() - t0
    nseg = max(1, min(len(picks), int(budget_s / max(t_one, 1e-3))))
    chosen = picks[:nseg] if nseg < len(picks) else picks
    mask = np.zeros(w.N, bool)
    mask[chosen] = True
    t0 = time.perf_counter()
    oracle.forward(q, k, v, u, w.seg_len, w.mode, w.topk, seg_mask=mask, nthreads=cores, swla=sw)
    dt = time.perf_counter() - t0
    ntok = sum(min(w.L, (n + 1) * w.seg_len) - n * w.seg_len for n in chosen)
    # tokens/s in the metric's unit: a token is one sequence position across all H heads
    rate = ntok * bh / dt / w.H
    desc = (f"fp64 oracle, heads 0..{bh - 1} of B*H={w.B * w.H}, segments {chosen} of N={w.N} "
            f"({ntok} positions x {bh} heads, all segment states computed), {dt:.1f} s wall; "
            f"tokens/s = positions*heads/time/H")
    return rate, cores, desc, dt


# ----------------------------------------------------------------------------- our arm

def run_ours(args, w, wname="long-grm"):
    import numpy as np
    import torch
    import torch.distributed as dist

    import memory_caching_linear_gb300 as mcl
    from memory_caching_linear_gb300 import build as mcbuild

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    mcbuild.build()
    mcl.load_library()

    q, k, v, u = mc_inputs.workload_inputs(w, device=dev)
    torch.cuda.synchronize()
    y = torch.empty_like(q)
    states = torch.empty((w.B, w.H, w.N, w.d, w.d), dtype=torch.float32, device=dev)
    fwd = mcl.mc_forward if w.dtype == "bf16" else mcl.mc_forward_f32
    sw = mc_inputs.workload_swla_scalars(w, device=dev) if w.swla else None

    def step():
        if sw is not None:
            mcl.mc_forward_swla(q, k, v, u, *sw, w.seg_len, w.mode, w.topk, y=y, states=states)
        else:
            fwd(q, k, v, u, w.seg_len, w.mode, w.topk, y=y, states=states)

    # warm-up (at least W steps and ~1 s so the clocks settle under load)
    sampler = ClockSampler(dev.index).start()
    time.sleep(0.4)
    t_w = time.perf_counter()
    nwarm = 0
    while nwarm < args.warmup or time.perf_counter() - t_w < args.warmup_seconds:
        step()
        torch.cuda.synchronize()
        nwarm += 1
        if nwarm > 10000:
            break

    if world > 1:
        dist.barrier()
    in_bytes = forward_inputs_bytes(w)
    ms, note = timed_steps(step, args.steps, in_bytes)
    if world > 1:
        dist.barrier()
    # Per-kernel times come from a second pass of the same K steps with events
    # between the kernels (the events keep consecutive kernels from overlapping,
    # so that pass is not the headline).
    prof = mcl.KernelProfile(capacity=args.steps * 8 + 8)
    with prof:
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
    sampler.stop()
    max_ms = reduce_max(ms, dist if world > 1 else None)
    value = aggregate(w.tokens, args.steps, max_ms, world)

    per_kernel = prof.per_kernel_ms()
    launches = prof.kernel_count()
    peaks = measured_peaks()
    flops = algorithmic_flops(w)

    # dominant kernel and its roofline
    dom = max(per_kernel.items(), key=lambda kv: sum(kv[1])) if per_kernel else (None, [])
    dom_name, dom_ms = dom
    roof = None
    kernels_ms = {n: round(sum(t) / len(t), 4) for n, t in per_kernel.items()}
    dtype_path = "f32"
    kbytes = kernel_bytes(w)
    if dom_name and "tc" in dom_name and workload_bound(w, peaks) == "hbm" and dom_name in kbytes:
        avg_ms = sum(dom_ms) / len(dom_ms)
        dtype_path = "bf16"
        achieved = kbytes[dom_name] / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(dom_name, wname), "kernel": dom_name,
                "launch_ms": round(avg_ms, 4), "algorithmic_bytes_per_launch": kbytes[dom_name],
                "peak_source": f"HBM copy ({peaks['source']})"}
    elif dom_name:
        avg_ms = sum(dom_ms) / len(dom_ms)
        tensor = "tc" in dom_name
        dtype_path = "bf16" if tensor else "f32"
        work = flops.get(dom_name, flops["readout"] if "readout" in dom_name else flops["state"])
        achieved = work / (avg_ms / 1e3) / 1e12
        if tensor:
            sustained = max_ms > 1000.0
            peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
            psrc = f"bf16 {'sustained' if sustained else 'burst'} ({peaks['source']})"
            bound = "tensor"
        else:
            peak = SMS * FP32_LANES_PER_SM * 2 * SM_MAX_GHZ / 1e3
            psrc = "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz"
            bound = "alu"
        roof = {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(dom_name, wname), "kernel": dom_name,
                "launch_ms": round(avg_ms, 4), "algorithmic_tflop_per_launch": round(work / 1e12, 4),
                "peak_source": psrc}

    clocks = sampler.summary()
    step_s = max_ms / 1e3 / args.steps
    res = {
        "metric": metric_name(w), "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": nwarm, "ms_per_step": round(max_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_path,
        "data": "synthetic (seeded numpy normals: q,k unit rows, v ~ N(0,1), u ~ N(0,1)/sqrt(d)"
                + ("; SWLA alpha = 1 - 0.1 sigmoid(z), beta, lambda = sigmoid(z))" if w.swla else ")"),
        "config": forward_config(w, world, note),
        "tc_fraction_of_bf16_peak": round(flops["total"] / step_s / 1e12 / peaks["bf16_tflops"], 4),
        "algorithmic_tflop_per_step": round(flops["total"] / 1e12, 4),
        "hbm_fraction": round(algorithmic_bytes(w) / step_s / 1e9 / peaks["hbm_gbs"], 4),
        "roofline": roof,
        "kernels_ms": kernels_ms,
        "gpu_launches": launches,
        "clocks": clocks,
    }

    # end to end through the host-buffer entry point (plain update only)
    if not args.no_e2e and not w.swla:
        qh, kh, vh, uh = (t.cpu().pin_memory() for t in (q, k, v, u))
        yh = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        for _ in range(3):  # first touches of the pinned pages and the device pool
            mcl.mc_forward_host(qh, kh, vh, uh, w.seg_len, w.mode, w.topk, y=yh)
        ksteps = max(1, min(args.steps, 10))
        if world > 1:
            dist.barrier()
        call_ms = []
        t0 = time.perf_counter()
        for _ in range(ksteps):
            t1 = time.perf_counter()
            mcl.mc_forward_host(qh, kh, vh, uh, w.seg_len, w.mode, w.topk, y=yh)
            call_ms.append((time.perf_counter() - t1) * 1e3)
        e2e_ms = (time.perf_counter() - t0) * 1e3
        e2e_max = reduce_max(e2e_ms, dist if world > 1 else None)
        elt = 2 if w.dtype == "bf16" else 4
        nin = 4 if w.mode != RESIDUAL else 3
        res["e2e"] = {"value": round(aggregate(w.tokens, ksteps, e2e_max, world), 1), "unit": UNIT,
                      "h2d_bytes_per_step": nin * q.numel() * elt, "d2h_bytes_per_step": y.numel() * elt,
                      "steps": ksteps, "warmup": 3, "call_ms": [round(x, 3) for x in call_ms],
                      "api": "mc_forward_host (pinned host buffers)"}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, desc, _ = oracle_sample(w, budget_s=args.cpu_budget)
        res["cpu_baseline"] = {"value": round(rate, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": desc}
    if world > 1:
        dist.destroy_process_group()
    return res if rank == 0 else None


def run_decode(args):
    """One recurrent decoding step (mc_decode_step) per sequence: B = 8, H = 16, d = 128,
    seg_len = 1024, position 63*1024 + 512 (63 cached segments, mid-segment), GRM.  The
    step reads every cached fp32 state once: reported against HBM."""
    import torch
    import memory_caching_linear_gb300 as mcl
    from memory_caching_linear_gb300 import build as mcbuild
    mcbuild.build()
    mcl.load_library()
    B, H, d, C, nmax = 8, 16, 128, 1024, 64
    t = 63 * C + 512
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device="cpu").manual_seed(6)
    cache = mcl.DecodeCache(B, H, d, C, nmax, device=dev)
    cache.states.copy_(torch.randn(cache.states.shape, generator=g) / d)
    cache.kbar.copy_(torch.nn.functional.normalize(torch.randn(cache.kbar.shape, generator=g), dim=-1))
    cache.online.copy_(torch.randn(cache.online.shape, generator=g) / d)
    cache.ksum.copy_(torch.randn(cache.ksum.shape, generator=g))
    q, k, v, u = (x[:, :, 0, :].contiguous() for x in mc_inputs.make_inputs(B, H, 1, d, 6, "bf16", device=dev))
    y = torch.empty_like(q)

    def step():
        cache.t = t
        mcl.mc_decode_step(cache, q, k, v, u, GRM, y=y)

    sampler = ClockSampler(dev.index).start()
    for _ in range(max(args.warmup, 50)):
        step()
    torch.cuda.synchronize()
    steps = max(args.steps, 200)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(steps):
        step()
    ev1.record()
    torch.cuda.synchronize()
    sampler.stop()
    ms = ev0.elapsed_time(ev1) / steps
    s_cached = t // C
    bytes_step = B * H * (s_cached * d * d * 4 + 2 * d * d * 4 + s_cached * d * 4 + 3 * d * 2)
    peak = measured_peaks()["hbm_gbs"]
    achieved = bytes_step / (ms / 1e3) / 1e9
    return {
        "metric": "tokens/sec MC-GRM decode step (d=128, 63 cached segments)", "value": round(B / (ms / 1e3), 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": max(args.warmup, 50),
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (random fp32 caches, seeded bf16 token)",
        "config": {"workload": f"decode-grm B{B} H{H} d{d} C{C} t={t}", "B": B, "H": H, "d": d, "seg_len": C,
                   "cached_segments": s_cached},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "decode_gates + decode_read", "algorithmic_bytes_per_step": bytes_step},
        "gpu_launches": 2 * steps, "clocks": sampler.summary(),
    }


def backward_flops(w):
    """Algorithmic work of the backward (all heads), in total and per kernel.  Per token and
    cached read: the read's value M q (2 d^2, needed for the gate gradient and not kept by
    the forward), dq (2 d^2) and the state gradient dy q^T (2 d^2); per token, twice the
    online write + read (8 d^2); per token and score, the score gradients du and the
    key-mean gradient (4 d).  Per kernel: the tensor-core cached pass does M q and dq of
    the cached reads, the G kernels the state gradients, the FFMA gate kernel the score
    gradients (and, without the tensor-core pass, the cached M q and dq too), the route
    kernel du and the key-mean kernel dkbar (half the score gradients each; the key-mean
    kernel runs on the tensor cores on the tensor-core path), the segment
    scan the online write and read (4 d^2 per token and run), the reverse scan / the
    tensor-core dk, dv kernel the online gradients (6 d^2 per token), the state kernel the
    online write (2 d^2 per token); the tensor-core gates kernel recomputes the router's
    scores (2 d per token and cached segment: forward work, outside the total)."""
    s, n = segment_counts(w)
    bh = w.B * w.H
    d = w.d
    routed = w.mode not in (RESIDUAL, mc_inputs.MEAN)
    score = 4 * d * sum(s) if routed else 0
    cached = 4 * d * d * sum(n)
    return {"total": bh * (6 * d * d * sum(n) + 8 * d * d * w.L + score),
            "bwd_cached_tc": bh * cached, "bwd_gates_simt": bh * (cached + score),
            "bwd_route_simt": bh * score // 2, "bwd_dkbar_simt": bh * score // 2, "bwd_dkbar_tc": bh * score // 2,
            "bwd_G_tc": bh * 2 * d * d * sum(n), "bwd_G_simt": bh * 2 * d * d * sum(n),
            "seg_scan_simt": bh * 4 * d * d * w.L, "bwd_scan_simt": bh * 6 * d * d * w.L,
            "bwd_kv_tc": bh * 6 * d * d * w.L, "seg_state_tc": bh * 2 * d * d * w.L,
            "gate_tiles_tc": bh * 2 * d * sum(st - 1 for st in s) if routed else 0}


def run_backward(args, w, wname):
    """The backward pass (mc_backward) on a forward workload: gradients of <y, dy> for
    seeded dy, inputs resident on the device; K timed steps with CUDA events."""
    import torch
    import memory_caching_linear_gb300 as mcl
    from memory_caching_linear_gb300 import build as mcbuild
    mcbuild.build()
    mcl.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, u = mc_inputs.workload_inputs(w, device=dev)
    g = torch.Generator(device="cpu").manual_seed(w.seed + 101)
    dy = torch.randn(q.shape, generator=g).to(device=dev, dtype=q.dtype)
    grads = [torch.empty_like(q) for _ in range(4)]

    def step():
        mcl.mc_backward(q, k, v, u, dy, w.seg_len, w.mode, w.topk, dq=grads[0], dk=grads[1], dv=grads[2],
                        du=grads[3])

    sampler = ClockSampler(dev.index).start()
    nwarm = max(args.warmup, 3)
    for _ in range(nwarm):
        step()
    torch.cuda.synchronize()
    tot_ms, note = timed_steps(step, args.steps, 5 * q.numel() * q.element_size())
    prof = mcl.KernelProfile(capacity=args.steps * 8 + 8)
    with prof:
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
    sampler.stop()
    ms = tot_ms / args.steps
    per_kernel = prof.per_kernel_ms()
    kernels_ms = {n: round(sum(t) / len(t) * (len(t) / args.steps), 4) for n, t in per_kernel.items()}
    flops = backward_flops(w)
    dom = max(kernels_ms, key=kernels_ms.get)
    dom_ms = kernels_ms[dom]
    key = dom
    # the segment scan runs twice per step (states and O_on, then M_t^T dy_t): its time is the sum
    work = flops[key] * (2 if dom == "seg_scan_simt" else 1)
    tensor = dom.endswith("_tc")
    if tensor:
        peaks = measured_peaks()
        peak, psrc, bound = peaks["bf16_tflops"], f"bf16 burst ({peaks['source']})", "tensor"
    else:
        peak, psrc, bound = SMS * FP32_LANES_PER_SM * 2 * SM_MAX_GHZ / 1e3, \
            "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz", "alu"
    achieved = work / (dom_ms / 1e3) / 1e12 if dom_ms else 0.0
    return {
        "metric": f"tokens/sec MC-{mc_inputs.MODE_NAMES[w.mode].upper()} backward ({w.name})",
        "value": round(w.tokens / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": nwarm, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16+f32" if "bwd_cached_tc" in kernels_ms else "f32",
        "data": "synthetic (the forward workload's seeded inputs; dy ~ N(0, 1))",
        "config": {"workload": f"bwd-{wname} {w.name}", "B": w.B, "H": w.H, "L": w.L, "d": w.d, "seg_len": w.seg_len,
                   "N": w.N, "agg": mc_inputs.MODE_NAMES[w.mode], "input_dtype": w.dtype,
                   "l2": note},
        "algorithmic_tflop_per_step": round(flops["total"] / 1e12, 4),
        "roofline": {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "kernel": dom, "launch_ms": dom_ms,
                     "algorithmic_tflop_per_launch": round(work / 1e12, 4), "peak_source": psrc},
        "kernels_tflops": {n: round(flops.get(n, 0) * (2 if n == "seg_scan_simt" else 1) / (t / 1e3) / 1e12, 2)
                           for n, t in kernels_ms.items() if t},
        "kernels_ms": kernels_ms, "gpu_launches": prof.kernel_count() // max(args.steps, 1) * args.steps,
        "clocks": sampler.summary(),
    }


LOGLINEAR = mc_inputs.Workload("loglinear-grm B1 H16 L65535 d128 log-segments bf16", 1, 16, 65535, 128, 65535, GRM,
                               "bf16", seed=7)


def run_segments(args):
    """Log-Linear++: GRM over the logarithmic segmentation of L = 65535 (16 segments of
    32768, 16384, ..., 1 tokens), B1 H16 d128 bf16, through mc_forward_segments."""
    import torch
    import memory_caching_linear_gb300 as mcl
    from memory_caching_linear_gb300 import build as mcbuild
    mcbuild.build()
    mcl.load_library()
    w = LOGLINEAR
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, u = mc_inputs.workload_inputs(w, device=dev)
    off = mcl.log_segments(w.L)
    lens = [b - a for a, b in zip(off[:-1], off[1:])]
    y = torch.empty_like(q)
    states = torch.empty((w.B, w.H, len(lens), w.d, w.d), dtype=torch.float32, device=dev)

    def step():
        mcl.mc_forward_segments(q, k, v, u, off, w.mode, y=y, states=states)

    sampler = ClockSampler(dev.index).start()
    nwarm = max(args.warmup, 3)
    for _ in range(nwarm):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    prof = mcl.KernelProfile(capacity=args.steps * 8 + 8)
    with prof:
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
    sampler.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    kernels_ms = {n: round(sum(t) / args.steps, 4) for n, t in prof.per_kernel_ms().items()}
    # algorithmic work per head: L 4 d^2 + 2 d^2 sum_t n_t + 2 d sum_t (n_t + 1), n_t = cached segments of t;
    # the segments that are whole 128-token chunks run on the tensor cores, the tail on the CUDA cores
    bh, d = w.B * w.H, w.d
    nbig = 0
    while nbig < len(lens) and off[nbig] % 128 == 0 and lens[nbig] % 128 == 0:
        nbig += 1
    if off[nbig] + 128 <= w.L:
        nbig = 0  # the CUDA-core path for all
    l_big = off[nbig]

    def read_flops(segs):
        toks = sum(lens[i] for i in segs)
        cached = sum(i * lens[i] for i in segs)
        return bh * (toks * 2 * d * d + 2 * d * d * cached + 2 * d * (cached + toks))

    big, tail = range(nbig), range(nbig, len(lens))
    f_state = bh * w.L * 2 * d * d
    work_of = {"seg_state_tc": bh * l_big * 2 * d * d, "readout_tc": read_flops(big),
               "seg_scan_simt": bh * (w.L - l_big) * 2 * d * d, "readout_simt": read_flops(tail),
               "tail_readout_simt": read_flops(tail)}
    dom = max(kernels_ms, key=kernels_ms.get)
    work = work_of.get(dom, 0)
    if dom.endswith("_tc"):
        peaks = measured_peaks()
        bound, peak = "tensor", peaks["bf16_tflops"]
        psrc = f"bf16 burst ({peaks['source']})"
    else:
        bound, peak = "alu", SMS * FP32_LANES_PER_SM * 2 * SM_MAX_GHZ / 1e3
        psrc = "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz"
    achieved = work / (kernels_ms[dom] / 1e3) / 1e12
    return {
        "metric": "tokens/sec Log-Linear++ (MC-GRM, logarithmic segments) forward", "value": round(w.tokens / (ms / 1e3), 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": nwarm, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if nbig else "f32",
        "data": "synthetic (seeded numpy normals: q,k unit rows, v ~ N(0,1), u ~ N(0,1)/sqrt(d))",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "segments": lens, "agg": "grm",
                   "input_dtype": w.dtype, "tensor_core_segments": nbig,
                   "l2": "inputs 1.00 GiB > L2 129 MB, not flushed"},
        "algorithmic_tflop_per_step": round((f_state + read_flops(range(len(lens)))) / 1e12, 4),
        "roofline": {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None, "kernel": dom, "launch_ms": kernels_ms[dom],
                     "algorithmic_tflop_per_launch": round(work / 1e12, 4), "peak_source": psrc},
        # stages of several launches: the tail readout (gates, partials, finish) and, on the CUDA-core
        # path with segments longer than 512 tokens, the piece-split scan (scan, piece prefix, fix-up)
        "kernels_ms": kernels_ms, "gpu_launches": prof.kernel_count() + 2 * prof.stages.count("tail_readout_simt") + (
            2 * prof.stages.count("seg_scan_simt") if (not nbig and max(lens) > 512) else 0),
        "clocks": sampler.summary(),
    }


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    budget = max(1.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, budget_s=budget)
    t0 = time.perf_counter()
    rates = []
    desc = ""
    cores = os.cpu_count() or 1
    for _ in range(args.steps):
        rate, cores, desc, _ = oracle_sample(w, budget_s=budget)
        rates.append(rate)
    wall = time.perf_counter() - t0
    value = statistics.median(rates)
    return {"impl": "reference", "metric": metric_name(w), "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall * 1e3 / args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same generator as the GPU arm)",
            "config": forward_config(w, world, l2_note(forward_inputs_bytes(w))),
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


WORKLOADS = {"long-grm": mc_inputs.LONG_GRM, "grm-d64": mc_inputs.GRM_D64, "ssc": mc_inputs.SSC_D128,
             "swla-grm": mc_inputs.SWLA_LONG, "fact-c32": mc_inputs.FACT_C32, "long-c512": mc_inputs.LONG_C512,
             "tiny": mc_inputs.TINY, **{f"sweep-c{w.seg_len}": w for w in mc_inputs.SWEEP}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["decode-grm", "loglinear-grm"] +
                    ["bwd-" + n for n in sorted(WORKLOADS)],
                    default="long-grm")
    ap.add_argument("--mode", choices=["residual", "grm", "soup", "ssc"], default=None,
                    help="override the workload's aggregation")
    ap.add_argument("--warmup-seconds", type=float, default=1.0,
                    help="keep warming up at least this long (clocks settle under load)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--heads", type=int, default=0,
                    help="run a slice of the workload: B = 1 and this many heads (for profiler captures)")
    ap.add_argument("--readout", choices=["auto", "factorised"], default="auto",
                    help="form of the cached readout (mc_set_readout_form)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "decode-grm":
        if args.impl == "ours":
            print(json.dumps(run_decode(args)), flush=True)
        return
    if args.workload == "loglinear-grm":
        if args.impl == "ours":
            print(json.dumps(run_segments(args)), flush=True)
        return
    if args.workload.startswith("bwd-"):
        if args.impl == "ours":
            name = args.workload[4:]
            wb = WORKLOADS[name]
            if args.heads:
                wb = wb.with_(B=1, H=args.heads, name=f"{wb.name} (slice: B1 H{args.heads})")
            print(json.dumps(run_backward(args, wb, name)), flush=True)
        return
    w = WORKLOADS[args.workload]
    if args.heads:
        w = w.with_(B=1, H=args.heads, name=f"{w.name} (slice: B1 H{args.heads})")
    if args.readout == "factorised" and args.impl == "ours":
        import memory_caching_linear_gb300 as mcl
        from memory_caching_linear_gb300 import build as mcbuild
        mcbuild.build()
        mcl.mc_set_readout_form(mcl.MC_READOUT_FACTORISED)
        w = w.with_(name=f"{w.name} (factorised readout)")
    if args.mode:
        w = w.with_(mode={"residual": RESIDUAL, "grm": GRM, "soup": 2, "ssc": SSC}[args.mode])
    res = run_reference(args, w) if args.impl == "reference" else run_ours(args, w, args.workload)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
