#!/usr/bin/env python3
"""Causal attention fwd+bwd throughput on GB300.

Workload: one Llama-2-7B attention layer, B=1, H=32, S=32768, D=128, causal,
bf16 Q/K/V/dO drawn i.i.d. N(0,1) from a seed (synthetic, no dataset), scale
1/sqrt(128). A step is the whole hot path once: attn_fwd, then the calls
attn_bwd makes (the Delta preprocess, zeroing of the tiled dQ accumulator, the
one-pass backward, dQ to bf16), all in libattn.so.

FLOP convention (causal, half of the S x S pairs): forward 2*B*H*S^2*D,
backward 2.5 x forward, step 7*B*H*S^2*D.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The line also carries, at N = 1, a "sizes" record (S = 131072 H32, S = 262144
H40, S = 524288 H32 with RoPE theta 1e6 on Q and K: fwd and bwd ms, TFLOP/s,
fractions of the tensor peak) and the zigzag ring emulation against monolithic
attention at S = 131072, P = 8, and Ulysses over P = 8 emulated ranks at
the same size (the all-to-all kernel's GB/s, fwd+bwd against monolithic).
Fractions use the measured burst bf16 peak
unless a timed region ran for seconds under the power cap (then the sustained
figure, as it was measured). After the timed loops the device status word is
read: a bounded wait that expired inside a kernel (its outputs then
unfinished) makes the run exit 3, with the word in "device_status".

With N > 1 (torchrun, one rank per GPU) every rank runs its own layer (the
path shards by independent problems, no collective); value is the whole
job's FLOP / the slowest rank's time. One JSON line is printed by rank 0.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal attn fwd+bwd TFLOP/s and % of GB300 BF16 peak at S=32K–512K, H=32, D=128"
UNIT = "TFLOP/s"
B, H, S, D = 1, 32, 32768, 128
WORKLOAD = "llama2-7b-attention-layer causal fwd+bwd B1 H32 S32768 D128"
L2_NOTE = "inputs larger than L2: q,k,v,dO are 268 MB each (1.07 GB per step) vs 129 MB L2; no flush"
# Oracle sample for the CPU legs: head 0, the causal prefix of this many tokens (fwd+bwd).
CPU_SAMPLE_S = 8192


def _set_shape(h, s):
    """Overrides the workload shape (used for small ncu captures, never for the bench line)."""
    global H, S, WORKLOAD, L2_NOTE
    H, S = h, s
    WORKLOAD = f"causal fwd+bwd B1 H{h} S{s} D128 (profiling case)"
    L2_NOTE = f"q,k,v,dO are {s * h * D * 2 / 1e6:.0f} MB each"


def max_over_ranks(x, world, device):
    """The largest value of a per-rank float over all ranks (every rank gets it)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flop_per_rank_step, steps, t_max):
    """Whole-job throughput: every rank's FLOP over the slowest rank's time."""
    return world * flop_per_rank_step * steps / t_max / 1e12


def step_flop(b, h, s, d):
    return 7.0 * b * h * s * s * d


def fwd_flop(b, h, s, d):
    return 2.0 * b * h * s * s * d


def input_checksums(named):
    """fp64 sum of the first 2^20 elements of each generated input (outside any
    timed region), so that a record identifies the synthetic data it ran on."""
    return {n: float(t.reshape(-1)[: 1 << 20].double().sum()) for n, t in named}


def kernel_source_hash(files):
    """sha256 over the kernel sources a recorded ncu figure was taken from."""
    import hashlib

    hsh = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "long_context_causal_blockwise_gb300", "csrc", f), "rb") as fh:
            hsh.update(fh.read())
    return hsh.hexdigest()[:16]


KERNEL_SOURCES = {
    "attn_fwd": ("attn_fwd.cu", "common.cuh", "tmem_ldst.cuh"),
    "bwd_fused": ("attn_bwd.cu", "common.cuh", "tmem_ldst.cuh"),
    "bwd_dkdv": ("attn_bwd.cu", "common.cuh", "tmem_ldst.cuh"),
    "bwd_dq": ("attn_bwd.cu", "common.cuh", "tmem_ldst.cuh"),
    "dq_untile": ("attn_bwd.cu", "common.cuh"),
    "bwd_preprocess": ("lse_merge.cu", "common.cuh"),
    "rope": ("rope.cu", "common.cuh"),
    "cross_entropy": ("cross_entropy.cu", "common.cuh"),
    "ulysses_a2a": ("ulysses.cu",),
}


def recorded_traffic(kernel):
    """DRAM bytes per launch at this workload from a committed ncu record
    (profiles/dram_traffic_b1h32s32768.txt), or None when the record is missing
    or was taken from a different version of the kernel's sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_b1h32s32768.txt")
    try:
        want = kernel_source_hash(KERNEL_SOURCES[kernel])
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 3 and parts[0] == kernel and parts[1] == want:
                    return int(parts[2])
    except (OSError, KeyError, ValueError):
        return None
    return None


def load_peaks():
    """Dense bf16 tensor peaks (burst, sustained) in TFLOP/s, HBM copy GB/s, and
    where they come from: the measured file, else the fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        burst = float(pk.get("bf16_tflops"))
        sus = float(pk.get("bf16_tflops_sustained", burst))
        hbm = float(pk.get("hbm_gbs"))
        return {"burst": burst, "sustained": sus, "hbm": hbm, "source": "measured"}
    except Exception:
        return {"burst": 1900.0, "sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def hbm_fields(prefix, nbytes, ms, peaks):
    """Achieved GB/s of an HBM-bound call (algorithmic bytes over CUDA-event
    milliseconds) and its fraction of the measured copy bandwidth."""
    gbs = nbytes / ms / 1e6
    return {prefix + "gbs": gbs, prefix + "frac_of_hbm": gbs / peaks["hbm"],
            "hbm_peak": peaks["hbm"], "hbm_peak_source": peaks["source"]}


def tensor_peak(peaks, timed_s, clocks):
    """The tensor peak that applies to a timed region: the burst figure (a
    short burst at full clocks), or the sustained one when the region ran for
    seconds under the power cap, as that figure was measured."""
    capped = "sw_power_cap" in (clocks or {}).get("reasons", [])
    if timed_s > 2.0 and capped:
        return peaks["sustained"], "sustained"
    return peaks["burst"], "burst"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def cpu_oracle_sample(q, k, v, do, s_sample):
    """Times the fp64 oracle (fwd + bwd by the definition) on head 0's causal prefix."""
    import numpy as np

    import oracle

    f64 = lambda t: t[:, :s_sample, :1].float().cpu().numpy().astype(np.float64)  # noqa: E731
    qs, ks, vs, dos = f64(q), f64(k), f64(v), f64(do)
    t0 = time.perf_counter()
    oracle.attn_bwd(qs, ks, vs, dos, True, D ** -0.5)
    dt = time.perf_counter() - t0
    return dt, step_flop(1, 1, s_sample, D)


def run_reference(args, rank, world):
    """The oracle as it stands on the host cores, same metric and unit."""
    if rank != 0:
        return 0
    import torch

    from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo

    q, k, v, do = gaussian_qkvdo(1, 1, CPU_SAMPLE_S, D, seed=0, device="cpu")
    times = []
    flop = None
    for i in range(args.warmup + args.steps):
        dt, flop = cpu_oracle_sample(q, k, v, do, CPU_SAMPLE_S)
        if i >= args.warmup:
            times.append(dt)
    t = sum(times)
    value = flop * len(times) / t / 1e12
    cores = os.cpu_count()
    sample = f"fp64 oracle fwd+bwd of one head's causal prefix of {CPU_SAMPLE_S} tokens (H=1 of 32, S={CPU_SAMPLE_S} of {S})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "S": S, "D": D, "causal": True,
                   "global_batch": 1, "seq_len": S, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "extrapolated_full_step_s": step_flop(B, H, S, D) / (value * 1e12),
                         "extrapolated_note": "extrapolated: the full step's FLOPs at the sample's rate"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import long_context_causal_blockwise_gb300 as lcb
    from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lcb.load()
    scale = D ** -0.5
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=rank, device=dev)
    checksums = input_checksums((("q", q), ("k", k), ("v", v), ("do", do)))
    # the oracle's sample (head 0's causal prefix), kept on the host for the cpu_baseline leg
    q_cpu, k_cpu, v_cpu, do_cpu = (t[:, :CPU_SAMPLE_S, :1].cpu() for t in (q, k, v, do))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, device=dev)
    delta = torch.empty(B, H, S, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dq_tiles = lcb.dq_tiles_zeros(B, H, S, dev)
    stream = torch.cuda.current_stream(dev)

    # The calls attn_bwd makes, one by one so that each is timed on its own:
    # Delta, zeroing of the tiled dQ accumulator, the one-pass backward, dQ to bf16.
    names = ("attn_fwd", "bwd_preprocess", "dq_zero", "bwd_fused", "dq_untile")

    def step(evs=None):
        def mark(j):
            if evs is not None:
                evs[j].record(stream)
        mark(0)
        lcb.attn_fwd(q, k, v, causal=True, scale=scale, o=o, lse=lse)
        mark(1)
        lcb.attn_bwd_preprocess(o, do, delta)
        mark(2)
        lcb.dq_tiles_zero_(dq_tiles)
        mark(3)
        lcb.attn_bwd_ex(q, k, v, lse, delta, do, dq_tiles, dk, dv, True, scale, passes="fused")
        mark(4)
        lcb.dq_untile(dq_tiles, dq)
        mark(5)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler attach before the timed work
    t_start.record(stream)
    for i in range(args.steps):
        step(events[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    t_max = max_over_ranks(elapsed, world, dev)
    per = {n: [] for n in names}
    for evs in events:
        for j, n in enumerate(names):
            per[n].append(evs[j].elapsed_time(evs[j + 1]) / 1e3)
    avg = {n: sum(v_) / len(v_) for n, v_ in per.items()}

    status_bits, status_where = lcb.take_device_status()  # a bounded wait that expired in the timed loop
    e2e = None if args.no_e2e else run_e2e(args, world, dev, q, k, v, do, o, lse, dq, dk, dv)
    if e2e is not None:
        b2, w2 = lcb.take_device_status()  # ... or in the end-to-end leg
        status_bits |= b2
        status_where = status_where or w2

    if rank != 0:
        return 0 if status_bits == 0 else 3

    peaks = load_peaks()
    hbm, src = peaks["hbm"], peaks["source"]
    peak, peak_kind = tensor_peak(peaks, t_max, clocks)
    flop = step_flop(B, H, S, D)
    value = whole_job_tflops(world, flop, args.steps, t_max)
    ms = 1e3 * t_max / args.steps
    pairs = B * H * S * S / 2.0  # causal (query, key) pairs, the R5 convention
    tiles_bytes = B * H * ((S + 127) // 128) * 128 * D * 4
    alg = {  # algorithmic work per launch
        "attn_fwd": ("tensor", 4 * D * pairs),            # S = QK^T and O += PV
        "bwd_fused": ("tensor", 10 * D * pairs),          # S^T, dP^T, dV, dK, dQ
        "bwd_preprocess": ("hbm", 2 * B * S * H * D * 2 + B * S * H * 4),
        "dq_zero": ("hbm", tiles_bytes),                  # async memset of the tiled accumulator
        "dq_untile": ("hbm", tiles_bytes + B * S * H * D * 2),
    }
    kernels = {}
    for n in names:
        kind, work = alg[n]
        t = avg[n]
        if kind == "tensor":
            ach = work / t / 1e12
            kernels[n] = {"ms": 1e3 * t, "tflops": ach, "frac_of_peak": ach / peak,
                          "frac_of_sustained": ach / peaks["sustained"]}
        else:
            ach = work / t / 1e9
            kernels[n] = {"ms": 1e3 * t, "gbs": ach, "frac_of_peak": ach / hbm}
    dom = max(names, key=lambda n: avg[n])
    kind, work = alg[dom]
    if kind == "tensor":
        ach = work / avg[dom] / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "frac_of_sustained": ach / peaks["sustained"],
                "traffic": recorded_traffic(dom) if (H, S) == (32, 32768) else None,
                "peak_source": f"{src} bf16 {peak_kind} (cuBLAS bf16 GEMM)",
                "work_per_launch": f"{work:.4e} FLOP = 10*D FLOP x {pairs:.4e} causal pairs"}
    else:
        ach = work / avg[dom] / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": recorded_traffic(dom) if (H, S) == (32, 32768) else None,
                "peak_source": f"{src} HBM copy"}
    fwd_t = avg["attn_fwd"]
    bwd_t = sum(avg[n] for n in names if n != "attn_fwd")
    fwd_tf = fwd_flop(B, H, S, D) / fwd_t / 1e12
    bwd_tf = 2.5 * fwd_flop(B, H, S, D) / bwd_t / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "S": S, "D": D, "causal": True, "l2": L2_NOTE,
                   "global_batch": world, "seq_len": S, "parallelism": f"dp{world} (one independent layer per GPU)",
                   "input_checksum_f64": checksums},
        "pct_of_peak": 100.0 * (value / world) / peak,
        "peak_tflops": peak, "peak_kind": peak_kind, "peak_source": f"{src} bf16 {peak_kind}",
        "peak_tflops_sustained": peaks["sustained"], "pct_of_sustained": 100.0 * (value / world) / peaks["sustained"],
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_frac_of_peak": fwd_tf / peak, "bwd_frac_of_peak": bwd_tf / peak,
        "kernels": kernels,
        "roofline": roof,
        "gpu_launches": 4 * args.steps,  # attn_fwd, bwd_preprocess, bwd_fused, dq_untile (dq_zero is a memset)
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_sizes:
        del q, k, v, do, o, lse, delta, dq, dk, dv, dq_tiles
        torch.cuda.empty_cache()
        sampler = ClockSampler(local_rank)
        sampler.start()
        time.sleep(0.3)
        sizes = [size_record(h_, s_, args.size_steps, args.warmup, theta, local_rank)
                 for h_, s_, theta in ((32, 131072, None), (40, 262144, None), (32, 524288, 1e6))]
        ring = zigzag_record(args.warmup, args.size_steps, local_rank)
        uly = ulysses_record(args.warmup, args.size_steps, local_rank)
        ring["rank_balance"] = ring_balance_record(local_rank)
        sclocks = sampler.stop()
        for rec in sizes:
            pk, kind_ = tensor_peak(peaks, rec["timed_s"], sclocks)
            rec.update({"peak_tflops": pk, "peak_kind": kind_, "fwd_frac_of_peak": rec["fwd_tflops"] / pk,
                        "bwd_frac_of_peak": rec["bwd_tflops"] / pk, "pct_of_peak": 100.0 * rec["tflops"] / pk,
                        "fwd_frac_of_burst": rec["fwd_tflops"] / peaks["burst"],
                        "bwd_frac_of_burst": rec["bwd_tflops"] / peaks["burst"]})
        line["sizes"] = sizes
        line["zigzag_ring"] = ring
        line["ulysses"] = uly
        line["sizes_clocks"] = sclocks
        b2, w2 = lcb.take_device_status()
        status_bits |= b2
        status_where = status_where or w2
    line["device_status"] = status_bits
    if status_bits:
        line["device_status_where"] = status_where
    if world == 1 and not args.no_cpu_baseline:
        dt, cflop = cpu_oracle_sample(q_cpu, k_cpu, v_cpu, do_cpu, CPU_SAMPLE_S)
        line["cpu_baseline"] = {
            "value": cflop / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of head 0's causal prefix of {CPU_SAMPLE_S} tokens, {dt:.1f} s",
            "extrapolated_full_step_s": step_flop(B, H, S, D) * dt / cflop,
            "extrapolated_note": "extrapolated: the full step's FLOPs at the sample's rate"}
    print(json.dumps(line), flush=True)
    return 0 if status_bits == 0 else 3


def run_e2e(args, world, dev, q, k, v, do, o, lse, dq, dk, dv):
    """The step end to end through the public calls attn_fwd and attn_bwd with
    host buffers in and out: every step copies its own inputs in from pinned
    host memory and its results out, inside the timed region. Two device
    buffer sets and two copy streams let step i+1's inputs arrive and step
    i-1's results leave while step i computes, as a training loop would
    overlap them."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb

    scale = D ** -0.5
    e2e_steps = max(4, args.steps)  # as many steps as the device-timed run: the pipeline's fill and drain amortise alike
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
    hq, hk, hv, hdo = (pin(t) for t in (q, k, v, do))
    for h_, d_ in ((hq, q), (hk, k), (hv, v), (hdo, do)):
        h_.copy_(d_)
    ho, hlse, hdq, hdk, hdv = pin(o), pin(lse), pin(dq), pin(dk), pin(dv)
    ws = torch.empty(lcb.attn_bwd_workspace_bytes(B, H, S, D), dtype=torch.uint8, device=dev)
    dev_in = [tuple(torch.empty_like(t) for t in (q, k, v, do)) for _ in range(2)]
    dev_out = [(torch.empty_like(o), torch.empty_like(lse), torch.empty_like(dq), torch.empty_like(dk),
                torch.empty_like(dv)) for _ in range(2)]
    s_comp, s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: [torch.cuda.Event() for _ in range(2)]  # noqa: E731
    # per buffer set: q, k, v in; dO in; inputs read; O, LSE ready; gradients ready; results out
    qkv_in, do_in, in_free, fwd_out, bwd_out, out_free = ev(), ev(), ev(), ev(), ev(), ev()

    def e2e_run(nsteps):
        for i in range(nsteps):
            bi = i % 2
            q_, k_, v_, do_ = dev_in[bi]
            o_, lse_, dq_, dk_, dv_ = dev_out[bi]
            s_h2d.wait_event(in_free[bi])  # step i-2 has finished reading this input set
            with torch.cuda.stream(s_h2d):
                for d_, h_ in ((q_, hq), (k_, hk), (v_, hv)):
                    d_.copy_(h_, non_blocking=True)
                qkv_in[bi].record(s_h2d)
                do_.copy_(hdo, non_blocking=True)  # only the backward reads dO
                do_in[bi].record(s_h2d)
            s_comp.wait_event(qkv_in[bi])
            s_comp.wait_event(out_free[bi])  # step i-2's results have left this output set
            with torch.cuda.stream(s_comp):
                lcb.attn_fwd(q_, k_, v_, causal=True, scale=scale, o=o_, lse=lse_)
                fwd_out[bi].record(s_comp)
                s_comp.wait_event(do_in[bi])
                lcb.attn_bwd(q_, k_, v_, o_, lse_, do_, causal=True, scale=scale, dq=dq_, dk=dk_, dv=dv_,
                             workspace=ws)
                in_free[bi].record(s_comp)
                bwd_out[bi].record(s_comp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(fwd_out[bi])  # O and LSE leave while the backward runs
                for h_, d_ in ((ho, o_), (hlse, lse_)):
                    h_.copy_(d_, non_blocking=True)
                s_d2h.wait_event(bwd_out[bi])
                for h_, d_ in ((hdq, dq_), (hdk, dk_), (hdv, dv_)):
                    h_.copy_(d_, non_blocking=True)
                out_free[bi].record(s_d2h)

    e2e_run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    e2e_run(e2e_steps)
    s_h2d.wait_stream(s_d2h)
    e1.record(s_h2d)
    torch.cuda.synchronize()
    e2e_t = max_over_ranks(e0.elapsed_time(e1) / 1e3 / e2e_steps, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    d2h = sum(t.numel() * t.element_size() for t in (o, lse, dq, dk, dv))
    # the e2e outputs must equal the device-resident run's: O, dK, dV bit for bit; dQ (fp32
    # sums in no fixed order, then bf16) within one bf16 rounding step
    ddq = (hdq.to(dev).float() - dq.float()).abs().max().item()
    same = bool(torch.equal(ho.to(dev), o) and torch.equal(hdk.to(dev), dk) and torch.equal(hdv.to(dev), dv)
                and ddq <= 2 ** -7 * dq.float().abs().max().item())
    del dev_in, dev_out, ws
    torch.cuda.empty_cache()
    return {"value": whole_job_tflops(world, step_flop(B, H, S, D), 1, e2e_t), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * e2e_t, "steps": e2e_steps,
            "matches_device_run": same,
            "overlap": "step i+1's host-to-device and step i-1's device-to-host copies run on two copy "
                       "streams during step i (double-buffered device tensors); the forward starts once q, k, "
                       "v are in, and O, LSE leave while the backward runs"}


def size_record(h, s, steps, warmup, rope_theta, local_rank):
    """One size of the metric's range: attn_fwd and attn_bwd (the public calls,
    workspace passed in) timed separately per step with CUDA events."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb
    from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo

    dev = torch.device("cuda", local_rank)
    scale = D ** -0.5
    q, k, v, do = gaussian_qkvdo(1, h, s, D, seed=0, device=dev)
    if rope_theta:  # positions 0..S-1, outside the timed region
        lcb.rope(q, rope_theta)
        lcb.rope(k, rope_theta)
    o, lse = torch.empty_like(q), torch.empty(1, h, s, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(lcb.attn_bwd_workspace_bytes(1, h, s, D), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        lcb.attn_fwd(q, k, v, causal=True, scale=scale, o=o, lse=lse)

    def bwd():
        lcb.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e in evs:
        e[0].record(stream)
        fwd()
        e[1].record(stream)
        bwd()
        e[2].record(stream)
    torch.cuda.synchronize()
    tf = sum(e[0].elapsed_time(e[1]) for e in evs) / steps / 1e3
    tb = sum(e[1].elapsed_time(e[2]) for e in evs) / steps / 1e3
    ff = fwd_flop(1, h, s, D)
    del q, k, v, do, o, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return {"workload": f"B1 H{h} S{s} D128 causal" + (f", Q/K RoPE theta={rope_theta:g}" if rope_theta else ""),
            "H": h, "S": s, "steps": steps, "warmup": warmup, "fwd_ms": 1e3 * tf, "bwd_ms": 1e3 * tb,
            "ms_per_step": 1e3 * (tf + tb), "tflops": 3.5 * ff / (tf + tb) / 1e12,
            "fwd_tflops": ff / tf / 1e12, "bwd_tflops": 2.5 * ff / tb / 1e12, "timed_s": steps * (tf + tb)}


def zigzag_record(warmup, steps, local_rank, detail=False):
    """The one-device zigzag ring (S = 131072, P = 8, H = 32) against monolithic
    attention on the same inputs, fwd+bwd per step, CUDA events."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb
    from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo
    from long_context_causal_blockwise_gb300.zigzag import ZigzagPlan

    Hz, Sz, Pz = 32, 131072, 8
    dev = torch.device("cuda", local_rank)
    q, k, v, do = gaussian_qkvdo(1, Hz, Sz, D, seed=0, device=dev)
    plan = ZigzagPlan(Sz, Pz, dev)
    c2 = Sz // Pz
    bufs = {
        "o_acc": torch.empty(1, Sz, Hz, D, device=dev), "lse": torch.empty(1, Hz, Sz, device=dev),
        "o_blk": torch.empty(1, c2, Hz, D, device=dev, dtype=torch.bfloat16),
        "lse_blk": torch.empty(1, Hz, c2, device=dev), "o": torch.empty_like(q),
    }
    g32 = tuple(torch.empty(1, Sz, Hz, D, device=dev) for _ in range(3))
    g16 = tuple(torch.empty_like(q) for _ in range(3))
    delta = torch.empty(1, Hz, Sz, device=dev)
    qz, kz, vz, doz = (plan.gather(x) for x in (q, k, v, do))
    tiles = lcb.dq_tiles_zeros(1, Hz, Sz, dev)

    def ring_fwd(fused=True):
        return lcb.zigzag_attention_fwd(qz, kz, vz, plan, fused=fused, **bufs)

    def ring():
        o, lse, _ = ring_fwd()
        lcb.zigzag_attention_bwd(qz, kz, vz, o, lse, doz, plan, delta=delta, grads32=g32, grads=g16, dq_tiles=tiles)

    o_m, lse_m = torch.empty_like(q), torch.empty(1, Hz, Sz, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(lcb.attn_bwd_workspace_bytes(1, Hz, Sz, D), dtype=torch.uint8, device=dev)

    def mono():
        lcb.attn_fwd(q, k, v, o=o_m, lse=lse_m)
        lcb.attn_bwd(q, k, v, o_m, lse_m, do, dq=dq, dk=dk, dv=dv, workspace=ws)

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    t_ring, t_mono = timed(ring, steps), timed(mono, steps)
    flop = step_flop(1, Hz, Sz, D)
    rec = {"workload": "zigzag ring emulation fwd+bwd, P=8 virtual ranks, B1 H32 S131072 D128, vs monolithic",
           "steps": steps, "warmup": warmup, "ring_ms": t_ring, "monolithic_ms": t_mono,
           "ring_overhead_pct": 100.0 * (t_ring / t_mono - 1.0),
           "ring_tflops": flop / t_ring / 1e9, "monolithic_tflops": flop / t_mono / 1e9}
    if detail:
        t_fwd_fused, t_fwd_unfused = timed(ring_fwd, steps), timed(lambda: ring_fwd(False), steps)
        t_fwd_mono = timed(lambda: lcb.attn_fwd(q, k, v, o=o_m, lse=lse_m), steps)
        # merge kernel alone: one LOWER/UPPER-sized merge (2c rows) timed in isolation
        oa, la = bufs["o_acc"][:, :c2], bufs["lse"][:, :, :c2]
        ob, lb = bufs["o_blk"], bufs["lse_blk"]
        t_merge = timed(lambda: lcb.attn_lse_merge(oa, la, ob, lb), 20)
        merge_bytes = c2 * Hz * (D * 4 * 2 + D * 2 + 12)
        hbm = load_peaks()["hbm"]
        rec.update({
            "fwd_ms": {"ring_fused_merge": t_fwd_fused, "ring_merge_kernel": t_fwd_unfused,
                       "monolithic": t_fwd_mono},
            "merge_ms_per_call": t_merge, "merge_rows": c2, "merge_gbs": merge_bytes / t_merge / 1e6,
            "merge_frac_of_hbm": merge_bytes / t_merge / 1e6 / hbm,
            "launches_per_ring_step": "fwd: 1 grouped launch of the P tasks (merge fused in the epilogue); bwd: 1 "
                                      "grouped one-pass launch of the P tasks; + preprocess, zeroing and untile "
                                      "once per pass"})
    del q, k, v, do, qz, kz, vz, doz, bufs, g32, g16, delta, tiles, o_m, lse_m, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return rec


def ring_balance_record(local_rank):
    """The rank-local ring driver at B1 H32 S131072 over P = 8 ranks, run
    through the one-process loopback, for the zigzag and the plain
    (contiguous) schedule: every rank's kernel time per ring step (CUDA
    events around its steps), the lockstep critical path (the slowest rank at
    each step, as the ranks of a real ring wait for each other) against a
    perfectly balanced one (total / P)."""
    import torch

    from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo
    from long_context_causal_blockwise_gb300.ring import LoopbackRing, RingRank
    import long_context_causal_blockwise_gb300 as lcb

    Hr, Sr, Pr = 32, 131072, 8
    dev = torch.device("cuda", local_rank)
    q, k, v, do = gaussian_qkvdo(1, Hr, Sr, D, seed=0, device=dev)
    out = {"workload": "rank-local ring driver, loopback of P=8 ranks on one GPU, B1 H32 S131072 D128 causal, "
                       "fwd+bwd; transfers are device copies between the ranks' kernels"}
    for sched in ("zigzag", "contiguous"):
        if sched == "zigzag":
            plan = lcb.zigzag.ZigzagPlan(Sr, Pr, dev)
            src = [plan.gather(x) for x in (q, k, v, do)]
        else:
            src = [q, k, v, do]
        n = Sr // Pr
        mine = [[x[:, r * n:(r + 1) * n].contiguous() for x in src] for r in range(Pr)]
        del src
        for warm in (True, False):
            hub = LoopbackRing(Pr, time_ranks=not warm)
            ranks = [RingRank(r, Pr, Sr, hub.transport(r), schedule=sched) for r in range(Pr)]
            fwd = hub.run([rk.forward_steps(*mine[r][:3]) for r, rk in enumerate(ranks)])
            hub.run([rk.backward_steps(*mine[r][:3], fwd[r][0], fwd[r][1], mine[r][3])
                     for r, rk in enumerate(ranks)])
            del fwd
        torch.cuda.synchronize()
        steps = [[a.elapsed_time(b) for a, b in evs] for evs in hub.events]
        per_rank = [sum(x) for x in steps]
        critical = sum(max(steps[r][j] for r in range(Pr)) for j in range(len(steps[0])))
        out[sched] = {"rank_ms": per_rank, "critical_path_ms": critical, "balanced_ms": sum(per_rank) / Pr,
                      "imbalance": critical / (sum(per_rank) / Pr)}
        del mine
        torch.cuda.empty_cache()
    return out


def ulysses_record(warmup, steps, local_rank):
    """Ulysses over P = 8 emulated ranks at B1 H32 S131072: the all-to-all
    kernel alone (bytes read + written per call against the HBM peak), and
    Ulysses fwd+bwd (4 all-to-alls in, 4 out, attention on the head layout)
    against monolithic attention on the same inputs."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb
    from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo

    Hu, Su, Pu = 32, 131072, 8
    dev = torch.device("cuda", local_rank)
    q, k, v, do = gaussian_qkvdo(1, Hu, Su, D, seed=0, device=dev)
    qh = torch.empty((Pu, Su, Hu // Pu, D), dtype=q.dtype, device=dev)
    back = torch.empty_like(q)
    o_m, lse_m = torch.empty_like(q), torch.empty(1, Hu, Su, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(lcb.attn_bwd_workspace_bytes(Pu, Hu // Pu, Su, D), dtype=torch.uint8, device=dev)

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    t_in = timed(lambda: lcb.ulysses_all_to_all(q, Pu, to_heads=True, out=qh), 20)
    t_out = timed(lambda: lcb.ulysses_all_to_all(qh, Pu, to_heads=False, out=back), 20)

    def uly():
        o, ctx = lcb.ulysses_attention_fwd(q, k, v, Pu)
        lcb.ulysses_attention_bwd(do, ctx, workspace=ws)

    def mono():
        lcb.attn_fwd(q, k, v, o=o_m, lse=lse_m)
        lcb.attn_bwd(q, k, v, o_m, lse_m, do, dq=dq, dk=dk, dv=dv, workspace=ws)

    t_u, t_m = timed(uly, steps), timed(mono, steps)
    nbytes = 2 * q.numel() * q.element_size()
    hbm = load_peaks()["hbm"]
    del q, k, v, do, qh, back, o_m, lse_m, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return {"workload": "Ulysses all-to-all around attention, P=8 emulated ranks (4 heads each), "
                        "B1 H32 S131072 D128 causal, vs monolithic",
            "a2a_ms_seq_to_head": t_in, "a2a_ms_head_to_seq": t_out, "a2a_bytes_per_call": nbytes,
            "a2a_gbs": nbytes / t_in / 1e6, "a2a_frac_of_hbm": nbytes / t_in / 1e6 / hbm,
            "a2a_gbs_head_to_seq": nbytes / t_out / 1e6,
            "ulysses_ms": t_u, "monolithic_ms": t_m, "ulysses_overhead_pct": 100.0 * (t_u / t_m - 1.0),
            "steps": steps, "warmup": warmup}


def run_zigzag(args):
    """Times the one-device zigzag ring against monolithic attention; prints one
    JSON line (not the headline bench line)."""
    import long_context_causal_blockwise_gb300 as lcb

    lcb.load()
    rec = zigzag_record(args.warmup, max(1, min(args.steps, 5)), 0, detail=True)
    rec["rank_balance"] = ring_balance_record(0)
    rec["metric"] = "zigzag ring emulation fwd+bwd (P=8, S=131072, H=32, D=128) vs monolithic"
    bits, _ = lcb.take_device_status()
    rec["device_status"] = bits
    print(json.dumps(rec), flush=True)
    return 0 if bits == 0 else 3


def run_ulysses(args):
    """Times Ulysses over P = 8 emulated ranks (all-to-all kernel and fwd+bwd
    against monolithic attention); prints one JSON line (not the headline)."""
    import long_context_causal_blockwise_gb300 as lcb

    lcb.load()
    rec = ulysses_record(max(3, args.warmup), max(1, min(args.steps, 5)), 0)
    rec["metric"] = "Ulysses all-to-all + attention, P=8 emulated ranks, B1 H32 S131072 D128"
    bits, _ = lcb.take_device_status()
    rec["device_status"] = bits
    print(json.dumps(rec), flush=True)
    return 0 if bits == 0 else 3


def run_rope(args):
    """Times the RoPE kernel (theta = 1e6) on one [1, S, H, 128] bf16 tensor at
    the long-context stress size S = 524288, H = 32 (4.3 GB), in place, and
    its inverse; prints one JSON line (not the headline bench line)."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb

    Sr, Hr, theta = 524288, 32, 1e6
    dev = torch.device("cuda", 0)
    lcb.load()
    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn(1, Sr, Hr, D, generator=g, device=dev).to(torch.bfloat16)

    def timed(fn, steps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(3, min(args.steps, 20))
    t_fwd = timed(lambda: lcb.rope(x, theta), steps)
    t_inv = timed(lambda: lcb.rope(x, theta, inverse=True), steps)
    nbytes = 2 * x.numel() * 2  # read and write every element once
    pk = load_peaks()
    print(json.dumps({
        "metric": "RoPE (theta=1e6) on one bf16 [1, 524288, 32, 128] tensor, in place",
        "ms": t_fwd, "ms_inverse": t_inv, "bytes_per_call": nbytes,
        **hbm_fields("", nbytes, t_fwd, pk), **hbm_fields("inverse_", nbytes, t_inv, pk),
        "inputs": "larger than L2 (4.3 GB); no flush"}), flush=True)
    return 0


def run_merge(args):
    """Times the stand-alone LSE merge (attn_lse_merge) of one bf16 block into
    the fp32 accumulator, 16384 rows x 32 heads x 128 (the ring step's merge at
    S = 131072, P = 8), in place; L2 flushed between calls (each call is 0.68
    GB, under L2 twice over); median of the timed calls. Prints one JSON line
    (not the headline bench line)."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb

    Bm, Rm, Hm = 1, 16384, 32
    dev = torch.device("cuda", 0)
    lcb.load()
    g = torch.Generator(device=dev).manual_seed(0)
    o_acc = torch.randn(Bm, Rm, Hm, D, generator=g, device=dev)
    lse_acc = torch.randn(Bm, Hm, Rm, generator=g, device=dev)
    o_b = torch.randn(Bm, Rm, Hm, D, generator=g, device=dev).to(torch.bfloat16)
    lse_b = torch.randn(Bm, Hm, Rm, generator=g, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        lcb.attn_lse_merge(o_acc, lse_acc, o_b, lse_b)
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(3, min(args.steps, 20))):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        lcb.attn_lse_merge(o_acc, lse_acc, o_b, lse_b)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = statistics.median(ts)
    nbytes = Bm * Rm * Hm * (D * (4 + 4 + 2) + 12)  # O_acc read and written, O_b read, statistics
    print(json.dumps({
        "metric": "LSE merge of a bf16 block into the fp32 accumulator, 16384 rows x 32 heads x 128, in place",
        "ms": ms, "bytes_per_call": nbytes, **hbm_fields("", nbytes, ms, load_peaks()),
        "inputs": "L2 flushed (256 MB written) before each timed call"}), flush=True)
    return 0


def run_ce(args):
    """Times the cross-entropy loss head, forward and in-place backward in one
    pass, on Llama-2's vocabulary (V = 32000) over a 32768-token sequence
    (2.1 GB of bf16 logits), or with --vocab V over as many tokens as keep the
    logits near that size (V = 128256, Llama-3: 8192 tokens, rows streamed);
    prints one JSON line (not the headline bench line). Bytes are the
    algorithmic ones: logits read once (and written once with the backward)."""
    import torch

    import long_context_causal_blockwise_gb300 as lcb

    V = args.vocab
    N = max(1, 32768 * 32000 // V)
    dev = torch.device("cuda", 0)
    lcb.load()
    g = torch.Generator(device=dev).manual_seed(0)
    x = (torch.randn(N, V, generator=g, device=dev) * 3).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), generator=g, device=dev)
    loss = torch.empty(N, device=dev)
    lse = torch.empty(N, device=dev)

    def timed(fn, steps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    steps = max(3, min(args.steps, 20))
    t_fwd = timed(lambda: lcb.cross_entropy(x, y, mode="fwd", loss=loss, lse=lse), steps)
    t_fb = timed(lambda: lcb.cross_entropy(x, y, mode="fwd_bwd", loss=loss, lse=lse), steps)
    nb_fwd = N * V * 2 + N * (8 + 8)
    nb_fb = 2 * N * V * 2 + N * (8 + 8)
    pk = load_peaks()
    print(json.dumps({
        "metric": f"cross-entropy loss head, V={V}, N={N} tokens, bf16 logits",
        "fwd_bwd_ms": t_fb, "fwd_ms": t_fwd, "tokens_per_s_fwd_bwd": N / t_fb * 1e3,
        **hbm_fields("fwd_bwd_", nb_fb, t_fb, pk), **hbm_fields("fwd_", nb_fwd, t_fwd, pk),
        "inputs": "larger than L2 (2.1 GB of logits); no flush"}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (its double-buffered tensors; for small ncu captures)")
    ap.add_argument("--no-sizes", action="store_true",
                    help="skip the S=128K-512K sizes and the zigzag ring record (for ncu captures)")
    ap.add_argument("--size-steps", type=int, default=3, help="timed steps per size of the sizes record")
    ap.add_argument("--H", type=int, default=H, help="heads (profiling of smaller cases only)")
    ap.add_argument("--S", type=int, default=S, help="sequence length (profiling of smaller cases only)")
    ap.add_argument("--vocab", type=int, default=32000, help="vocabulary size of --ce")
    ap.add_argument("--merge", action="store_true",
                    help="time the stand-alone LSE merge (attn_lse_merge) at the ring step's size and exit")
    ap.add_argument("--ce", action="store_true",
                    help="time the cross-entropy loss head (V=32000, 32768 tokens)")
    ap.add_argument("--rope", action="store_true",
                    help="time the RoPE kernel on a [1, 524288, 32, 128] tensor")
    ap.add_argument("--zigzag", action="store_true",
                    help="time the one-device zigzag ring (S=131072, P=8) against monolithic attention")
    ap.add_argument("--ulysses", action="store_true",
                    help="time Ulysses over P=8 emulated ranks (S=131072, H=32) against monolithic attention")
    ap.add_argument("--print-kernel-hashes", action="store_true",
                    help="print the source hash of each kernel (for recording ncu traffic) and exit")
    args = ap.parse_args()
    if args.zigzag:
        return run_zigzag(args)
    if args.rope:
        return run_rope(args)
    if args.merge:
        return run_merge(args)
    if args.ulysses:
        return run_ulysses(args)
    if args.ce:
        return run_ce(args)
    if args.print_kernel_hashes:
        for k, files in KERNEL_SOURCES.items():
            print(k, kernel_source_hash(files))
        return 0
    if (args.H, args.S) != (H, S):
        _set_shape(args.H, args.S)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
