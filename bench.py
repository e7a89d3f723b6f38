#!/usr/bin/env python
"""Benchmark: exact fused attention forward + backward on GB300 (sm_103a).

One step = one forward (attn_fwd) and one backward (attn_bwd: preprocess, main
kernel, dQ conversion) over the causal BF16 workload B=8, H=16, N=4096, d=128,
scale 1/sqrt(128), inputs ~ N(0, 1).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --shape B,H,N,d[,noncausal][,fp16]   (another shape, for profiling)
  python bench.py --sweep | --decode-shape ... | --dsa-shape ...   (the tables, one line each)

value        whole-job TFLOPS of the step, FLOP convention fwd 4 B H N^2 d and
             bwd 10 B H N^2 d, each halved for causal; inputs resident in HBM.
e2e          the same metric through the C ABI with HOST (pinned) buffers:
             q, k, v, dO copied in and o, lse, dq, dk, dv copied out every step.
fwd_pct_peak / bwd_pct_peak
             % of the GB300 dense BF16 tensor peak at the SM clock sampled
             during the timed region (SMs x 8192 FLOP/clk x MHz); the same
             against the measured cuBLAS burst and sustained peaks alongside.
roofline     the backward main kernel (the dominant one): its algorithmic FLOPs
             per launch / its median CUDA-event duration, against the measured
             burst bf16 peak (the kernel is timed launch by launch); traffic
             from a committed ncu capture when it matches the current kernel
             source, else null.
cpu_baseline the FP64 oracle, as it stands, on a bounded sample of the same
             workload on this host's cores (rank 0, N=1 only).
--impl reference  times that oracle alone, each step a bounded sample.

Multi-GPU: every rank runs its own copy of the workload on its own GPU (heads
are independent, no data-path collective); value = all ranks' FLOPs / max time.
Launched under torchrun (RANK / WORLD_SIZE set) each process is one rank; with
--gpus N > 1 and no WORLD_SIZE, bench.py starts the N ranks itself through
torch.distributed.run (rendezvous on 127.0.0.1).
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "attention fwd / bwd TFLOPS (BF16, d=128, causal) and % of GB300 BF16 peak"
WORKLOAD = dict(B=8, H=16, N=4096, d=128, causal=True)
DTYPE = "bf16"  # 16-bit type of q, k, v, dO (--shape may ask for fp16)
DEFAULT_WORKLOAD = dict(WORKLOAD)
WORKLOAD_NAME = "causal MHA BF16 fwd+bwd B=8 H=16 N=4096 d=128, scale 1/sqrt(128), q,k,v,dO ~ N(0,1)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Dense BF16 tensor-core work per SM per clock on sm_103a: one 128 x 256 x 16 MMA (2 x 128 x 256 x 16
# FLOP) every 128 cycles.
NOMINAL_FLOP_PER_CLK = 8192


def nominal_bf16_tflops(n_sm, sm_mhz):
    return n_sm * NOMINAL_FLOP_PER_CLK * sm_mhz * 1e6 / 1e12


# The sources the attention forward / backward kernels are compiled from (the other kernels of
# the library do not change their DRAM traffic).
ATTN_KERNEL_SOURCES = ("attn_bwd.cu", "attn_fwd.cu", "attn_internal.h", "ptx.cuh", "seq.cuh")


def kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_flashattention_gb300", "csrc")
    for name in ATTN_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key):
    """DRAM bytes per launch from profiles/traffic.json, if it was taken on the
    current kernel source (same sha); otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- oracle sample
def oracle_sample(n_heads, rows_per_head, seed=4242, threads=None):
    """Time the FP64 oracle on a bounded sample of the workload: n_heads heads,
    each restricted to rows_per_head query rows spread evenly over [0, N) (so the
    causal work per row averages that of the whole head).  One head at a time per
    thread, `threads` threads (default: one per head).
    Returns (seconds, algorithmic FLOPs of the sample, threads)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    import seeded_inputs as si

    B, H, N, d, causal = (WORKLOAD[k] for k in ("B", "H", "N", "d", "causal"))
    scale = d ** -0.5
    heads = [(h * 37) % (B * H) for h in range(n_heads)]
    data = {n: si.tensor_heads(seed, n, B * H, N, d, 1.0, heads=heads) for n in ("q", "k", "v", "do")}
    stride = max(1, N // rows_per_head)
    rows = np.arange(stride // 2, N, stride)[:rows_per_head]
    f64 = [{n: si.bits_to_f32(data[n][i], "bf16").astype(np.float64) for n in data} for i in range(n_heads)]
    oracle.build()

    def one(i):
        x = f64[i]
        oracle.attn_bwd_rowset(x["q"], x["k"], x["v"], x["do"], rows, scale, causal)

    threads = threads or n_heads
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, range(n_heads)))
    dt = time.perf_counter() - t0
    # pages' convention: 14 d FLOPs (fwd 4 d + bwd 10 d) per unmasked (query, key) pair
    pairs = float(np.sum(rows + 1)) if causal else float(len(rows) * N)
    flops = 14.0 * d * pairs * n_heads
    return dt, flops, threads


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    cores = host_cores()
    n_heads = min(cores, 16)
    rows = 64
    for _ in range(args.warmup):
        oracle_sample(n_heads, rows)
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, fl, _ = oracle_sample(n_heads, rows)
        times.append(dt)
        flops = fl
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = (f"{n_heads} heads x {rows} query rows (rows spread evenly over N) of the {WORKLOAD_NAME} "
              f"workload, full fwd+bwd work of those rows, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, **WORKLOAD},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": n_heads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_flashattention_gb300 as attn
    from exact_attention_flashattention_gb300 import flops as F

    B, H, N, d, causal = (WORKLOAD[k] for k in ("B", "H", "N", "d", "causal"))
    scale = d ** -0.5
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    shape = (B, H, N, d)
    tdt = torch.bfloat16 if DTYPE == "bf16" else torch.float16
    q, k, v, do = (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(tdt) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fwd_fl = F.fwd_flops(B, H, N, d, causal)
    bwd_fl = F.bwd_flops(B, H, N, d, causal)
    launches_per_step = 4  # forward kernel + preprocess + backward main + dQ conversion

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        attn.attn_fwd(q, k, v, o, lse, scale, causal, stream)
        if ev is not None:
            ev[1].record(stream)
        attn.attn_bwd_stage(0, q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, stream)
        if ev is not None:
            ev[2].record(stream)
        attn.attn_bwd_stage(1, q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, stream)
        if ev is not None:
            ev[3].record(stream)
        attn.attn_bwd_stage(2, q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, stream)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if attn.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error word set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    if attn.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error word set during the timed region")

    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    pre_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    main_ms = statistics.median(e[2].elapsed_time(e[3]) for e in evs)
    conv_ms = statistics.median(e[3].elapsed_time(e[4]) for e in evs)
    fwd_med = fwd_ms
    bwd_med = statistics.median(e[1].elapsed_time(e[4]) for e in evs)
    ms_per_step = max_over_ranks(total_ms / args.steps, world)
    value = (fwd_fl + bwd_fl) * world / ms_per_step / 1e9

    # ---- end to end through the C ABI with host buffers.  Every step copies its inputs in from
    # pinned host memory and its results (O, L, dQ, dK, dV) back out.  The steps are pipelined
    # the way a throughput-oriented caller would run them: two device buffer sets, the input
    # copies, the kernels and the output copies on three streams, events guarding each set's
    # reuse, so step s's copies overlap the kernels of its neighbours.
    e2e = None
    if not args.no_e2e:
        pin = {n: t.cpu().pin_memory() for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
        outs = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs.values())
        sets = [dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv, ws=ws)]
        sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_free = [ev(), ev()]     # the set's inputs have been read by its kernels
        out_free = [ev(), ev()]    # the set's outputs have been copied out
        for e_ in in_free + out_free:
            e_.record(stream)

        def e2e_step(si):
            x = sets[si % 2]
            with torch.cuda.stream(s_in):
                s_in.wait_event(in_free[si % 2])
                for n in ("q", "k", "v", "do"):
                    x[n].copy_(pin[n], non_blocking=True)
                loaded = ev()
                loaded.record(s_in)
            stream.wait_event(loaded)
            stream.wait_event(out_free[si % 2])
            attn.attn_fwd(x["q"], x["k"], x["v"], x["o"], x["lse"], scale, causal, stream)
            attn.attn_bwd(x["q"], x["k"], x["v"], x["o"], x["do"], x["lse"], x["dq"], x["dk"], x["dv"], x["ws"],
                          scale, causal, stream)
            in_free[si % 2].record(stream)
            done = ev()
            done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for n in ("o", "lse", "dq", "dk", "dv"):
                    outs[n].copy_(x[n], non_blocking=True)
                out_free[si % 2].record(s_out)

        for si in range(2):
            e2e_step(si)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 20))
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_event(a)
        for si in range(n_e2e):
            e2e_step(si)
        stream.wait_stream(s_out)
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(a.elapsed_time(b) / n_e2e, world)
        e2e = {"value": (fwd_fl + bwd_fl) * world / e2e_ms / 1e9, "unit": "TFLOPS", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipeline": "two buffer sets; input copies, kernels, output copies on three streams"}
        del sets

    if rank != 0:
        return 0

    props = torch.cuda.get_device_properties(dev)
    n_sm = props.multi_processor_count
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    main_tflops = bwd_fl / main_ms / 1e9
    tensor_mb = B * H * N * d * 2 / 1e6
    l2_note = ("inputs larger than L2 (q, k, v, dO: {:.0f} MB each; 129 MB L2), no flush" if 4 * tensor_mb > 129
               else "inputs fit in L2 (q, k, v, dO: {:.0f} MB each; 129 MB L2), no flush").format(tensor_mb)
    # the committed counters belong to the default workload's backward
    traffic = committed_traffic("attn_bwd_kernel<128,bf16>") if (WORKLOAD == DEFAULT_WORKLOAD and DTYPE == "bf16") else None
    fwd_tf = fwd_fl / fwd_med / 1e9
    bwd_tf = bwd_fl / bwd_med / 1e9
    # The tensor pipe's dense rate at the SM clock sampled during the timed region (the clock the
    # kernels ran at), or at the maximum clock when no sample could be taken.
    sm_mhz = clocks["sm_mhz"] if clocks else float(peaks.get("sm_max_mhz", 2070.0))
    nominal = nominal_bf16_tflops(n_sm, sm_mhz)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        threads = min(host_cores(), 16)
        n_heads = 2 * threads
        rows = WORKLOAD["N"]
        dt, fl, thr = oracle_sample(n_heads, rows, threads=threads)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOPS", "cores": thr, "kind": "oracle",
               "sample": f"{n_heads} whole heads ({rows} query rows each) of the same workload, full fwd+bwd work, "
                         f"{dt:.1f} s wall on {thr} threads",
               "seconds": dt}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": DTYPE,
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, **WORKLOAD, "parallelism": f"replicas{world}", "l2": l2_note},
        "fwd_tflops": fwd_tf,
        "bwd_tflops": bwd_tf,
        "fwd_pct_peak": 100.0 * fwd_tf / nominal,
        "bwd_pct_peak": 100.0 * bwd_tf / nominal,
        "pct_peak_basis": (f"GB300 dense BF16 tensor peak at the SM clock: {n_sm} SMs x {NOMINAL_FLOP_PER_CLK} "
                           f"FLOP/clk/SM x {sm_mhz:.0f} MHz ({'median sampled during the timed region' if clocks else 'maximum clock, no sample'}) "
                           f"= {nominal:.1f} TFLOP/s"),
        "fwd_pct_measured_burst_peak": 100.0 * fwd_tf / peak_burst,
        "bwd_pct_measured_burst_peak": 100.0 * bwd_tf / peak_burst,
        "fwd_pct_measured_sustained_peak": 100.0 * fwd_tf / peak_sus,
        "bwd_pct_measured_sustained_peak": 100.0 * bwd_tf / peak_sus,
        "measured_peaks": {"bf16_tflops": peak_burst, "bf16_tflops_sustained": peak_sus, "source": peak_src},
        "kernel_ms": {"attn_fwd": fwd_ms, "bwd_preprocess": pre_ms, "bwd_main": main_ms, "bwd_dq_convert": conv_ms,
                      "statistic": f"median over the {args.steps} timed steps (CUDA events per kernel)"},
        "roofline": {
            "kernel": f"attn_bwd_kernel<{d},{DTYPE}> (backward main)",
            "bound": "tensor",
            "achieved": main_tflops,
            "peak": peak_burst,
            "unit": "TFLOP/s",
            "frac": main_tflops / peak_burst,
            "peak_kind": f"bf16_tflops (cuBLAS burst; the kernel is timed launch by launch), {peak_src}",
            "sm_mhz": sm_mhz,
            "frac_of_nominal_at_clock": main_tflops / nominal,
            "traffic": traffic,
            "algorithmic_flops_per_launch": bwd_fl,
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def time_calls(fn, stream, iters, warmup):
    """Median device time of one call of fn (ms): `warmup` untimed calls, then `iters` calls
    each bracketed by CUDA events on `stream`."""
    import torch
    for _ in range(warmup):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


SWEEP = [
    # name, B, H, N, d, causal, dtype, sigma_qk
    ("tiny B=1 H=2 N=128 d=64 causal", 1, 2, 128, 64, True, "bf16", 1.0),
    ("tiny B=1 H=2 N=128 d=64 non-causal", 1, 2, 128, 64, False, "bf16", 1.0),
    ("causal B=8 H=16 N=4096 d=128", 8, 16, 4096, 128, True, "bf16", 1.0),
    ("non-causal B=4 H=16 N=4096 d=128", 4, 16, 4096, 128, False, "bf16", 1.0),
    ("non-causal B=2 H=16 N=8192 d=128", 2, 16, 8192, 128, False, "bf16", 1.0),
    ("non-causal B=1 H=16 N=16384 d=128", 1, 16, 16384, 128, False, "bf16", 1.0),
    ("fp16 causal B=4 H=16 N=1024 d=64", 4, 16, 1024, 64, True, "fp16", 1.0),
    ("fp16 causal B=4 H=16 N=2048 d=64", 4, 16, 2048, 64, True, "fp16", 1.0),
    ("fp16 causal B=4 H=16 N=4096 d=64", 4, 16, 4096, 64, True, "fp16", 1.0),
    ("stress causal B=1 H=32 N=32768 d=128 sigma_qk=2", 1, 32, 32768, 128, True, "bf16", 2.0),
]


# Decode (one query per head against a key/value cache): name, B, Hq, Hkv, cache length, d.
DECODE_SWEEP = [
    ("decode GQA B=8 Hq=32 Hkv=8 N=32768 d=128", 8, 32, 8, 32768, 128),
    ("decode MHA B=32 H=32 N=4096 d=128", 32, 32, 32, 4096, 128),
    ("decode GQA B=1 Hq=32 Hkv=8 N=131072 d=128", 1, 32, 8, 131072, 128),
    ("decode MHA B=64 H=16 N=2048 d=64", 64, 16, 16, 2048, 64),
]


# Sparse top-k attention backward with shared latent key/value rows: the shapes of the
# cudnn-frontend DSA backward pull request's tables (seqlen 4096, BF16, d_v 512, sink on,
# every row's top-k length = topk).
DSA_SWEEP = [
    # s_q = s_kv, H, d_qk, topk
    (4096, 64, 512, 128), (4096, 64, 512, 512), (4096, 64, 512, 2048),
    (4096, 128, 512, 2048),
    (4096, 128, 576, 128), (4096, 128, 576, 512), (4096, 128, 576, 2048),
    (4096, 64, 576, 2048),
]


def dsa_prepare(s_q, s_kv, H, d_qk, topk, causal, seed=17):
    """Synthetic inputs of the sparse top-k backward on the GPU (seeded_inputs.dsa_device_draws:
    q, kv, dO ~ N(0, 1) bf16, sink ~ N(0, 1), each row's list = topk distinct random keys,
    keys 0..i when causal, padded with -1) and the forward's O (bf16) and L (FP32) from a
    plain PyTorch FP32 computation over the gathered keys (input preparation, not timed)."""
    import torch

    import seeded_inputs as si
    dev = torch.device("cuda", 0)
    d_v = 512
    x = si.dsa_device_draws(s_q, s_kv, H, d_qk, topk, causal, seed=seed, d_v=d_v)
    q, kv, sink, idx = x["q"], x["kv"], x["sink"], x["idx"]
    o = torch.empty((s_q, H, d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s_q, H), dtype=torch.float32, device=dev)
    scale = d_qk ** -0.5
    kvf = kv.float()
    for r0 in range(0, s_q, 64):
        r1 = min(s_q, r0 + 64)
        ix = idx[r0:r1].long()
        valid = ix >= 0
        K = kvf[ix.clamp(min=0)]                                   # [r, topk, d_qk]
        S = torch.einsum("rhd,rkd->rhk", q[r0:r1].float(), K) * scale
        S = S.masked_fill(~valid[:, None, :], float("-inf"))
        allS = torch.cat([S, sink[None, :, None].expand(r1 - r0, H, 1)], dim=2)
        L = torch.logsumexp(allS, dim=2)
        P = torch.exp(S - L[:, :, None])
        o[r0:r1] = torch.einsum("rhk,rkd->rhd", P, K[:, :, :d_v]).to(torch.bfloat16)
        lse[r0:r1] = L
    return dict(x, o=o, lse=lse, scale=scale)


def dsa_flops(s_q, H, d_qk, topk, d_v=512, entries=None):
    """2 s_q H topk (3 d_qk + 2 d_v): S, dP, dQ, dK, dV over every listed key (the pull
    request's formula).  `entries`: the number of valid list entries over all rows, when rows
    are shorter than topk (causal lists), in place of s_q topk."""
    n = s_q * topk if entries is None else entries
    return 2.0 * n * H * (3 * d_qk + 2 * d_v)


def run_dsa(s_q, s_kv, H, d_qk, topk, causal=False, iters=100, warmup=20, build=True):
    """Time attn_dsa_bwd (its memsets and both kernels) with CUDA events (median of `iters`
    calls); one JSON line with TFLOPS by dsa_flops and the fraction of the measured dense
    BF16 peak."""
    import torch

    if build:
        import __graft_entry__
        __graft_entry__.build()
    import exact_attention_flashattention_gb300 as attn
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    x = dsa_prepare(s_q, s_kv, H, d_qk, topk, causal)
    dq = torch.empty_like(x["q"])
    dkv = torch.empty_like(x["kv"])
    dsink = torch.empty_like(x["sink"])
    ws = torch.empty(attn.attn_dsa_bwd_workspace_size(s_kv, d_qk), dtype=torch.uint8, device=dev)

    def call():
        attn.attn_dsa_bwd(x["q"], x["kv"], x["o"], x["do"], x["lse"], x["sink"], x["idx"], x["lens"], dq, dkv, dsink,
                          ws, x["scale"], causal, stream)

    ms = time_calls(call, stream, iters, warmup)
    if attn.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error word set")
    tf = dsa_flops(s_q, H, d_qk, topk, entries=int(x["lens"].sum().item())) / ms / 1e9
    print(json.dumps({"sweep": f"dsa bwd s={s_q} H={H} QK={d_qk} V=512 topk={topk}" + (" causal" if causal else ""),
                      "dtype": "bf16", "ms": ms, "tflops": tf, "pct_peak": 100 * tf / peak,
                      "peak_basis": f"dense BF16 {peak} TFLOPS ({src})"}), flush=True)
    return 0


def run_sweep(iters=100, warmup=20):
    """Forward and backward TFLOPS of every workload of the list (CUDA events around each
    call, `warmup` untimed and `iters` timed calls, median).  One JSON line per workload;
    not the bench contract line."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import exact_attention_flashattention_gb300 as attn
    from exact_attention_flashattention_gb300 import flops as F
    peaks, src = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    for name, B, H, N, d, causal, dtype, sig in SWEEP:
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        q, k = ((torch.randn((B, H, N, d), generator=g, device=dev) * sig).to(tdt) for _ in range(2))
        v, do = (torch.randn((B, H, N, d), generator=g, device=dev).to(tdt) for _ in range(2))
        o, lse = torch.empty_like(q), torch.empty((B, H, N), device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(attn.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        sc = d ** -0.5

        def timed(fn):
            return time_calls(fn, stream, iters, warmup)

        clk = ClockSampler(torch.cuda.current_device())
        clk.start()
        fms = timed(lambda: attn.attn_fwd(q, k, v, o, lse, sc, causal, stream))
        bms = timed(lambda: attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, sc, causal, stream))
        clocks = clk.stop()
        if attn.attn_last_device_error(stream) != 0:
            raise RuntimeError("device error word set")
        ftf = F.fwd_flops(B, H, N, d, causal) / fms / 1e9
        btf = F.bwd_flops(B, H, N, d, causal) / bms / 1e9
        line = {"sweep": name, "dtype": dtype, "fwd_ms": fms, "fwd_tflops": ftf, "bwd_ms": bms, "bwd_tflops": btf,
                "fwd_pct_burst_peak": 100 * ftf / burst, "bwd_pct_burst_peak": 100 * btf / burst,
                "burst_peak_basis": f"bf16 burst {burst} ({src})"}
        if clocks:
            nominal = nominal_bf16_tflops(n_sm, clocks["sm_mhz"])
            line.update({"fwd_pct_at_clock": 100 * ftf / nominal, "bwd_pct_at_clock": 100 * btf / nominal,
                         "clock_basis": f"{n_sm} SMs x {NOMINAL_FLOP_PER_CLK} FLOP/clk x {clocks['sm_mhz']:.0f} MHz "
                                        f"(median sampled) = {nominal:.1f} TFLOP/s", "clocks": clocks})
        print(json.dumps(line), flush=True)
        del q, k, v, do, o, lse, dq, dk, dv, ws
    # the same causal d = 128 work in the token-major layouts: BSHD, and 32 packed sequences of
    # lengths 512, 752, ..., 7952 (135424 tokens; most not a multiple of 128)
    lens = [512 + 240 * i for i in range(32)]
    for name, layout in (("layout BSHD causal B=8 H=16 N=4096 d=128", "bshd"),
                         (f"layout packed causal 32 sequences, {sum(lens)} tokens, H=16 d=128", "packed")):
        H, d = 16, 128
        if layout == "bshd":
            B, N = 8, 4096
            shape, cu, total, maxlen = (B, N, H, d), None, B * N, N
            flop_f, flop_b = F.fwd_flops(B, H, N, d, True), F.bwd_flops(B, H, N, d, True)
        else:
            B, total, maxlen = len(lens), sum(lens), max(lens)
            shape = (total, H, d)
            cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32, device=dev)
            flop_f = sum(F.fwd_flops(1, H, n, d, True) for n in lens)
            flop_b = sum(F.bwd_flops(1, H, n, d, True) for n in lens)
        g = torch.Generator(device=dev)
        g.manual_seed(13)
        q, k, v, do = (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N) if layout == "bshd" else (H, total), device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(attn.attn_bwd_layout_workspace_size(B, H, maxlen, d, layout, total), dtype=torch.uint8,
                         device=dev)
        sc = d ** -0.5

        def timed_l(fn):
            return time_calls(fn, stream, iters, warmup)

        fms = timed_l(lambda: attn.attn_fwd_layout(q, k, v, o, lse, sc, True, layout, cu, maxlen, stream))
        bms = timed_l(lambda: attn.attn_bwd_layout(q, k, v, o, do, lse, dq, dk, dv, ws, sc, True, layout, cu, maxlen,
                                                   stream))
        if attn.attn_last_device_error(stream) != 0:
            raise RuntimeError("device error word set")
        print(json.dumps({"sweep": name, "dtype": "bf16", "fwd_ms": fms, "fwd_tflops": flop_f / fms / 1e9,
                          "bwd_ms": bms, "bwd_tflops": flop_b / bms / 1e9}), flush=True)
        del q, k, v, do, o, lse, dq, dk, dv, ws
    for name, B, Hq, Hkv, N, d in DECODE_SWEEP:
        run_decode(name, B, Hq, Hkv, N, d, iters=iters, warmup=warmup, build=False)
    for s, H, d_qk, topk in DSA_SWEEP:
        run_dsa(s, s, H, d_qk, topk, iters=iters, warmup=warmup, build=False)
    return 0


def run_decode(name, B, Hq, Hkv, N, d, iters=100, warmup=20, build=True):
    """Decode against a key/value cache: HBM-bound, reported in GB/s of the cache bytes read
    (CUDA events, `warmup` untimed and `iters` timed calls of attn_decode, median).  One JSON
    line."""
    import torch

    if build:
        import __graft_entry__
        __graft_entry__.build()
    import exact_attention_flashattention_gb300 as attn
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    q = torch.randn((B, Hq, d), generator=g, device=dev).to(torch.bfloat16)
    kc, vc = (torch.randn((B, Hkv, N, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(2))
    o, lse = torch.empty_like(q), torch.empty((B, Hq), device=dev)
    ws = torch.empty(attn.attn_decode_workspace_size(B, Hq, Hkv, N, d), dtype=torch.uint8, device=dev)
    ms = time_calls(lambda: attn.attn_decode(q, kc, vc, o, lse, ws, d ** -0.5, None, stream), stream, iters,
                    warmup)
    if attn.attn_last_device_error(stream) != 0:
        raise RuntimeError("device error word set")
    cache_bytes = 2 * B * Hkv * N * d * 2          # K and V, each read once
    gbs = cache_bytes / ms / 1e6
    print(json.dumps({"sweep": name, "dtype": "bf16", "decode_us": 1e3 * ms, "cache_gb": cache_bytes / 1e9,
                      "gbs": gbs, "pct_hbm": 100 * gbs / hbm, "peak_basis": f"HBM copy {hbm} GB/s ({src})"}),
          flush=True)
    return 0


def spawn_ranks(n, argv):
    """Start n ranks of this script with torch.distributed.run on this node (one per GPU,
    LOCAL_RANK = GPU index) and return the launcher's exit code.  Rank 0 prints the line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="print fwd / bwd TFLOPS of every workload of the list instead of the bench line")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d[,noncausal][,fp16] instead of the default workload (smaller cases for profiling)")
    ap.add_argument("--dsa-shape", default=None,
                    help="s_q,s_kv,H,d_qk,topk[,causal]: time the sparse top-k backward on that shape")
    ap.add_argument("--decode-shape", default=None,
                    help="B,Hq,Hkv,N,d: time decode on that cache (--steps timed calls, --warmup untimed)")
    args = ap.parse_args()
    if args.shape:
        parts = args.shape.split(",")
        WORKLOAD.update(B=int(parts[0]), H=int(parts[1]), N=int(parts[2]), d=int(parts[3]),
                        causal="noncausal" not in parts[4:])
        global WORKLOAD_NAME, DTYPE
        DTYPE = "fp16" if "fp16" in parts[4:] else "bf16"
        WORKLOAD_NAME = ("{} MHA {} fwd+bwd B={B} H={H} N={N} d={d}, q,k,v,dO ~ N(0,1)"
                         .format("causal" if WORKLOAD["causal"] else "non-causal", DTYPE.upper(), **WORKLOAD))
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and not (args.sweep or args.decode_shape or args.dsa_shape):
        return spawn_ranks(args.gpus, sys.argv[1:])
    if args.sweep:
        return run_sweep()
    if args.decode_shape:
        B, Hq, Hkv, N, d = (int(x) for x in args.decode_shape.split(","))
        return run_decode(f"decode B={B} Hq={Hq} Hkv={Hkv} N={N} d={d}", B, Hq, Hkv, N, d, iters=args.steps,
                          warmup=args.warmup)
    if args.dsa_shape:
        parts = args.dsa_shape.split(",")
        s_q, s_kv, H, d_qk, topk = (int(x) for x in parts[:5])
        return run_dsa(s_q, s_kv, H, d_qk, topk, causal=len(parts) > 5 and parts[5] == "causal", iters=args.steps,
                       warmup=args.warmup)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
