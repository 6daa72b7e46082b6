"""Benchmark of the MLA prolog on one GB300 (or N independent replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {cuda,reference}]

One step = one mla_prolog() call (all kernels of the prolog) over one batch of synthetic
DeepSeek-V3-shaped input: T = 32 decode tokens (the headline workload).  The L2 cache is
flushed (a 2 x L2-size buffer is rewritten) before every timed step, outside the timed
events.  Rank 0 prints one JSON line.

--impl reference times the CPU oracle (fp64 C, OpenMP) on the host cores instead, on a
bounded sample of tokens of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "decode_t32"
PREFILL = "prefill_t8192"
PREPROCESS = "pp_decode_t32"
METRIC = "MLA prolog tokens/s & µs/call (T=32 decode, T=8192) + % HBM/tensor roofline"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ byte / flop model

def step_bytes(s, q_int8=False):
    """Algorithmic bytes of one call: every input read once, every output and cache row written once."""
    W = s.He * (s.Hcq + s.Hckv + s.Dr) + s.Hcq * s.N * (s.D + s.Dr) + s.N * s.D * s.Hckv
    per_tok = (s.He * 2 + 2 * s.Dr * 2 + 8 + s.N * s.Hckv * (1 if q_int8 else 2) + s.N * s.Dr * 2
               + s.Hckv * 2 + s.Dr * 2 + (s.N * 4 if q_int8 else 0))
    return W * 2 + (s.Hcq + s.Hckv) * 2 + s.T * per_tok


def int8_step_bytes(s, kv_int8=True):
    """Algorithmic bytes of one int8-input call (int8 tokenX and weights W^DQ, W^UqQr, W^DkvKr at
    one byte, W^UK bf16, fp32 scales, int8 queryOut with its (T, N, 1) scales, int8 kv rows)."""
    w8 = s.He * (s.Hcq + s.Hckv + s.Dr) + s.Hcq * s.N * (s.D + s.Dr)
    vectors = (s.Hcq + s.N * (s.D + s.Dr) + s.Hckv + s.Dr + s.Hckv) * 4 + (s.Hcq + s.Hckv) * 2
    per_tok = (s.He + 4 + 2 * s.Dr * 2 + 8 + s.N * s.Hckv + s.N * 4 + s.N * s.Dr * 2
               + s.Hckv * (1 if kv_int8 else 2) + s.Dr * 2)
    return w8 + s.N * s.D * s.Hckv * 2 + vectors + s.T * per_tok


def k2_bytes(s):
    """Up-projection c^Q . W^UqQr: the weight, c^Q in, q^C and q^R out (bf16)."""
    return s.Hcq * s.N * (s.D + s.Dr) * 2 + s.T * s.Hcq * 2 + s.T * s.N * (s.D + s.Dr) * 2


def k2_flops(s):
    return 2 * s.T * s.Hcq * s.N * (s.D + s.Dr)


def kernel_bytes(s):
    """Algorithmic bytes per launch of each kernel the library can launch for a bf16 call."""
    ncols1 = s.Hcq + s.Hckv + s.Dr
    return {
        # the whole prolog in one launch
        "decode_persist": step_bytes(s),
        # x . [W^DQ | W^DkvKr]: weights, x, fp32 product rows
        "k1_down_proj": s.He * ncols1 * 2 + s.T * s.He * 2 + s.T * ncols1 * 4,
        "k2_up_proj": k2_bytes(s),
        # q^C . W^UK per head: weights, q^C in, q^N out
        "k3_absorb_uk": s.N * s.D * s.Hckv * 2 + s.T * s.N * s.D * 2 + s.T * s.N * s.Hckv * 2,
    }


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
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
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ multi-rank timing

def job_rate(total_ms_local, tokens_per_rank, world, dist=None, device=None):
    """Whole-job throughput of N replicas (weak scaling: every rank runs the full workload):
    the units all ranks processed divided by the slowest rank's time (MAX over ranks).
    Returns (max total ms, tokens/s)."""
    import torch
    t = torch.tensor([float(total_ms_local)], dtype=torch.float64, device=device)
    if dist is not None and world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total = float(t.item())
    return total, tokens_per_rank * world / (total / 1e3)


# ------------------------------------------------------------------ GPU arm

def run_cuda(args, rank, world):
    import torch
    from attention_pre_processing_gb300 import build as cuda_build
    from attention_pre_processing_gb300 import workloads, mla_prolog, mla_prolog_timing_enable, mla_prolog_timing_read
    from attention_pre_processing_gb300.runner import PrologCall

    cuda_build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    peaks = _peaks()
    cfg = workloads.config(HEADLINE)
    s = cfg.shape
    inp = workloads.make_inputs(cfg)
    call = PrologCall(cfg, inp, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # Write 2 x L2 bytes, then read another 2 x L2 bytes: the call starts with none of its
        # data in L2 and with clean lines only (no write-back of the flush charged to it).
        flush_w.fill_(1)
        flush_r.sum()

    # warm-up
    for _ in range(args.warmup):
        flush_l2()
        call(stream)
    torch.cuda.synchronize(dev)
    if call.status(stream) != 0:
        raise RuntimeError("device status bits set during warm-up")

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        t_wall0 = time.perf_counter()
        for i in range(K):
            flush_l2()
            starts[i].record(stream)
            call(stream)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        t_wall = time.perf_counter() - t_wall0
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    if call.status(stream) != 0:
        raise RuntimeError("device status bits set during the timed region")
    total_ms, value = job_rate(sum(step_ms), s.T * K, world, dist, dev)
    ms_per_step = total_ms / K
    # the distribution over more calls: cold L2 (flushed before each call) and hot L2 (back to
    # back: the 128 MB of weights mostly stay in the 129 MB L2 between calls)
    dist_cold = _call_stats(call, stream, dev, 200, flush_l2)
    dist_hot = _call_stats(call, stream, dev, 200, None)

    # per-kernel durations (each kernel alone, events between kernels) for the roofline
    mla_prolog_timing_enable(True)
    per_kernel = {}
    for i in range(max(K, 10)):
        flush_l2()
        call(stream)
        for name, ms in mla_prolog_timing_read():
            per_kernel.setdefault(name, []).append(ms)
    mla_prolog_timing_enable(False)
    kern_ms = {k: statistics.mean(v) for k, v in per_kernel.items()}
    kernels_per_step = len(kern_ms)
    # the dominant kernel: the longest one of the call (the whole call when it is one launch)
    kb = kernel_bytes(s)
    dom = max((k for k in kern_ms if k in kb), key=lambda k: kern_ms[k], default=None)
    dom_ms = kern_ms.get(dom) if dom else None
    dom_bytes = kb.get(dom) if dom else None
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9 if dom_ms else None
    traffic = _read_traffic(dom, HEADLINE) if dom else None
    roofline = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": (achieved / peaks["hbm_gbs"]) if achieved else None,
                "traffic": traffic, "peak_source": peaks["source"] + " (HBM copy, burst)",
                "algorithmic_bytes": dom_bytes, "launch_ms": dom_ms,
                "timing": "CUDA events on the call's stream around the kernel, L2 flushed before each call"}

    # end to end: host inputs -> device, call, results -> host, every step
    e2e = _e2e(call, cfg, stream, dev, K, flush_l2)

    # whole-call roofline (bytes / measured HBM)
    sbytes = step_bytes(s)
    step_roof = {"bytes": sbytes, "achieved_gbs": sbytes / (ms_per_step / 1e3) / 1e9,
                 "frac_of_measured_hbm": sbytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
                 "frac_of_nominal_8tbs": sbytes / (ms_per_step / 1e3) / 1e9 / 8000.0}

    prefill = None
    if not args.skip_prefill:
        prefill = _prefill(dev, stream, flush_l2, peaks, max(3, min(K, 10)))

    pre = None
    if not args.skip_preprocess:
        pre = _preprocess(dev, stream, flush_l2, peaks, max(3, min(K, 20)))

    # the other two DeepSeek-V3-shaped configurations: T = 256 with the int8 q^N output, and
    # int8 inputs at T = 64
    others = {}
    if not args.skip_others:
        for name, nbytes in (("decode_t256_qint8", lambda c: step_bytes(c.shape, q_int8=True)),
                             ("int8_t64", lambda c: int8_step_bytes(c.shape))):
            others[name] = _other(name, nbytes, dev, stream, flush_l2, peaks, max(3, min(K, 50)))

    cpu = None
    cpu_1t = None
    if rank == 0 and not args.skip_cpu:
        cpu = cpu_baseline(cfg, inp, budget_s=args.cpu_budget)
        cpu_1t = {}
        for name in ("tiny", "decode_t32", "decode_t256_qint8", "int8_t64"):
            c = workloads.config(name)
            cpu_1t[name] = cpu_baseline(c, workloads.make_inputs(c), budget_s=2.0, threads=1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_call": ms_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, DeepSeek-V3-shaped random weights)",
            "config": dict(workload_config(cfg, world),
                           l2=("flushed before every step: 2 x L2 bytes written, then another 2 x L2 bytes "
                               "read, outside the timed events"),
                           timing="CUDA events around each mla_prolog call on its stream"),
            "roofline": roofline, "step_roofline": step_roof, "kernels_ms": kern_ms,
            "gpu_launches": kernels_per_step * K,
            "us_per_call_mean": statistics.mean(step_ms) * 1e3,
            "us_per_call_median": statistics.median(step_ms) * 1e3,
            "calls_200_cold_l2": dist_cold, "calls_200_hot_l2": dist_hot,
            "clocks": clk.summary(), "e2e": e2e, "wall_s_timed": t_wall,
            "cpu_baseline": cpu, "cpu_oracle_1_thread": cpu_1t, "prefill": prefill, "preprocess": pre,
            "other_configs": others,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def _call_stats(call, stream, dev, n, flush_l2):
    """µs per call over n event-timed calls: median, mean, 10th and 90th percentile.  With
    flush_l2 the L2 is flushed before each call (outside the events); without it the calls run
    back to back with whatever the previous call left in L2 (labelled hot L2)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        if flush_l2 is not None:
            flush_l2()
        starts[i].record(stream)
        call(stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends))
    return {"calls": n, "l2": "flushed before each call" if flush_l2 is not None else "hot (no flush)",
            "us_median": statistics.median(us), "us_mean": statistics.mean(us),
            "us_p10": us[n // 10], "us_p90": us[(9 * n) // 10],
            "tokens_per_s_median": call.cfg.shape.T / (statistics.median(us) / 1e6)}


def _other(name, nbytes, dev, stream, flush_l2, peaks, K):
    """One more configuration beside the headline: µs per call (cold L2), tokens/s, algorithmic
    bytes against the measured HBM bandwidth, and each kernel's own duration."""
    import torch
    from attention_pre_processing_gb300 import workloads, mla_prolog_timing_enable, mla_prolog_timing_read
    from attention_pre_processing_gb300.runner import PrologCall
    cfg = workloads.config(name)
    call = PrologCall(cfg, workloads.make_inputs(cfg), device=dev)
    for _ in range(3):
        flush_l2()
        call(stream)
    st = _call_stats(call, stream, dev, K, flush_l2)
    mla_prolog_timing_enable(True)
    per = {}
    for _ in range(min(K, 10)):
        flush_l2()
        call(stream)
        for kname, t in mla_prolog_timing_read():
            per.setdefault(kname, []).append(t)
    mla_prolog_timing_enable(False)
    kern = {k: statistics.mean(v) for k, v in per.items()}
    b = nbytes(cfg)
    ok = call.status(stream) == 0
    del call
    torch.cuda.empty_cache()
    ms = st["us_median"] / 1e3
    return {"workload": cfg.workload, "us_per_call_median": st["us_median"], "us_per_call_mean": st["us_mean"],
            "tokens_per_s": cfg.shape.T / (ms / 1e3), "algorithmic_bytes": b,
            "achieved_gbs": b / (ms / 1e3) / 1e9, "frac_of_measured_hbm": b / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "kernels_ms": kern, "launches_per_call": len(kern), "status_clean": ok,
            "traffic": _read_traffic(max(kern, key=kern.get), name) if kern else None,
            "dominant_kernel": max(kern, key=kern.get) if kern else None}


def _read_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, when one exists for this kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return j.get(workload, {}).get(kernel)
    except Exception:
        return None


def _e2e(call, cfg, stream, dev, K, flush_l2):
    """The headline call end to end: each step copies its inputs (tokenX, rope tables,
    cacheIndex) from pinned host memory, runs mla_prolog through the C ABI and reads queryOut and
    queryRopeOut back into pinned host memory, all on the call's stream, inside the step's events.
    The per-token tensors are views of one device buffer each way (PrologCall packed_io), so a
    step makes one copy in each direction."""
    import torch
    from attention_pre_processing_gb300.runner import PrologCall
    from attention_pre_processing_gb300 import workloads
    s = cfg.shape
    pc = PrologCall(cfg, workloads.make_inputs(cfg), device=dev, packed_io=True)
    host_in = pc.io_in.cpu().pin_memory()
    host_out = torch.empty(pc.io_out.shape, dtype=torch.uint8, pin_memory=True)
    bi = host_in.numel()
    bo = host_out.numel()
    with torch.cuda.stream(stream):
        for _ in range(3):
            pc.io_in.copy_(host_in, non_blocking=True)
            pc(stream)
            host_out.copy_(pc.io_out, non_blocking=True)
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            flush_l2()
            starts[i].record(stream)
            pc.io_in.copy_(host_in, non_blocking=True)
            pc(stream)
            host_out.copy_(pc.io_out, non_blocking=True)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K
    return {"value": s.T / (ms / 1e3), "unit": "tokens/s", "us_per_call": ms * 1e3,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "copies_per_step": 2,
            "path": "pinned host -> device copy of the per-token inputs, mla_prolog (C ABI), "
                    "device -> pinned host copy of queryOut | queryRopeOut"}


def _prefill(dev, stream, flush_l2, peaks, K):
    """T = 8192 prefill, reported beside the headline (tensor-core bound)."""
    import torch
    from attention_pre_processing_gb300 import workloads, mla_prolog_timing_enable, mla_prolog_timing_read
    from attention_pre_processing_gb300.runner import PrologCall
    cfg = workloads.config(PREFILL)
    s = cfg.shape
    inp = workloads.make_inputs(cfg)
    call = PrologCall(cfg, inp, device=dev)
    for _ in range(3):
        call(stream)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush_l2()
        starts[i].record(stream)
        call(stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K
    mla_prolog_timing_enable(True)
    per = {}
    for _ in range(K):
        flush_l2()
        call(stream)
        for name, t in mla_prolog_timing_read():
            per.setdefault(name, []).append(t)
    mla_prolog_timing_enable(False)
    kern = {k: statistics.mean(v) for k, v in per.items()}
    flops = workloads.flops_per_token(s) * s.T
    k2 = kern.get("k2_up_proj")
    k2_tf = k2_flops(s) / (k2 / 1e3) / 1e12 if k2 else None
    ok = call.status(stream) == 0
    del call
    torch.cuda.empty_cache()
    return {"workload": cfg.workload, "us_per_call": ms * 1e3, "tokens_per_s": s.T / (ms / 1e3),
            "tflops": flops / (ms / 1e3) / 1e12, "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
            "roofline_k2": {"bound": "tensor", "achieved": k2_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": (k2_tf / peaks["bf16_tflops"]) if k2_tf else None},
            "kernels_ms": kern, "status_clean": ok}


def pp_bytes(cfg):
    """Algorithmic bytes of one aclnnMlaPreprocess call: every input read once (int8 weights at one
    byte), qOut written once, one cache row per token."""
    s = cfg.shape
    n1, n2 = s.Hcq + s.Hckv + s.Dr, s.N * (s.D + s.Dr)
    e = 2   # bf16 / fp16
    weights = n1 * s.He + n2 * s.Hcq + s.N * s.D * s.Hckv * e
    vectors = (n1 + n2) * 4 * (2 if cfg.with_bias else 1) + (2 * s.He + 2 * s.Hcq + s.Hckv + 2) * e + 2
    per_token = s.He * e + 2 * s.Dr * e + 4 + s.N * (s.Hckv + s.Dr) * e + (s.Hckv + s.Dr) * e
    return weights + vectors + s.T * per_token


def _preprocess(dev, stream, flush_l2, peaks, K):
    """The aclnnMlaPreprocess variant at T = 32 (DeepSeek-V3 shapes, int8 weights), beside the headline."""
    import torch
    from attention_pre_processing_gb300 import workloads, mla_prolog_timing_enable, mla_prolog_timing_read
    from attention_pre_processing_gb300.runner import PreprocessCall
    cfg = workloads.pp_config(PREPROCESS)
    s = cfg.shape
    call = PreprocessCall(cfg, workloads.make_pp_inputs(cfg), device=dev)
    for _ in range(3):
        flush_l2()
        call(stream)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush_l2()
        starts[i].record(stream)
        call(stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K
    mla_prolog_timing_enable(True)
    per = {}
    for _ in range(K):
        flush_l2()
        call(stream)
        for name, t in mla_prolog_timing_read():
            per.setdefault(name, []).append(t)
    mla_prolog_timing_enable(False)
    kern = {k: statistics.mean(v) for k, v in per.items()}
    b = pp_bytes(cfg)
    ok = call.status(stream) == 0
    del call
    torch.cuda.empty_cache()
    return {"workload": cfg.workload, "us_per_call": ms * 1e3, "tokens_per_s": s.T / (ms / 1e3),
            "algorithmic_bytes": b, "achieved_gbs": b / (ms / 1e3) / 1e9,
            "frac_of_measured_hbm": b / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "kernels_ms": kern, "gpu_launches_per_call": len(kern), "status_clean": ok}


# ------------------------------------------------------------------ CPU oracle

def cpu_baseline(cfg, inp, budget_s=12.0, steps=None, threads=None):
    """Times the oracle on growing token samples until ~budget_s of CPU work, on all host
    cores (or on `threads` threads)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from attention_pre_processing_gb300 import workloads

    class Dims:
        pass

    d = Dims()
    for k in ("T", "He", "Hcq", "N", "D", "Dr", "Hckv", "block_num", "block_size"):
        setattr(d, k, getattr(cfg.shape, k))
    oracle.build()
    if threads is None:
        threads = os.cpu_count() or oracle.max_threads()
    done, elapsed, n = 0, 0.0, max(1, threads)
    while elapsed < budget_s:
        tok = (workloads.sample_tokens(cfg.shape.T, n, seed=done + 1) if n < cfg.shape.T
               else list(range(cfg.shape.T)))
        t0 = time.perf_counter()
        oracle.prolog(inp, dims=d, eps_cq=cfg.eps_cq, eps_ckv=cfg.eps_ckv, x_int8=cfg.x_int8,
                      uqqr_int8=cfg.x_int8 or cfg.uqqr_int8, kv_int8=cfg.kv_int8, kr_int8=cfg.kr_int8,
                      q_int8=cfg.q_int8, tokens=tok, with_intermediates=False, num_threads=threads)
        elapsed += time.perf_counter() - t0
        done += len(tok)
        n = min(n * 2, cfg.shape.T)
    return {"value": done / elapsed, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} tokens of {cfg.workload} in {elapsed:.1f} s (fp64 C, OpenMP over tokens)"}


def workload_config(cfg, world):
    """The workload keys of a bench line's config: the same on both arms."""
    s = cfg.shape
    return {"workload": cfg.workload, "T": s.T, "He": s.He, "Hcq": s.Hcq, "N": s.N, "D": s.D, "Dr": s.Dr,
            "Hckv": s.Hckv, "kv_cache": f"{s.block_num}x{s.block_size}", "global_batch": s.T * world,
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from attention_pre_processing_gb300 import workloads
    cfg = workloads.config(HEADLINE)
    inp = workloads.make_inputs(cfg)
    budget = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(cfg, inp, budget_s=0.5)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(cfg, inp, budget_s=budget))
    wall = time.perf_counter() - t0
    tok = sum(float(v["sample"].split()[0]) for v in vals)
    value = tok / sum(float(v["sample"].split(" in ")[1].split()[0]) for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, DeepSeek-V3-shaped random weights)",
            "config": dict(workload_config(cfg, world),
                           timing="wall clock of the oracle's token loop on the host cores (OpenMP over tokens)"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": f"{int(tok)} tokens over {args.steps} steps"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_kernels_only(args):
    """Just `warmup + steps` prolog calls on one workload (no flush, no extras): the command
    the ncu captures profile."""
    import torch
    from attention_pre_processing_gb300 import build as cuda_build
    from attention_pre_processing_gb300 import workloads
    from attention_pre_processing_gb300.runner import PrologCall, PreprocessCall
    cuda_build.build()
    if args.workload.startswith("pp_"):   # the aclnnMlaPreprocess variant
        cfg = workloads.pp_config(args.workload, **({"T": args.T} if args.T else {}))
        call = PreprocessCall(cfg, workloads.make_pp_inputs(cfg))
        for _ in range(args.warmup + args.steps):
            call()
        torch.cuda.synchronize()
        if call.status() != 0:
            raise SystemExit("device status bits set")
        return
    cfg = workloads.config(args.workload)
    if args.T:
        over = {"T": args.T}
        if cfg.sequences is not None:   # same number of sequences, shorter ones
            over["sequences"] = (cfg.sequences[0], args.T // cfg.sequences[0])
        cfg = workloads.config(args.workload, **over)
    call = PrologCall(cfg, workloads.make_inputs(cfg))
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    if call.status() != 0:
        raise SystemExit("device status bits set")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-preprocess", action="store_true", help="skip the aclnnMlaPreprocess variant's line")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-others", action="store_true", help="skip the T=256 int8-q^N and int8-input lines")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--kernels-only", action="store_true", help="only warmup+steps calls of --workload")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--T", type=int, default=0, help="--kernels-only: token count other than the workload's")
    args = ap.parse_args()
    if args.kernels_only:
        run_kernels_only(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_cuda(args, rank, world)


if __name__ == "__main__":
    main()
