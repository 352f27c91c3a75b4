"""Benchmark: causal GQA prefill TFLOP/s at S=10231 (Hq=64, Hkv=8, D=128).

One step = one h3gqa_causal_fwd call over the whole workload (every query
row of every head), inputs resident in HBM. L2 is flushed (a 256 MB write)
before every step, outside the per-step CUDA events; the reported time is the
sum of the per-step kernel times measured with CUDA events on the launching
stream. Rank 0 prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload s10231]
  python bench.py --impl reference ...   # the fp64 CPU oracle, bounded sample

Multi-GPU: one process per GPU (torchrun); every rank runs an independent
replica of the workload (no data-path collective); value = all ranks' FLOPs
/ the slowest rank's time.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from long_causal_gqa_gb300 import binding  # noqa: E402
from long_causal_gqa_gb300.inputs import (HEADLINE, WORKLOADS, make_workload_inputs,  # noqa: E402
                                         norm_weights, rope_tables)

METRIC = "causal GQA prefill TFLOP/s at S=10231 (Hq64/Hkv8/D128), % of BF16 peak"
EPILOGUES = {"bf16_head": (False, False), "bf16_token": (True, False), "int8_token": (True, True),
             "int8_head": (False, True)}


def metric_name(w, epilogue, prologue=False):
    if w.name == HEADLINE and epilogue == "bf16_head" and not prologue:
        return METRIC
    kind = "causal GQA prefill" if w.causal else "bidirectional GQA attention"
    return "%s TFLOP/s, workload %s (Hq%d/Hkv%d/D%d), output %s%s" % (
        kind, w.name, w.n_q_heads, w.n_kv_heads, w.head_dim, epilogue,
        ", with Q/K RMS-norm + RoPE prologue" if prologue else "")
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def kernel_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    or None when there is none or the kernel sources changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "causal_gqa_fwd_%s.json" % workload)
    try:
        with open(path) as f:
            prof = json.load(f)
        h = hashlib.sha256()
        for rel in prof["kernel_source_files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != prof["kernel_source_sha256"]:
            return None
        return float(prof["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.samples = []
        self._stop = threading.Event()
        self._thread = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(
                    ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                     "--format=csv,noheader,nounits"], capture_output=True, text=True,
                    timeout=5).stdout.strip()
                if out:
                    self.samples.append((time.time(), [c.strip() for c in out.split(",")]))
            except (OSError, subprocess.SubprocessError):
                return
            self._stop.wait(0.05)

    def start(self):
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=10)

    def summary(self, t0, t1):
        inside = [s for t, s in self.samples if t0 - 0.1 <= t <= t1 + 0.1] or \
                 [s for _, s in self.samples]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        sm = [float(s[0]) for s in inside if s[0].replace(".", "").isdigit()]
        smax = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 3 + i and s[3 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_rank, world, ms_slowest):
    """TFLOP/s of the whole job: every rank's FLOPs over the slowest rank's time."""
    return flops_per_rank * world / (ms_slowest * 1e-3) / 1e12


def oracle_sample_rate(x, w, seconds, seed):
    """Times the fp64 oracle on a seeded sample of (head, row) pairs of the
    workload for about `seconds`; returns (TFLOP/s, description, cores, n_rows)."""
    from oracle import causal_gqa as orc
    cu = x["cu_seqlens"].numpy()
    starts = np.repeat(cu[:-1], np.diff(cu))
    rng = np.random.default_rng(seed)
    T = int(cu[-1])

    ends = np.repeat(cu[1:], np.diff(cu))

    def run(n):
        rows = np.stack([rng.integers(0, w.n_q_heads, n), rng.integers(0, T, n)], axis=1)
        if w.causal:
            keys = rows[:, 1] - starts[rows[:, 1]] + 1
        else:
            keys = ends[rows[:, 1]] - starts[rows[:, 1]]
        t0 = time.perf_counter()
        orc.causal_gqa_rows(x["q"], x["k"], x["v"], cu, w.n_q_heads, w.n_kv_heads, w.scale, rows,
                            causal=w.causal)
        dt = time.perf_counter() - t0
        return float(keys.sum()) * 4 * w.head_dim, dt

    flops, dt = run(64)                      # calibration
    n = int(max(64, min(2_000_000, 64 * seconds / max(dt, 1e-3))))
    flops, dt = run(n)
    desc = ("%d random (head, query row) pairs of %s, each row's full attention in fp64; "
            "FLOPs counted as 4*D per visible (query, key) pair" % (n, w.name))
    return flops / dt / 1e12, desc, orc.max_threads(), n


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample of rows."""
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    x = make_workload_inputs(w)
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    rates = []
    desc, cores = "", 0
    for i in range(args.warmup + args.steps):
        r, desc, cores, _ = oracle_sample_rate(x, w, per_step, seed=w.seed + i)
        if i >= args.warmup:
            rates.append(r)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": metric_name(w, args.epilogue), "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": w.metric_flops() / (value * 1e12) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "seqlens": list(w.seqlens), "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + "; %.1f s per step" % per_step},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    binding.load()
    w = WORKLOADS[args.workload]
    token_major, out_int8 = EPILOGUES[args.epilogue]
    x = make_workload_inputs(w)
    cu = x["cu_seqlens"]
    plan = binding.h3gqa_attention_plan(cu, w.n_q_heads, w.n_kv_heads, w.head_dim, w.causal)
    stream = torch.cuda.Stream(device)
    q, k, v = (x[n].to(device) for n in ("q", "k", "v"))
    oshape = (w.total_tokens, w.n_q_heads, w.head_dim) if token_major else tuple(q.shape)
    o = torch.empty(oshape, dtype=torch.int8 if out_int8 else torch.bfloat16, device=device)
    o_scale = (torch.empty(oshape[:2], dtype=torch.float32, device=device) if out_int8
               else None)
    lse = torch.empty((w.n_q_heads, w.total_tokens), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    sh = stream.cuda_stream
    default_call = w.causal and args.epilogue == "bf16_head" and not args.prologue
    pro = {}
    if args.prologue:
        wq, wk = norm_weights(w.head_dim, w.seed)
        cos, sin = rope_tables(w.seqlens, w.head_dim)
        pro = dict(wq=wq.to(device), wk=wk.to(device), cos=cos.to(device), sin=sin.to(device),
                   k_out=torch.empty_like(k))
    opts = binding.make_options(
        w.causal, binding.H3GQA_LAYOUT_TOKEN_MAJOR if token_major
        else binding.H3GQA_LAYOUT_HEAD_MAJOR, out_int8,
        o_scale.data_ptr() if o_scale is not None else None, 0,
        *([pro["wq"].data_ptr(), pro["wk"].data_ptr(), pro["cos"].data_ptr(),
           pro["sin"].data_ptr(), pro["k_out"].data_ptr()] if pro else []))

    def launch():
        if default_call:
            binding.h3gqa_causal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), cu, w.n_q_heads, w.n_kv_heads,
                                     w.head_dim, w.scale, sh)
        else:
            binding.h3gqa_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), cu, w.n_q_heads, w.n_kv_heads,
                                        w.head_dim, w.scale, opts, sh)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            launch()
    binding.h3gqa_sync_and_check(sh)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(device)
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    t1 = time.time()
    sampler.stop()
    binding.h3gqa_sync_and_check(sh)
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = float(np.mean(times))
    ms_max = max_over_ranks(ms, world, device)

    # End to end: every step copies its inputs from pinned host memory, runs
    # the kernel and reads o and lse back. Steps are pipelined the way a
    # caller would run them: copies in, compute and copies out on three
    # streams with two device buffer sets, so step i+1's upload and step
    # i-1's download overlap step i's kernel.
    qh, kh, vh = (x[n].pin_memory() for n in ("q", "k", "v"))
    oh = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    sch = (torch.empty(o_scale.shape, dtype=o_scale.dtype, pin_memory=True)
           if o_scale is not None else None)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size() + \
        (sch.numel() * sch.element_size() if sch is not None else 0)
    bufs = [dict(q=q, k=k, v=v, o=o, lse=lse, sc=o_scale)]
    bufs.append(dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                     o=torch.empty_like(o), lse=torch.empty_like(lse),
                     sc=torch.empty_like(o_scale) if o_scale is not None else None))
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    e2e_steps = max(4, min(args.steps, 20))
    n_total = e2e_steps + 2
    ev_in = [torch.cuda.Event() for _ in range(n_total)]
    ev_comp = [torch.cuda.Event() for _ in range(n_total)]
    ev_out = [torch.cuda.Event() for _ in range(n_total)]

    def e2e_step(i):
        b = bufs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])          # this buffer's inputs are free
            b["q"].copy_(qh, non_blocking=True)
            b["k"].copy_(kh, non_blocking=True)
            b["v"].copy_(vh, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])             # this buffer's outputs were read
        bopts = binding.make_options(
            w.causal, opts.out_layout, out_int8, b["sc"].data_ptr() if b["sc"] is not None else None,
            0, opts.q_norm_weight, opts.k_norm_weight, opts.rope_cos, opts.rope_sin, opts.k_out,
            opts.norm_eps)
        binding.h3gqa_attention_fwd(b["q"].data_ptr(), b["k"].data_ptr(), b["v"].data_ptr(),
                                    b["o"].data_ptr(), b["lse"].data_ptr(), cu, w.n_q_heads,
                                    w.n_kv_heads, w.head_dim, w.scale, bopts, sh)
        ev_comp[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[i])
            oh.copy_(b["o"], non_blocking=True)
            lh.copy_(b["lse"], non_blocking=True)
            if sch is not None:
                sch.copy_(b["sc"], non_blocking=True)
            ev_out[i].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(device)
    te0 = time.perf_counter()
    for i in range(2, n_total):
        e2e_step(i)
    torch.cuda.synchronize(device)
    e2e_ms = (time.perf_counter() - te0) * 1e3 / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    binding.h3gqa_sync_and_check(sh)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    value = whole_job_value(w.metric_flops(), world, ms_max)
    achieved = plan.causal_flops / (ms * 1e-3) / 1e12
    line = {
        "metric": metric_name(w, args.epilogue, args.prologue), "value": value, "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 q/k/v; no dataset)",
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "config": {"workload": w.name, "seqlens": list(w.seqlens), "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "causal": w.causal,
                   "output": args.epilogue, "qk_prologue": bool(args.prologue),
                   "scale": w.scale, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed before every step (256 MB write, outside the kernel events)",
                   "flops_per_step_metric": w.metric_flops(),
                   "flops_per_step_causal_exact": plan.causal_flops},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak,
                     "traffic": kernel_traffic(w.name)
                     if args.epilogue == "bf16_head" and not args.prologue else None,
                     "traffic_unit": "bytes per launch (ncu dram read+write)",
                     "peak_source": "%s bf16_tflops (burst)" % peak_src,
                     "kernel": "h3gqa::causal_gqa_fwd_kernel",
                     "work": "4*D FLOPs per visible (query, key, head) pair per launch"},
        "e2e": {"value": whole_job_value(w.metric_flops(), world, e2e_ms), "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "h3gqa_attention_fwd via the Python binding; pinned host buffers; "
                       "upload / compute / download on three streams, two device buffer sets"},
        "gpu_launches": args.steps * (2 if args.prologue else 1),
        "clocks": sampler.summary(t0, t1),
        "kernel_ms": {"mean": ms, "min": float(np.min(times)), "max": float(np.max(times))},
    }
    if not args.no_cpu_baseline:
        r, desc, cores, _ = oracle_sample_rate(x, w, args.cpu_seconds, seed=w.seed)
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--epilogue", choices=sorted(EPILOGUES), default="bf16_head",
                    help="output form: bf16 or int8 codes (+ per-row scales), head- or token-major")
    ap.add_argument("--prologue", action="store_true",
                    help="add the Q/K RMS-norm + rotary prologue (K pass + Q in-kernel)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
