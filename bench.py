"""Benchmark: causal GQA prefill TFLOP/s at S=10231 (Hq=64, Hkv=8, D=128).

One step = one h3gqa_causal_fwd call over the whole workload (every query
row of every head), inputs resident in HBM. L2 is flushed (a 256 MB write)
before every step, outside the per-step CUDA events; the reported time is the
mean of the per-step kernel times measured with CUDA events on the launching
stream. Rank 0 prints one JSON line. After the headline's timed region the
same line measures the other long workloads (the packed 4-sequence batch and
S=32768 with outlier channels) under `extra_workloads`, each with its own
clock record.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload s10231]
  python bench.py --impl reference ...   # the fp64 CPU oracle, bounded sample
  torchrun ... bench.py --gpus N --shard heads   # one problem split by KV heads

Multi-GPU: one process per GPU (torchrun). By default every rank runs an
independent replica of the workload (weak scaling, no data-path
collective); value = all ranks' FLOPs / the slowest rank's time. With
--shard heads the ranks split one workload's KV heads into contiguous ranges
(strong scaling, again no data-path collective: the heads are independent);
value = the workload's FLOPs / the slowest rank's time.
"""
import argparse
import ctypes
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
EXTRA_WORKLOADS = ("varlen4", "s32768_outlier")


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


# ----------------------------------------------------------------- clocks
REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlSampler:
    """Read-only NVML queries (SM clock, max SM clock, power, clock event
    reasons) of one GPU about every millisecond, on a background thread, so a
    timed region of a few tens of milliseconds still gets tens of samples.
    Only getters are called: no setting of the GPU is changed."""

    def __init__(self, device_index, period_s=0.001):
        self.period = period_s
        self.samples = []            # (time, sm_mhz, power_w, reasons bitmask)
        self._stop = threading.Event()
        self._thread = None
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.nv = nv
        self.handle = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(device_index)
        bus = ("%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id,
                                     props.pci_device_id)).encode()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.handle)):
            raise OSError("no NVML device at %s" % bus.decode())
        self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        nv.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))     # 1 = SM clock
        self.sm_max = float(mx.value)

    def _one(self):
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)):
            return None
        self.nv.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(pw))
        self._reasons(self.handle, ctypes.byref(rs))
        return (time.perf_counter(), float(clk.value), pw.value / 1000.0, int(rs.value))

    def _run(self):
        while not self._stop.is_set():
            s = self._one()
            if s is not None:
                self.samples.append(s)
            time.sleep(self.period)

    def start(self):
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join(timeout=10)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no samples"],
                    "samples": 0, "source": "nvml"}
        reasons = sorted({name for s in inside for bit, name in REASON_BITS.items()
                          if s[3] & bit})
        return {"sm_mhz": float(np.median([s[1] for s in inside])), "sm_max_mhz": self.sm_max,
                "sm_mhz_min": float(min(s[1] for s in inside)),
                "power_w_max": float(max(s[2] for s in inside)), "reasons": reasons,
                "samples": len(inside), "window_ms": (t1 - t0) * 1e3,
                "source": "nvml, read-only queries every %.1f ms" % (self.period * 1e3)}


class SmiSampler:
    """Fallback: nvidia-smi clock / clock-event-reason samples."""
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
                    self.samples.append((time.perf_counter(), [c.strip() for c in out.split(",")]))
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
                "reasons": reasons, "samples": len(inside), "source": "nvidia-smi"}


def make_sampler(local):
    try:
        return NvmlSampler(local)
    except (OSError, AttributeError):
        return SmiSampler(local)


# -------------------------------------------------------------- ranks
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


def shard_of(args, w, world, rank):
    """KV heads (begin, count) this rank computes: all of them for replicas,
    a contiguous balanced range with --shard heads."""
    if args.shard == "heads":
        return binding.shard_heads(w.n_kv_heads, world, rank)
    return 0, w.n_kv_heads


def config_of(w, args, world):
    """The workload and the protocol, as both arms report them."""
    return {"workload": w.name, "seqlens": list(w.seqlens), "n_q_heads": w.n_q_heads,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "causal": w.causal,
            "output": args.epilogue, "qk_prologue": bool(args.prologue), "scale": w.scale,
            "parallelism": ("heads" if args.shard == "heads" else "replicas") if world > 1
            else "single",
            "l2": "flushed before every step (256 MB write, outside the kernel events)",
            "flops_per_step_metric": w.metric_flops(),
            "flops_per_step_causal_exact": w.exact_flops()}


# ---------------------------------------------------------- reference arm
def oracle_sample_rate(x, w, seconds, seed):
    """Times the fp64 oracle on a seeded sample of (head, row) pairs of the
    workload for about `seconds`; returns (TFLOP/s, description, cores,
    seconds actually timed)."""
    from oracle import causal_gqa as orc
    cu = x["cu_seqlens"].numpy()
    starts = np.repeat(cu[:-1], np.diff(cu))
    ends = np.repeat(cu[1:], np.diff(cu))
    rng = np.random.default_rng(seed)
    T = int(cu[-1])

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
    return flops / dt / 1e12, desc, orc.max_threads(), dt


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample of rows."""
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    x = make_workload_inputs(w)
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    rates, secs = [], []
    desc, cores = "", 0
    for i in range(args.warmup + args.steps):
        r, desc, cores, dt = oracle_sample_rate(x, w, per_step, seed=w.seed + i)
        if i >= args.warmup:
            rates.append(r)
            secs.append(dt)
    value = float(np.mean(rates))
    sample_s = float(np.mean(secs))
    line = {
        "impl": "reference", "metric": metric_name(w, args.epilogue, args.prologue),
        "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": w.metric_flops() / (value * 1e12) * 1e3,
        "ms_per_step_kind": "extrapolated from sample: one full pass of the workload at the "
                            "sampled rate (the timed steps each ran the sample below)",
        "sample_s_per_step": sample_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16 q/k/v; no dataset)",
        "config": config_of(w, args, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + "; %.2f s timed per step" % sample_s},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- our arm
class Case:
    """Device buffers and the launch of one workload (one rank's shard)."""

    def __init__(self, w, args, device, stream, kv_range):
        self.w = w
        self.token_major, self.out_int8 = EPILOGUES[args.epilogue]
        self.x = make_workload_inputs(w)
        self.cu = self.x["cu_seqlens"]
        self.kv_begin, self.kv_count = kv_range
        self.plan = binding.h3gqa_attention_plan(self.cu, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                 w.causal)
        self.frac_heads = self.kv_count / w.n_kv_heads
        self.q, self.k, self.v = (self.x[n].to(device) for n in ("q", "k", "v"))
        T = w.total_tokens
        oshape = (T, w.n_q_heads, w.head_dim) if self.token_major else tuple(self.q.shape)
        self.o = torch.empty(oshape, dtype=torch.int8 if self.out_int8 else torch.bfloat16,
                             device=device)
        self.o_scale = (torch.empty(oshape[:2], dtype=torch.float32, device=device)
                        if self.out_int8 else None)
        self.lse = torch.empty((w.n_q_heads, T), dtype=torch.float32, device=device)
        self.sh = stream.cuda_stream
        self.default_call = (w.causal and args.epilogue == "bf16_head" and not args.prologue
                             and self.kv_count == w.n_kv_heads)
        self.launches_per_step = 2 if args.prologue else 1
        pro = {}
        if args.prologue:
            wq, wk = norm_weights(w.head_dim, w.seed)
            cos, sin = rope_tables(w.seqlens, w.head_dim)
            pro = dict(wq=wq.to(device), wk=wk.to(device), cos=cos.to(device),
                       sin=sin.to(device), k_out=torch.empty_like(self.k))
        self.pro = pro
        self.opts = self.options(self.o_scale)

    def options(self, o_scale):
        p = self.pro
        return binding.make_options(
            self.w.causal, binding.H3GQA_LAYOUT_TOKEN_MAJOR if self.token_major
            else binding.H3GQA_LAYOUT_HEAD_MAJOR, self.out_int8,
            o_scale.data_ptr() if o_scale is not None else None, self.kv_begin,
            *([p["wq"].data_ptr(), p["wk"].data_ptr(), p["cos"].data_ptr(), p["sin"].data_ptr(),
               p["k_out"].data_ptr()] if p else [None] * 5),
            1e-6, self.kv_count)

    def launch(self, q=None, k=None, v=None, o=None, lse=None, opts=None):
        w = self.w
        q, k, v = q if q is not None else self.q, k if k is not None else self.k, \
            v if v is not None else self.v
        o, lse = o if o is not None else self.o, lse if lse is not None else self.lse
        if self.kv_count == 0:
            return
        if self.default_call and opts is None:
            binding.h3gqa_causal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), self.cu, w.n_q_heads, w.n_kv_heads,
                                     w.head_dim, w.scale, self.sh)
        else:
            binding.h3gqa_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), self.cu, w.n_q_heads, w.n_kv_heads,
                                        w.head_dim, w.scale, opts or self.opts, self.sh)


def time_steps(case, steps, warmup, stream, flush, device, world):
    """Warm-up, then `steps` launches each preceded by an L2 flush, timed with
    CUDA events on the launching stream. Returns (per-step ms list, t0, t1)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.fill_(1.0)
            case.launch()
    binding.h3gqa_sync_and_check(case.sh)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            case.launch()
            ends[i].record(stream)
    torch.cuda.synchronize(device)
    t1 = time.perf_counter()
    barrier(world)
    binding.h3gqa_sync_and_check(case.sh)
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], t0, t1


def measure_e2e(case, args, device, stream, world):
    """End to end: every step copies its inputs from pinned host memory, runs
    the kernel and reads o and lse back. Steps are pipelined the way a caller
    would run them: copies in, compute and copies out on three streams with
    two device buffer sets, so step i+1's upload and step i-1's download
    overlap step i's kernel. A head shard moves only its own heads' rows."""
    w = case.w
    T = w.total_tokens
    g = w.n_q_heads // w.n_kv_heads
    qh_rows = slice(case.kv_begin * g, (case.kv_begin + case.kv_count) * g)
    kv_rows = slice(case.kv_begin, case.kv_begin + case.kv_count)
    qh, kh, vh = case.x["q"][qh_rows].pin_memory(), case.x["k"][kv_rows].pin_memory(), \
        case.x["v"][kv_rows].pin_memory()

    def o_part(t):
        return t[:, qh_rows] if case.token_major else t[qh_rows]

    oh = torch.empty(o_part(case.o).shape, dtype=case.o.dtype, pin_memory=True)
    lh = torch.empty((qh.shape[0], T), dtype=torch.float32, pin_memory=True)
    sch = (torch.empty(o_part(case.o_scale).shape, dtype=torch.float32, pin_memory=True)
           if case.o_scale is not None else None)
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size() + \
        (sch.numel() * sch.element_size() if sch is not None else 0)
    bufs = [dict(q=case.q, k=case.k, v=case.v, o=case.o, lse=case.lse, sc=case.o_scale)]
    bufs.append(dict(q=torch.empty_like(case.q), k=torch.empty_like(case.k),
                     v=torch.empty_like(case.v), o=torch.empty_like(case.o),
                     lse=torch.empty_like(case.lse),
                     sc=torch.empty_like(case.o_scale) if case.o_scale is not None else None))
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    e2e_steps = max(4, min(args.steps, 20))
    n_windows = 3
    n_total = n_windows * e2e_steps + 2
    ev_in = [torch.cuda.Event() for _ in range(n_total)]
    ev_comp = [torch.cuda.Event() for _ in range(n_total)]
    ev_out = [torch.cuda.Event() for _ in range(n_total)]

    def e2e_step(i):
        b = bufs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])          # this buffer's inputs are free
            b["q"][qh_rows].copy_(qh, non_blocking=True)
            b["k"][kv_rows].copy_(kh, non_blocking=True)
            b["v"][kv_rows].copy_(vh, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])             # this buffer's outputs were read
        case.launch(b["q"], b["k"], b["v"], b["o"], b["lse"], case.options(b["sc"]))
        ev_comp[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[i])
            oh.copy_(o_part(b["o"]), non_blocking=True)
            lh.copy_(b["lse"][qh_rows], non_blocking=True)
            if sch is not None:
                sch.copy_(o_part(b["sc"]), non_blocking=True)
            ev_out[i].record(s_out)

    for i in range(2):
        e2e_step(i)
    # three timed windows of e2e_steps pipelined steps each (the pipeline
    # drains between windows); the median window is reported, so one stall
    # of the host does not stand for the whole measurement
    windows = []
    for wi in range(n_windows):
        torch.cuda.synchronize(device)
        barrier(world)
        te0 = time.perf_counter()
        for i in range(2 + wi * e2e_steps, 2 + (wi + 1) * e2e_steps):
            e2e_step(i)
        torch.cuda.synchronize(device)
        windows.append((time.perf_counter() - te0) * 1e3 / e2e_steps)
    binding.h3gqa_sync_and_check(case.sh)
    e2e_ms = float(np.median(windows))
    return max_over_ranks(e2e_ms, world, device), h2d, d2h, windows


def run_ours(args, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    binding.load()
    w = WORKLOADS[args.workload]
    stream = torch.cuda.Stream(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    case = Case(w, args, device, stream, shard_of(args, w, world, rank))
    sampler = make_sampler(local)
    sampler.start()
    time.sleep(0.05)
    times, t0, t1 = time_steps(case, args.steps, args.warmup, stream, flush, device, world)
    clocks = sampler.summary(t0, t1)
    ms = float(np.mean(times))
    ms_max = max_over_ranks(ms, world, device)

    extras = []
    if not args.no_extra and w.name == HEADLINE and world == 1:
        for name in EXTRA_WORKLOADS:
            ew = WORKLOADS[name]
            ec = Case(ew, args, device, stream, (0, ew.n_kv_heads))
            et, e0, e1 = time_steps(ec, max(3, min(args.steps, 20)), 3, stream, flush, device, 1)
            ems = float(np.mean(et))
            extras.append((ew, ec, et, ems, sampler.summary(e0, e1)))
            del ec
    sampler.stop()

    e2e_ms, h2d, d2h, e2e_windows = measure_e2e(case, args, device, stream, world)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    if args.shard == "heads":
        value = w.metric_flops() / (ms_max * 1e-3) / 1e12
        e2e_value = w.metric_flops() / (e2e_ms * 1e-3) / 1e12
        scaling = "strong"
    else:
        value = whole_job_value(w.metric_flops(), world, ms_max)
        e2e_value = whole_job_value(w.metric_flops(), world, e2e_ms)
        scaling = "weak"
    # rank 0's own launch: the causal FLOPs of its heads over its mean time
    achieved = case.plan.causal_flops * case.frac_heads / (ms * 1e-3) / 1e12
    plain = args.epilogue == "bf16_head" and not args.prologue and case.frac_heads == 1
    line = {
        "metric": metric_name(w, args.epilogue, args.prologue), "value": value, "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": scaling, "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 q/k/v; no dataset)",
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "config": config_of(w, args, world),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak,
                     "traffic": kernel_traffic(w.name) if plain else None,
                     "traffic_unit": "bytes per launch (ncu dram read+write)",
                     "peak_source": "%s bf16_tflops (burst)" % peak_src,
                     "kernel": "h3gqa::causal_gqa_fwd_kernel",
                     "work": "4*D FLOPs per visible (query, key, head) pair per launch"},
        "e2e": {"value": e2e_value, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step_windows": [round(x, 4) for x in e2e_windows],
                "api": "h3gqa_attention_fwd via the Python binding; pinned host buffers; "
                       "upload / compute / download on three streams, two device buffer sets; "
                       "median of three timed windows"},
        "gpu_launches": args.steps * case.launches_per_step if case.kv_count else 0,
        "clocks": clocks,
        "kernel_ms": {"mean": ms, "min": float(np.min(times)), "max": float(np.max(times))},
    }
    if args.shard == "heads":
        line["shard"] = {"kind": "contiguous KV-head ranges, one launch per rank, no collective",
                         "rank0_kv_heads": [case.kv_begin, case.kv_count]}
    if extras:
        line["extra_workloads"] = []
        for ew, ec, et, ems, eclk in extras:
            ach = ec.plan.causal_flops / (ems * 1e-3) / 1e12
            line["extra_workloads"].append({
                "workload": ew.name, "seqlens": list(ew.seqlens),
                "metric": metric_name(ew, args.epilogue, args.prologue),
                "value": ew.metric_flops() / (ems * 1e-3) / 1e12, "unit": UNIT,
                "frac": ach / peak, "achieved_causal_exact": ach,
                "steps": len(et), "warmup": 3,
                "kernel_ms": {"mean": ems, "min": float(np.min(et)), "max": float(np.max(et))},
                "traffic": kernel_traffic(ew.name) if plain else None,
                "gpu_launches": len(et) * ec.launches_per_step, "clocks": eclk})
    if not args.no_cpu_baseline:
        r, desc, cores, dt = oracle_sample_rate(case.x, w, args.cpu_seconds, seed=w.seed)
        line["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc + "; %.1f s timed" % dt}
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
    ap.add_argument("--shard", choices=["replicas", "heads"], default="replicas",
                    help="N>1: independent replicas (weak) or one workload split by KV heads "
                         "(strong)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the extra long workloads measured after the headline")
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
