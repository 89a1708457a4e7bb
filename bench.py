"""Benchmark of libgqa on GB300: one JSON line on rank 0.

A step is one pass of the whole hot path over one batch of synthetic input,
on the two largest single-GPU configurations:
  1. gqa_decode on decode_b8_cap131072 (B=8, 32/8 heads, D=128, capacity =
     lengths = 131072, q_scale 0.5, seed 2: 4.29 GB of K/V read) -- split
     kernel + LSE merge; and
  2. nvfp4_paged_ctx_attn on ctx_b2_q4096_kv65536 (batch 2, 4096 queries
     ending a 65536-key sequence, NVFP4 HND pages through a shuffled block
     table, seed 4: 8.52e12 causal FLOP).
The headline `value` is the decode's HBM GB/s (K/V bytes read / decode
time); the context attention's causal TFLOP/s is reported under
"ctx_attn".  `roofline` is that of the step's dominant kernel (the context
attention); every kernel's roofline is in "configs".

Then each of the five configurations is timed on its own ("configs"): the
median of >= 50 CUDA-event-timed calls, L2 flushed (a 512 MB read) before
each call, with its roofline and a cpu_baseline (the fp64 oracle on the host
cores, on a bounded sample).  decode_b2_cap256 is launch-latency bound and
is also given in microseconds per call.

Timing: CUDA events on the launching stream around each call, W untimed
warm-up steps, K timed steps bracketed by a barrier and a synchronize,
median per rank, max over ranks.  Inputs are generated on the GPU (CUDA
generator, the recipe of gqa_workloads) and resident in HBM before timing.

--impl reference times the fp64 CPU oracle instead (the reference arm): each
step is a bounded sample of the headline workload on the host cores.
--workload NAME benchmarks a single named workload (see gqa_workloads).
--study times every instantiated ring-depth schedule (gqa_set_schedule)
against the production depths on the context and decode workloads,
interleaved, L2 flushed before each call, and checks that every schedule's
output is byte-identical to the production one.

Multi-GPU: `--gpus N` under torchrun runs N independent replicas (the path
has no exchange step); value = bytes all ranks processed / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GQA decode HBM GB/s (% of GB300 peak); NVFP4 ctx attn TFLOP/s (% FP8 peak)"
DECODE_WL = "decode_b8_cap131072"
CTX_WL = "ctx_b2_q4096_kv65536"
ALL_CONFIGS = ["decode_b2_cap256", "decode_b64_cap8192", "decode_b8_cap131072",
               "ctx_b4_q2048_kv2048", "ctx_b2_q4096_kv65536"]
# Latency-bound rows of the results table of "GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단
# packed K/V ring" (GB300, its kernel after the change), read as batch x q_len x kv_len: context for the
# workloads of the same shape, not a target of this metric.
PAGE_ROWS_US = {"ctx_b2_q1_kv4096": ("2 x 1 x 4096", 44.5), "ctx_b1_q32_kv32768": ("1 x 32 x 32768", 329.8)}
# Decode-shaped context workloads, reported against HBM (their page bytes) rather than the tensor peak.
MEMORY_BOUND_CTX = {"ctx_b64_q1_kv8192", "ctx_b64_q8_kv8192"}
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0
FP8_OVER_BF16 = 2.0        # nominal dense ratio (4.5 / 2.25 PFLOP/s)
HBM_NOMINAL_GBS = 7900.0   # GB300 HBM3e, nominal: a read-only stream may exceed the measured copy figure
# Committed ncu summaries: DRAM bytes per launch, valid while the digest of the sources the kernel is built
# from (its header plus the shared ones) matches.
_DEC_SRC = ["decode.cu", "common.cuh", "kernels.h"]
_CTX_COMMON = ["ctx_kernel.cuh", "ctx_nvfp4.cu", "common.cuh", "nvfp4.cuh", "tcgen05.cuh", "kernels.h"]
_CTX_SRC = _CTX_COMMON                                  # one CTA per unit (and its split-KV form)
_CTX_PERSISTENT_SRC = _CTX_COMMON + ["ctx_persistent.cuh"]
_CTX_DECODE_SRC = _CTX_COMMON + ["ctx_decode.cuh"]
PROFILES = {
    "decode_b64_cap8192": ("decode_split_kernel_decode_b64_cap8192.md", _DEC_SRC),
    "decode_b8_cap131072": ("decode_split_kernel_decode_b8_cap131072.md", _DEC_SRC),
    "ctx_b4_q2048_kv2048": ("ctx_nvfp4_persistent_kernel_ctx_b4_q2048_kv2048.md", _CTX_PERSISTENT_SRC),
    "ctx_b2_q4096_kv65536": ("ctx_nvfp4_kernel_ctx_b2_q4096_kv65536.md", _CTX_SRC),
    "ctx_b64_q1_kv8192": ("ctx_nvfp4_decode_kernel_ctx_b64_q1_kv8192.md", _CTX_DECODE_SRC),
}


# ------------------------------------------------------------- peaks/files --

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM, "bf16_tflops": FALLBACK_BF16, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gqa_attention_kv_split_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """(DRAM bytes per launch, where from) from a committed ncu summary of this
    workload, or (None, why) when there is none or the kernel source changed
    since the counters were taken.  Not a measurement of this run."""
    if workload not in PROFILES:
        return None, "no ncu capture of this workload"
    md, files = PROFILES[workload]
    try:
        txt = open(os.path.join(ROOT, "profiles", md)).read()
    except OSError:
        return None, f"profiles/{md} missing"
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not s:
        return None, f"profiles/{md} has no traffic figure"
    if s.group(1) != source_digest(files):
        return None, f"kernel changed since profiles/{md} was captured"
    return float(m.group(1)), f"ncu capture in profiles/{md} (dram__bytes_read+write), not this run"


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the process runs; summaries of
    named windows."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None
        self.marks = {}

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self, which):
        self.marks[which] = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self, start="start", stop="stop"):
        """Samples inside [start, stop]; if that window was shorter than the
        sampling period, the samples of the preceding second (the same kernels
        warming up) are added and the window says so."""
        t0, t1 = self.marks.get(start), self.marks.get(stop)
        window = "timed region"
        lines = [l for (t, l) in self.lines if t0 is not None and t0 <= t <= t1 + 0.05]
        if len(lines) < 3 and t0 is not None:
            lines = [l for (t, l) in self.lines if t0 - 1.0 <= t <= t1 + 0.05]
            window = "timed region and the preceding 1 s of warm-up"
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm), "window": window}


# -------------------------------------------------------------- distributed --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, backend_device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=backend_device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- GPU arm --

def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _quantiles(ms):
    s = sorted(ms)
    q = lambda f: s[min(len(s) - 1, int(round(f * (len(s) - 1))))]
    return {"median": statistics.median(s), "p10": q(0.1), "p90": q(0.9), "min": s[0]}


class L2Flush:
    """Evicts L2 by reading a 512 MB buffer (4x the 129 MB L2).  A read leaves
    only clean lines behind, so the timed call pays no write-back of the
    flush's own data (a write flush would leave ~129 MB of dirty lines for
    the next kernel to write back)."""

    def __init__(self, torch, dev):
        self.buf = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.sum()


def time_reps(torch, stream, call, flush, min_reps=50, min_seconds=0.4, warmup=10):
    """Median etc. of `call` over >= min_reps CUDA-event-timed calls (and at
    least ~min_seconds of them), each preceded by an L2 flush."""
    for _ in range(warmup):
        flush()
        call()
    torch.cuda.synchronize()
    a, b = _events(torch, 2)
    a.record(stream)
    call()
    b.record(stream)
    torch.cuda.synchronize()
    est = max(a.elapsed_time(b), 1e-3) + 0.08  # + the flush
    reps = max(min_reps, min(20000, int(min_seconds * 1e3 / est)))
    evs = [_events(torch, 2) for _ in range(reps)]
    for e in evs:
        flush()
        e[0].record(stream)
        call()
        e[1].record(stream)
    torch.cuda.synchronize()
    ms = [e[0].elapsed_time(e[1]) for e in evs]
    out = _quantiles(ms)
    out["reps"] = reps
    return out


class Workload:
    """One named workload resident on the GPU, with its call and figures."""

    def __init__(self, gqa, W, name, dev):
        self.name = name
        self.gqa = gqa
        self.kind = "decode" if name.startswith("decode") else "ctx"
        if self.kind == "decode":
            self.x = W.decode_workload(name, device=dev)
            self.paged = isinstance(self.x, W.PagedDecodeInputs)
            self.out = torch_mod().empty_like(self.x.q)
            plan = gqa.gqa_decode_plan(self.x.batch, self.x.capacity)
            self.plan = plan
            self.launches = plan["num_launches"]
            self.work = self.x.kv_bytes_read()  # bytes
        else:
            self.x = W.ctx_workload(name, device=dev)
            self.paged = False
            self.args = (self.x.q_fp8, self.x.k_fp4, self.x.k_sf, self.x.v_fp4, self.x.v_sf, self.x.block_table,
                         self.x.qo_indptr, self.x.kv_lens)
            self.out = torch_mod().empty_like(self.x.q_fp8)
            self.plan = gqa.gqa_ctx_plan(self.x.block_table.shape[0], self.x.q_fp8.shape[0],
                                         self.x.block_table.shape[1])
            self.launches = self.plan["num_launches"]
            self.work = self.x.causal_flops()  # FLOPs

    def call(self):
        x = self.x
        if self.kind == "decode":
            if self.paged:
                self.gqa.gqa_decode_paged(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, out=self.out,
                                          q_scale=x.q_scale)
            else:
                self.gqa.gqa_decode(x.q, x.kv, x.seq_lens, out=self.out, q_scale=x.q_scale)
        else:
            self.gqa.nvfp4_paged_ctx_attn(*self.args, q_scale=x.q_scale, out_scale=x.out_scale, out=self.out)

    @property
    def kernel(self):
        """The attention kernel(s) one call launches, as the launch plan chooses them."""
        if self.kind == "decode":
            return "decode_split_kernel" + (" + decode_merge_kernel" if self.launches > 1 else "")
        if self.plan.get("decode_shaped"):
            return "ctx_nvfp4_decode_kernel + ctx_merge_kernel"
        if self.plan.get("persistent") and self.launches == 1:
            return "ctx_nvfp4_persistent_kernel"
        return "ctx_nvfp4_kernel" + (" + ctx_merge_kernel" if self.launches > 1 else "")

    def rate(self, ms):
        """GB/s (decode) or TFLOP/s (ctx) for one call of `ms` milliseconds."""
        return self.work / (ms * 1e-3) / (1e9 if self.kind == "decode" else 1e12)

    @property
    def unit(self):
        return "GB/s" if self.kind == "decode" else "TFLOP/s"

    def roofline(self, ms, peaks):
        traffic, src = profiled_traffic(self.name)
        a = self.rate(ms)
        if self.kind == "decode":
            return {"bound": "hbm", "achieved": round(a, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(a / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                    "peak_nominal": HBM_NOMINAL_GBS, "frac_nominal": round(a / HBM_NOMINAL_GBS, 4),
                    "traffic": traffic, "traffic_source": src,
                    "algorithmic": f"{self.work} B = sum of lengths x 4096 B (K+V, 8 heads x 128 x fp16)",
                    "kernel": self.kernel + " inside the same events"}
        fp8 = peaks["bf16_tflops"] * FP8_OVER_BF16
        if self.name in MEMORY_BOUND_CTX:
            # decode-shaped: a few query rows per KV head, so the page bytes, not the tensor work, bound it
            gbs = self.x.page_bytes_read() / (ms * 1e-3) / 1e9
            return {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_nominal": HBM_NOMINAL_GBS,
                    "frac_nominal": round(gbs / HBM_NOMINAL_GBS, 4), "traffic": traffic, "traffic_source": src,
                    "algorithmic": f"{self.x.page_bytes_read()} B = every used page's packed codes and scales, "
                                   "K and V, once", "tflops": round(a, 2),
                    "kernel": self.kernel}
        return {"bound": "tensor", "achieved": round(a, 2), "peak": round(fp8, 1), "unit": "TFLOP/s",
                "frac": round(a / fp8, 4),
                "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16} (nominal dense FP8:bf16)",
                "traffic": traffic, "traffic_source": src,
                "algorithmic": f"{self.work} FLOP = 4 x 128 x 32 heads x visible (query, key) pairs",
                "kernel": self.kernel}

    def config(self):
        x = self.x
        if self.kind == "decode":
            return {"batch": x.batch, "capacity": x.capacity, "q_scale": x.q_scale,
                    "kv_layout": "64-token HND pages, shuffled block table" if self.paged
                    else "stacked [B,2,8,cap,128]", "kv_bytes_read": self.work, "plan": self.plan}
        return {"batch": x.batch, "total_q": x.total_q, "num_pages": int(x.k_fp4.shape[0]),
                "max_kv": int(x.kv_lens.max().item()), "q_scale": x.q_scale, "out_scale": x.out_scale,
                "causal_flops": self.work, "plan": self.plan}


_torch = None


def torch_mod():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def e2e_decode(torch, gqa, wl, stream, steps):
    """gqa_decode through the C ABI with pinned host buffers: the H2D staging
    of the inputs and the D2H copy of the output inside the timed region."""
    x = wl.x
    hq = torch.empty(x.q.shape, dtype=x.q.dtype, pin_memory=True).copy_(x.q)
    hl = torch.empty(x.seq_lens.shape, dtype=torch.int32, pin_memory=True).copy_(x.seq_lens)
    hkv = torch.empty(x.kv.shape, dtype=x.kv.dtype, pin_memory=True).copy_(x.kv)
    hout = torch.empty(hq.shape, dtype=hq.dtype, pin_memory=True)
    for _ in range(2):
        gqa.gqa_decode(hq, hkv, hl, out=hout, q_scale=x.q_scale)
    ts = []
    for _ in range(steps):
        a, b = _events(torch, 2)
        a.record(stream)
        gqa.gqa_decode(hq, hkv, hl, out=hout, q_scale=x.q_scale)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    lens = hl.clamp(0, x.capacity).to(torch.int64)
    h2d = hq.numel() * 2 + int(lens.sum()) * 16 * 256 + hl.numel() * 4  # each sequence's first len tokens
    d2h = hout.numel() * 2
    ms = statistics.median(ts)
    # the link on its own: one plain pinned H2D copy of the same K/V bytes (cudaMemcpyAsync)
    dst = torch.empty_like(x.kv)
    cts = []
    for _ in range(3):
        a, b = _events(torch, 2)
        a.record(stream)
        dst.copy_(hkv, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        cts.append(a.elapsed_time(b))
    kv_bytes = hkv.numel() * 2
    copy_gbs = kv_bytes / (min(cts) * 1e-3) / 1e9
    del dst, hkv
    return {"value": round(wl.work / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4), "steps": steps,
            "path": "gqa_decode with pinned host buffers (library stages the bytes the kernels read)",
            "h2d_copy_gbs": round(copy_gbs, 1),
            "h2d_copy": f"one pinned cudaMemcpyAsync of the whole {kv_bytes} B K/V tensor, best of 3: "
                        "the link's rate, for context"}


def e2e_ctx(torch, gqa, wl, stream, steps):
    """nvfp4_paged_ctx_attn with pinned host buffers (all inputs staged, output copied back)."""
    x = wl.x
    host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in wl.args]
    hout = torch.empty(x.q_fp8.shape, dtype=torch.uint8, pin_memory=True)
    for _ in range(2):
        gqa.nvfp4_paged_ctx_attn(*host, q_scale=x.q_scale, out_scale=x.out_scale, out=hout)
    ts = []
    for _ in range(steps):
        a, b = _events(torch, 2)
        a.record(stream)
        gqa.nvfp4_paged_ctx_attn(*host, q_scale=x.q_scale, out_scale=x.out_scale, out=hout)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    return {"value": round(wl.work / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host),
            "d2h_bytes_per_step": hout.numel(), "ms_per_step": round(ms, 4), "steps": steps,
            "path": "nvfp4_paged_ctx_attn with pinned host buffers"}


def run_gpu(args):
    import torch

    import gqa_attention_kv_split_gb300 as gqa
    import gqa_workloads as W

    world, rank, local = dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    gqa.lib()  # fails loudly if the library is missing

    if args.workload:
        step_names = [args.workload]
        config_names = [args.workload] if not args.no_configs else []
    else:
        step_names = [DECODE_WL, CTX_WL]
        config_names = [] if args.no_configs else list(ALL_CONFIGS)
    names = list(dict.fromkeys(step_names + config_names))
    wls = {n: Workload(gqa, W, n, dev) for n in names}
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)
    step_wls = [wls[n] for n in step_names]

    def step(evs):
        for i, wl in enumerate(step_wls):
            flush()
            evs[2 * i].record(stream)
            wl.call()
            evs[2 * i + 1].record(stream)

    n_ev = 2 * len(step_wls)
    all_evs = [_events(torch, n_ev) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let the sampler start before the GPU is loaded
        for _ in range(args.warmup):
            step(_events(torch, n_ev))
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        clk.mark("start")
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(all_evs[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        clk.mark("stop")
        barrier()
        # each configuration on its own
        clk.mark("cfg_start")
        cfg_times = {n: time_reps(torch, stream, wls[n].call, flush) for n in config_names}
        clk.mark("cfg_stop")
    per_wl_ms = {wl.name: [e[2 * i].elapsed_time(e[2 * i + 1]) for e in all_evs] for i, wl in enumerate(step_wls)}
    med = {n: max_over_ranks(statistics.median(v), dev) for n, v in per_wl_ms.items()}
    step_ms = [sum(e[2 * i].elapsed_time(e[2 * i + 1]) for i in range(len(step_wls))) for e in all_evs]
    step_med = max_over_ranks(statistics.median(step_ms), dev)

    e2e = ctx_e2e = None
    head = step_wls[0]
    if rank == 0 and head.kind == "decode" and not head.paged:
        e2e = e2e_decode(torch, gqa, head, stream, max(3, min(args.steps, 10)))
    ctx_step = next((w for w in step_wls if w.kind == "ctx"), None)
    if rank == 0 and ctx_step is not None:
        ctx_e2e = e2e_ctx(torch, gqa, ctx_step, stream, max(3, min(args.steps, 10)))

    if rank != 0:
        return
    clocks = clk.summary("start", "stop")
    line = {"metric": METRIC}
    hv = head.rate(med[head.name]) * world
    line.update({
        "value": round(hv, 2), "unit": head.unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_med, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if head.kind == "decode" else "e4m3", "data": "synthetic (CUDA generator, seeded)",
        "config": {"workload": head.name, **head.config(),
                   "step": " + ".join(w.name for w in step_wls),
                   "l2": "L2 flushed (512 MB read) before every timed call; decode inputs also exceed L2",
                   "parallelism": f"replicas{world}"},
    })
    # roofline of the step's dominant kernel (by median device time)
    dom = max(step_wls, key=lambda w: med[w.name])
    line["roofline"] = {**dom.roofline(med[dom.name], peaks), "workload": dom.name,
                        "share_of_step": round(med[dom.name] / step_med, 4)}
    if head.kind == "decode":
        line["decode_roofline"] = head.roofline(med[head.name], peaks)
    if ctx_step is not None:
        ctx_obj = {"value": round(ctx_step.rate(med[ctx_step.name]) * world, 2), "unit": "TFLOP/s",
                   "ms": round(med[ctx_step.name], 4), "workload": ctx_step.name, "dtype": "e4m3",
                   **ctx_step.config(), "roofline": ctx_step.roofline(med[ctx_step.name], peaks), "e2e": ctx_e2e}
        if ctx_step.name in PAGE_ROWS_US:
            label, us = PAGE_ROWS_US[ctx_step.name]
            ctx_obj["page_row"] = {"label": label, "us": us, "ours_us": round(med[ctx_step.name] * 1e3, 2)}
        line["ctx_attn"] = ctx_obj
    line["e2e"] = e2e if e2e is not None else (ctx_e2e if head.kind == "ctx" else None)
    line["gpu_launches"] = args.steps * sum(w.launches for w in step_wls)
    line["clocks"] = clocks
    line["wall_s_timed_region"] = round(wall, 4)
    # per-configuration entries
    configs = []
    cpu_ok = args.cpu_baseline and world == 1
    for n in config_names:
        wl, t = wls[n], cfg_times[n]
        entry = {"workload": n, "value": round(wl.rate(t["median"]), 2),
                 "unit": wl.unit, "ms_median": round(t["median"], 5), "ms_p10": round(t["p10"], 5),
                 "ms_p90": round(t["p90"], 5), "reps": t["reps"], "launches_per_call": wl.launches,
                 **wl.config(), "roofline": wl.roofline(t["median"], peaks)}
        if n == "decode_b2_cap256":
            entry["us_per_call"] = round(t["median"] * 1e3, 2)
            entry["note"] = ("launch-latency bound: 0.82 MB of K/V per call; the time is launch and prologue, "
                             "not bandwidth")
        if n in PAGE_ROWS_US:
            label, us = PAGE_ROWS_US[n]
            entry["page_row"] = {"label": label, "us": us, "ours_us": round(t["median"] * 1e3, 2)}
        if cpu_ok:
            entry["cpu_baseline"] = (oracle_decode_sample(wl.x, budget_s=args.cpu_budget) if wl.kind == "decode"
                                     else oracle_ctx_sample(wl.x, budget_s=args.cpu_budget))
        configs.append(entry)
    line["configs"] = configs
    line["clocks_configs"] = clk.summary("cfg_start", "cfg_stop") if config_names else None
    if cpu_ok:
        hb = next((c.get("cpu_baseline") for c in configs if c["workload"] == head.name), None)
        line["cpu_baseline"] = hb or (oracle_decode_sample(head.x, budget_s=args.cpu_budget)
                                      if head.kind == "decode" else oracle_ctx_sample(head.x, budget_s=args.cpu_budget))
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- ring-depth study --

def run_study(args):
    """One JSON line: per workload and schedule, the median of interleaved
    event-timed calls and whether the output is byte-identical to the
    production depths'."""
    import torch

    import gqa_attention_kv_split_gb300 as gqa
    import gqa_workloads as W
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    gqa.lib()
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)
    names = [args.workload] if args.workload else ["ctx_b2_q4096_kv65536", "ctx_b4_q2048_kv2048", "ctx_b64_q1_kv8192",
                                                   "decode_b8_cap131072", "decode_b64_cap8192"]
    rows = []
    # every ring depth on the same grid: the study instances run one CTA per unit, so the production depths do too
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PER_UNIT)
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        clk.mark("start")
        for name in names:
            wl = Workload(gqa, W, name, dev)
            if wl.kind == "ctx":
                scheds = [(st, sl, 0) for st, sl in gqa.CTX_SCHEDULES]
            else:
                scheds = [(0, 0, d) for d in gqa.DECODE_SCHEDULES]
            outs, evs = {}, {sc: [] for sc in scheds}
            for sc in scheds:  # warm-up and the output of every schedule
                gqa.gqa_set_schedule(*sc)
                for _ in range(3):
                    wl.call()
                torch.cuda.synchronize()
                outs[sc] = wl.out.clone()
            reps = 20 if name == "ctx_b2_q4096_kv65536" else 100
            for _ in range(reps):
                for sc in scheds:
                    gqa.gqa_set_schedule(*sc)
                    flush()
                    a, b = _events(torch, 2)
                    a.record(stream)
                    wl.call()
                    b.record(stream)
                    evs[sc].append((a, b))
            torch.cuda.synchronize()
            gqa.gqa_set_schedule(0, 0, 0)
            base = None
            for sc in scheds:
                ms = statistics.median(a.elapsed_time(b) for a, b in evs[sc])
                base = base or ms
                rows.append({"workload": name, "ctx_packed_stages": sc[0] or None, "ctx_kv_slots": sc[1] or None,
                             "decode_stages": sc[2] or None, "ms_median": round(ms, 5),
                             "value": round(wl.rate(ms), 2), "unit": wl.unit, "speed_vs_production": round(base / ms, 4),
                             "byte_identical": bool(torch.equal(outs[sc], outs[scheds[0]])), "reps": reps})
            del wl
            torch.cuda.empty_cache()
        clk.mark("stop")
    gqa.gqa_set_ctx_grid(gqa.CTX_GRID_PLANNED)
    print(json.dumps({"study": "ring depths (gqa_set_schedule), context calls on the one-CTA-per-unit grid",
                      "rows": rows, "clocks": clk.summary()}), flush=True)


# ---------------------------------------------------------- oracle (CPU) --

def _decode_sample(dx, n_seq):
    import gqa_workloads as W
    idx = list(range(n_seq))
    if isinstance(dx, W.PagedDecodeInputs):  # the pages stay whole; the table rows are sampled
        return W.PagedDecodeInputs(dx.q[idx].cpu(), dx.k_pages.cpu(), dx.v_pages.cpu(), dx.block_table[idx].cpu(),
                                   dx.seq_lens[idx].cpu(), dx.q_scale)
    return W.DecodeInputs(dx.q[idx].cpu(), dx.kv[idx].cpu(), dx.seq_lens[idx].cpu(), dx.q_scale)


def _oracle_decode(sub, threads):
    import gqa_workloads as W
    import oracle
    if isinstance(sub, W.PagedDecodeInputs):
        return oracle.gqa_decode_paged(sub.q.numpy(), sub.k_pages.numpy(), sub.v_pages.numpy(),
                                       sub.block_table.numpy(), sub.seq_lens.numpy(), sub.q_scale, threads=threads)
    return oracle.gqa_decode(sub.q.numpy(), sub.kv.numpy(), sub.seq_lens.numpy(), sub.q_scale, threads=threads)


def oracle_decode_sample(dx, budget_s=10.0):
    """Time the oracle on the first n sequences (all 32 heads), n grown until
    the sample takes about `budget_s` / 3 seconds or covers the workload."""
    import oracle
    threads = oracle.default_threads()
    n, took, sub = 1, 0.0, None
    while True:
        sub = _decode_sample(dx, n)
        t0 = time.perf_counter()
        _oracle_decode(sub, threads)
        took = time.perf_counter() - t0
        if n >= dx.batch or took >= budget_s / 3:
            break
        n = min(dx.batch, max(n * 2, int(n * budget_s / 3 / max(took, 1e-3))))
    gbs = sub.kv_bytes_read() / took / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {dx.batch} sequences, all 32 heads ({sub.kv_bytes_read()} KV bytes), "
                      f"{took:.2f} s"}


def oracle_ctx_sample(cx, budget_s=10.0, rows=None):
    """Time the oracle on random (row, head) items; each call also dequantises
    every page the sequences use (the oracle as it stands)."""
    import numpy as np

    import oracle
    threads = oracle.default_threads()
    total = cx.total_q * 32
    rng = np.random.default_rng(0)
    n = rows or 256
    host = [t.cpu().numpy() for t in (cx.q_fp8, cx.k_fp4, cx.k_sf, cx.v_fp4, cx.v_sf, cx.block_table,
                                      cx.qo_indptr, cx.kv_lens)]
    while True:
        pick = rng.choice(total, size=min(n, total), replace=False)
        items = np.stack([pick // 32, pick % 32], axis=1)
        t0 = time.perf_counter()
        oracle.nvfp4_paged_ctx_attn(host[0], cx.q_scale, *host[1:], cx.out_scale, items=items, threads=threads)
        took = time.perf_counter() - t0
        if rows or n >= total or took >= budget_s / 3:
            break
        n = min(total, max(n * 2, int(n * budget_s / 3 / max(took, 1e-3))))
    # FLOPs of the sampled (row, head) items
    qi = host[6].tolist()
    kl = host[7].tolist()
    pairs = 0
    for r in (items[:, 0]).tolist():
        b = max(i for i in range(len(kl)) if qi[i] <= r)
        ql = qi[b + 1] - qi[b]
        pairs += max(0, min(kl[b], kl[b] - ql + (r - qi[b]) + 1))
    flops = 4 * 128 * pairs
    return {"value": round(flops / took / 1e12, 8), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(items)} random (row, head) items of {total} (plus the dequantisation of every page "
                      f"the sequences use), {took:.2f} s"}


def run_reference(args):
    """The reference arm: the fp64 CPU oracle as it stands, on host cores,
    on the headline workload (bounded samples per step)."""
    import torch

    import gqa_workloads as W
    world, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.workload or DECODE_WL
    import oracle
    threads = oracle.default_threads()
    if name.startswith("ctx"):
        cx = W.ctx_workload(name, device="cuda" if torch.cuda.is_available() else "cpu")
        samples = []
        for i in range(args.warmup + args.steps):
            r = oracle_ctx_sample(cx, rows=args.ref_rows or 64)
            if i >= args.warmup:
                samples.append(r)
        value = statistics.fmean(s["value"] for s in samples)
        unit, dtype = "TFLOP/s", "f64"
        cfg = {"workload": name}
        sample = samples[0]["sample"]
    else:
        dx = W.decode_workload(name, device="cuda" if torch.cuda.is_available() else "cpu")
        per_step = max(1, args.ref_seqs or 1)
        times, byts = [], []
        for i in range(args.warmup + args.steps):
            lo = (i * per_step) % dx.batch
            idx = [(lo + k) % dx.batch for k in range(per_step)]
            if isinstance(dx, W.PagedDecodeInputs):
                sub = W.PagedDecodeInputs(dx.q[idx].cpu(), dx.k_pages.cpu(), dx.v_pages.cpu(),
                                          dx.block_table[idx].cpu(), dx.seq_lens[idx].cpu(), dx.q_scale)
            else:
                sub = W.DecodeInputs(dx.q[idx].cpu(), dx.kv[idx].cpu(), dx.seq_lens[idx].cpu(), dx.q_scale)
            t0 = time.perf_counter()
            _oracle_decode(sub, threads)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                times.append(dt)
                byts.append(sub.kv_bytes_read())
        value = sum(byts) / sum(times) / 1e9
        unit, dtype = "GB/s", "f64"
        cfg = {"workload": name, "batch": dx.batch, "capacity": dx.capacity}
        sample = f"{per_step} sequence(s) (all 32 heads) per step, rotating through the batch"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic (CUDA generator, seeded)", "config": cfg,
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "kind": "oracle", "cores": threads,
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_peaks(seconds_sustained: float = 4.0) -> dict:
    """Context figures for the rooflines, on this GPU: a read-only HBM stream
    (sum of a 4 GiB tensor), dense GEMMs 8192^3 in bf16 (torch.matmul) and in
    FP8 E4M3 with bf16 output (torch._scaled_mm): best of 10, and the FP8 GEMM
    again in a loop of `seconds_sustained` seconds.  The rooflines bench.py
    reports keep the measured copy bandwidth and bf16 x 2 as their peaks."""
    import torch
    dev = torch.device("cuda:0")
    out = {}

    def best_ms(fn, reps=10):
        ts = []
        for _ in range(reps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); fn(); b.record(); torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return min(ts[2:])

    x = torch.ones(2 * 1024 ** 3, dtype=torch.bfloat16, device=dev)  # 4 GiB
    ms = best_ms(lambda: x.sum())
    out["hbm_read_gbs"] = round(x.numel() * 2 / (ms * 1e-3) / 1e9, 1)
    del x
    n = 8192
    a = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    b = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    ms = best_ms(lambda: torch.matmul(a, b))
    out["bf16_tflops"] = round(2 * n ** 3 / (ms * 1e-3) / 1e12, 1)
    try:
        a8 = a.to(torch.float8_e4m3fn)
        b8 = b.to(torch.float8_e4m3fn).t().contiguous().t()  # column-major second operand
        one = torch.ones((), device=dev, dtype=torch.float32)
        f8 = lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        ms = best_ms(f8)
        out["fp8_tflops"] = round(2 * n ** 3 / (ms * 1e-3) / 1e12, 1)
        cnt, t0 = 0, time.perf_counter()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        while time.perf_counter() - t0 < seconds_sustained:
            for _ in range(50):
                f8()
            cnt += 50
            torch.cuda.synchronize()
        s1.record(); torch.cuda.synchronize()
        out["fp8_tflops_sustained"] = round(2 * n ** 3 * cnt / (s0.elapsed_time(s1) * 1e-3) / 1e12, 1)
    except Exception as e:  # noqa: BLE001 -- report why, keep the other figures
        out["fp8_error"] = f"{type(e).__name__}: {e}"[:200]
    out["device"] = torch.cuda.get_device_name(dev)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="a single named workload from gqa_workloads")
    ap.add_argument("--no-configs", dest="no_configs", action="store_true",
                    help="skip the per-configuration pass (timed step only)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=6.0, help="seconds of oracle time per configuration")
    ap.add_argument("--ref-seqs", type=int, default=0, help="reference arm: sequences per step (decode)")
    ap.add_argument("--ref-rows", type=int, default=0, help="reference arm: (row, head) items per step (ctx)")
    ap.add_argument("--study", action="store_true",
                    help="time every instantiated ring-depth schedule against the production depths and exit")
    ap.add_argument("--peaks", action="store_true",
                    help="measure context peaks (read-only HBM stream, bf16 and FP8 GEMMs) and exit")
    args = ap.parse_args(argv)
    if args.peaks:
        with ClockSampler(0) as clk:
            time.sleep(0.3)
            clk.mark("start")
            res = measure_peaks()
            clk.mark("stop")
        res["clocks"] = clk.summary()
        print(json.dumps(res))
        return
    if args.study:
        run_study(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        print("note: warm-up raised to the minimum of 3 steps", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
