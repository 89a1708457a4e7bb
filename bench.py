"""Benchmark of libgqa on GB300: one JSON line on rank 0.

A step is one pass of the whole hot path over one batch of synthetic input:
  1. gqa_decode on decode_b64_cap8192 (B=64, 32/8 heads, D=128, capacity 8192,
     lengths U{1..8192}, seed 1) -- split kernel + LSE merge; and
  2. nvfp4_paged_ctx_attn on ctx_b4_q2048_kv2048 (batch 4, q_len = kv_len =
     2048, NVFP4 HND pages through a shuffled block table, seed 3).
The headline metric is decode HBM GB/s (KV bytes read / decode time); the
context attention's causal TFLOP/s is reported beside it under "ctx_attn".

Timing: CUDA events on the launching stream around each call, W untimed
warm-up steps, K timed steps bracketed by a barrier and a synchronize, max
over ranks.  The decode reads 1.08 GB per step (larger than the 129 MB L2);
before each context call a 512 MB buffer is written to flush L2.

--impl reference times the fp64 CPU oracle instead (the reference arm):
each step is a bounded sample of the same workloads on the host cores.
--workload NAME benchmarks a single named workload (see gqa_workloads).

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
DECODE_WL = "decode_b64_cap8192"
CTX_WL = "ctx_b4_q2048_kv2048"
# Latency-bound rows of the results table of "GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단
# packed K/V ring" (GB300, its kernel after the change), read as batch x q_len x kv_len: context for the
# workloads of the same shape, not a target of this metric.
PAGE_ROWS_US = {"ctx_b2_q1_kv4096": ("2 x 1 x 4096", 44.5), "ctx_b1_q32_kv32768": ("1 x 32 x 32768", 329.8)}
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)


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


def profiled_traffic(profile_md: str, files):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", profile_md)
    try:
        txt = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not s or s.group(1) != source_digest(files):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

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
        setattr(self, which, time.perf_counter())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self):
        """Samples inside the timed region; if that region was shorter than
        the sampling period, the samples of the preceding second of warm-up
        (same kernels, same load) are used and the window says so."""
        t0, t1 = getattr(self, "start", None), getattr(self, "stop", None)
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
                "samples": len(sm), "window": window}


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

    dec_name = args.workload if (args.workload or "").startswith("decode") else DECODE_WL
    ctx_name = args.workload if (args.workload or "").startswith("ctx") else CTX_WL
    run_decode = not (args.workload or "").startswith("ctx")
    run_ctx = not (args.workload or "").startswith("decode")

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    dx = W.decode_workload(dec_name, device=dev) if run_decode else None
    paged = isinstance(dx, W.PagedDecodeInputs)
    dec_out = torch.empty_like(dx.q) if dx is not None else None

    def decode_call(q, kv_like, lens, out):
        # kv_like: the stacked kv tensor, or (k_pages, v_pages, block_table) of a paged cache
        if paged:
            gqa.gqa_decode_paged(q, *kv_like, lens, out=out, q_scale=dx.q_scale)
        else:
            gqa.gqa_decode(q, kv_like, lens, out=out, q_scale=dx.q_scale)
    cx = W.ctx_workload(ctx_name, device=dev) if run_ctx else None
    ctx_args = None
    ctx_out = None
    ctx_ok = run_ctx
    ctx_err = None
    if cx is not None:
        ctx_args = (cx.q_fp8, cx.k_fp4, cx.k_sf, cx.v_fp4, cx.v_sf, cx.block_table, cx.qo_indptr, cx.kv_lens)
        ctx_out = torch.empty_like(cx.q_fp8)
        try:
            gqa.nvfp4_paged_ctx_attn(*ctx_args, q_scale=cx.q_scale, out_scale=cx.out_scale, out=ctx_out)
            torch.cuda.synchronize()
        except gqa.GqaError as e:
            ctx_ok = False
            ctx_err = str(e)

    def step(evs):
        if dx is not None:
            evs[0].record(stream)
            decode_call(dx.q, (dx.k_pages, dx.v_pages, dx.block_table) if paged else dx.kv, dx.seq_lens, dec_out)
            evs[1].record(stream)
        if ctx_ok:
            flush.zero_()
            evs[2].record(stream)
            gqa.nvfp4_paged_ctx_attn(*ctx_args, q_scale=cx.q_scale, out_scale=cx.out_scale, out=ctx_out)
            evs[3].record(stream)

    all_evs = [_events(torch, 4) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let the sampler start before the GPU is loaded
        for _ in range(args.warmup):
            step(_events(torch, 4))
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
    dec_ms = [e[0].elapsed_time(e[1]) for e in all_evs] if dx is not None else []
    ctx_ms = [e[2].elapsed_time(e[3]) for e in all_evs] if ctx_ok else []
    dec_mean = statistics.fmean(dec_ms) if dec_ms else 0.0
    ctx_mean = statistics.fmean(ctx_ms) if ctx_ms else 0.0
    dec_max = max_over_ranks(dec_mean, dev)
    ctx_max = max_over_ranks(ctx_mean, dev)

    # e2e through the C ABI with host buffers (pinned): H2D of inputs and D2H
    # of the output inside the timed region, every step.
    e2e = None
    if rank == 0 and dx is not None:
        hq, hl = dx.q.cpu().pin_memory(), dx.seq_lens.cpu().pin_memory()
        if paged:
            hkv = tuple(t.cpu().pin_memory() for t in (dx.k_pages, dx.v_pages, dx.block_table))
        else:
            hkv = dx.kv.cpu().pin_memory()
        hout = torch.empty_like(hq).pin_memory()
        for _ in range(2):
            decode_call(hq, hkv, hl, hout)
        n_e2e = max(3, min(args.steps, 10))
        ts = []
        for _ in range(n_e2e):
            a, b = _events(torch, 2)
            a.record(stream)
            decode_call(hq, hkv, hl, hout)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        lens = hl.clamp(0, dx.capacity).to(torch.int64)
        if paged:  # the host path stages every page and the table
            h2d = hq.numel() * 2 + sum(t.numel() * t.element_size() for t in hkv) + hl.numel() * 4
        else:      # the host path stages each sequence's first len tokens
            h2d = hq.numel() * 2 + int(lens.sum()) * 16 * 256 + hl.numel() * 4
        d2h = hout.numel() * 2
        e2e_ms = statistics.fmean(ts)
        e2e = {"value": round(dx.kv_bytes_read() / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "steps": n_e2e,
               "path": ("gqa_decode_paged" if paged else "gqa_decode") + " with pinned host buffers"}
        del hkv

    if rank != 0:
        return
    clocks = clk.summary()
    line = {"metric": METRIC}
    n_launch_dec = gqa.gqa_decode_plan(dx.batch, dx.capacity)["num_launches"] if dx is not None else 0
    ctx_plan = (gqa.gqa_ctx_plan(cx.block_table.shape[0], cx.q_fp8.shape[0], cx.block_table.shape[1])
                if cx is not None else None)
    n_launch_ctx = ctx_plan["num_launches"] if (ctx_plan is not None and ctx_ok) else 0
    if dx is not None:
        gbs = dx.kv_bytes_read() * world / (dec_max * 1e-3) / 1e9
        # the committed counters were taken on decode_b64_cap8192 only
        traffic = (profiled_traffic("decode_split_kernel_decode_b64_cap8192.md", ["decode.cu", "common.cuh"])
                   if dec_name == DECODE_WL else None)
        line.update({
            "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dec_max + ctx_max, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": dec_name, "batch": dx.batch, "capacity": dx.capacity, "q_heads": 32,
                       "kv_layout": "64-token HND pages, shuffled block table" if paged else "stacked [B,2,8,cap,128]",
                       "kv_heads": 8, "head_dim": 128, "kv_bytes_read_per_step": dx.kv_bytes_read(),
                       "l2": "decode inputs larger than L2; L2 flushed (512 MB write) before each ctx call",
                       "parallelism": f"replicas{world}",
                       "ctx_workload": ctx_name if run_ctx else None},
            "decode_ms": round(dec_max, 4),
            "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / world / peaks["hbm_gbs"], 4),
                         "traffic": traffic,
                         "kernel": "decode_split_kernel (+ decode_merge_kernel inside the same events)",
                         "peak_source": peaks["source"] + " copy bandwidth"},
        })
    ctx_obj = None
    if run_ctx:
        if ctx_ok:
            flops = cx.causal_flops()
            tf = flops / (ctx_max * 1e-3) / 1e12
            fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
            # the committed counters were taken on ctx_b4_q2048_kv2048 only
            traffic_c = (profiled_traffic("ctx_nvfp4_kernel_ctx_b4_q2048_kv2048.md",
                                          ["ctx_nvfp4.cu", "common.cuh", "nvfp4.cuh"])
                         if ctx_name == CTX_WL else None)
            ctx_obj = {"value": round(tf * world, 2), "unit": "TFLOP/s", "ms": round(ctx_max, 4),
                       "causal_flops_per_step": flops, "workload": ctx_name, "dtype": "e4m3", "plan": ctx_plan,
                       "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": round(fp8_peak, 1),
                                    "unit": "TFLOP/s", "frac": round(tf / fp8_peak, 4), "traffic": traffic_c,
                                    "peak_source": f"{peaks['source']} bf16 x {FP8_OVER_BF16} (nominal FP8:bf16)"}}
            if ctx_name in PAGE_ROWS_US:
                label, us = PAGE_ROWS_US[ctx_name]
                ctx_obj["page_row"] = {"label": label, "us": us, "ours_us": round(ctx_max * 1e3, 2)}
        else:
            ctx_obj = {"unavailable": ctx_err or "not run"}
    if dx is None and ctx_ok:
        line.update({"value": ctx_obj["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                     "warmup": args.warmup, "ms_per_step": round(ctx_max, 4), "higher_is_better": True,
                     "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
                     "config": {"workload": ctx_name, "l2": "flushed before each call (512 MB write)",
                                "parallelism": f"replicas{world}"},
                     "roofline": ctx_obj["roofline"]})
    if ctx_obj is not None:
        line["ctx_attn"] = ctx_obj
    line["e2e"] = e2e
    line["gpu_launches"] = args.steps * (n_launch_dec + n_launch_ctx)
    line["clocks"] = clocks
    line["wall_s_timed_region"] = round(wall, 4)
    if args.cpu_baseline and dx is not None:
        line["cpu_baseline"] = oracle_decode_sample(dx, budget_s=args.cpu_budget)
    elif args.cpu_baseline and cx is not None:
        line["cpu_baseline"] = oracle_ctx_sample(cx, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


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


def oracle_decode_sample(dx, budget_s=15.0):
    """Time the oracle on the first n sequences (all 32 heads), n grown until
    the sample takes about `budget_s` seconds or covers the workload."""
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


def oracle_ctx_sample(cx, budget_s=15.0, rows=None):
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
    return {"value": round(flops / took / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(items)} random (row, head) items of {total}, {took:.2f} s"}


def run_reference(args):
    """The reference arm: the fp64 CPU oracle as it stands, on host cores."""
    import torch

    import gqa_workloads as W
    world, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.workload or DECODE_WL
    if name.startswith("ctx"):
        cx = W.ctx_workload(name)
        samples = []
        for i in range(args.warmup + args.steps):
            r = oracle_ctx_sample(cx, rows=args.ref_rows or 64)
            if i >= args.warmup:
                samples.append(r)
        value = statistics.fmean(s["value"] for s in samples)
        unit, dtype = "TFLOP/s", "f64"
        cfg = {"workload": name}
    else:
        dx = W.decode_workload(name, device="cuda" if torch.cuda.is_available() else "cpu")
        if isinstance(dx, W.PagedDecodeInputs):
            dx = W.PagedDecodeInputs(*(t.cpu() for t in (dx.q, dx.k_pages, dx.v_pages, dx.block_table, dx.seq_lens)),
                                     dx.q_scale)
        else:
            dx = W.DecodeInputs(dx.q.cpu(), dx.kv.cpu(), dx.seq_lens.cpu(), dx.q_scale)
        per_step = max(1, args.ref_seqs or 2)
        import oracle
        threads = oracle.default_threads()
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
        samples = [{"sample": f"{per_step} sequences (all 32 heads) per step", "cores": threads}]
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "kind": "oracle",
                             "cores": samples[0]["cores"], "sample": samples[0]["sample"]},
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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="a single named workload from gqa_workloads")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-seqs", type=int, default=0, help="reference arm: sequences per step (decode)")
    ap.add_argument("--ref-rows", type=int, default=0, help="reference arm: (row, head) items per step (ctx)")
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
    if args.warmup < 3 and args.impl == "ours":
        print("note: warm-up raised to the minimum of 3 steps", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
