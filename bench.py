"""Benchmark: paged FP8 decode on one GB300 (dense decode workload).

Workload: batch 64, 8 KV heads, GQA8 (64 query heads), head_dim 128, query
length 1, page 16, context lengths uniform in [1024, 8192], pages dealt from a
random permutation of a 40,000-page pool, FP8 e4m3 K/V with per-tensor scales,
BF16 Q/output (synthetic, seeded).

One step = one pa_decode call over the whole batch. The KV bytes of one call
(604 MB) are larger than L2 (129 MB), and each timed step is preceded by a
read-only pass over a 512 MiB buffer (outside the events; read-only so that L2
holds no dirty lines whose write-back the decode would pay), as in the pages'
cold-sample protocol; the decode itself is timed with CUDA events on the
stream it is launched on.
`value` is achieved algorithmic HBM bandwidth (K/V of visible tokens,
block-table entries, context lengths, Q and output, counted once per call),
aggregated over all ranks; `us_per_call` is the mean device time per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

For N > 1 (torchrun) every rank decodes its own batch (replicas; no
collective on the data path) and rank 0 reports the aggregate over the max
time across ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time
from typing import Optional

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import pa_workloads as pw  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of GB300 peak) for paged FP8 decode, 1 GPU"
WORKLOAD = ("dense FP8 paged decode: batch 64, 8 KV heads, GQA8, head_dim 128, query length 1, "
            "page 16, contexts U[1024, 8192], 40k-page pool, per-tensor scales")
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
CPU_SAMPLE_UNITS = 48


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "hbm"):
            if key in peaks and float(peaks[key]) > 0:
                return float(peaks[key]), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# Sources that define each kernel: its own translation units and headers,
# plus the shared header and the host code that sets its launch.
KERNEL_SOURCES = {
    "pa_tile": ("pa_tile.cuh", "pa_tile_fp8_d128.cu", "pa_tile_fp8_d256.cu", "pa_tile_bf16.cu",
                "pa_tile_bf16_q16.cu", "pa_tile_fp4.cu", "pa_tile_bf16_tv.cu", "pa_tile_bf16_tv_q16.cu"),
    "pa_mtp": ("pa_tile.cuh", "pa_tc.cuh", "pa_mtp.cuh", "pa_mtp_fp8.cu", "pa_mtp_bf16.cu"),
    "pa_reduce": ("pa_tile.cuh", "pa_reduce.cu"),
    "pa_logits": ("pa_tile.cuh", "pa_tc.cuh", "pa_logits.cu"),
}
SHARED_SOURCES = ("pa_internal.h", "pa_host.cu")


def _code_only(text: str) -> str:
    """Source text without C/C++ comments and blank lines (what compiles)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str = "pa_tile") -> str:
    """Hash of the code (comments excluded) of the sources defining a kernel."""
    csrc = os.path.join(ROOT, "paged_attention_decode_attn_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(set(KERNEL_SOURCES[kernel]) | set(SHARED_SOURCES)):
        h.update(name.encode())
        h.update(_code_only(open(os.path.join(csrc, name), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profile_name(args, kernel: str) -> Optional[str]:
    """Name of the committed ncu summary for this bench line's kernel and
    workload (<kernel>_<workload>[_bf16][_ql<N>]), or None when the line runs
    a non-default size or variant (no summary covers it)."""
    if args.batch or args.page != 16 or args.window or args.sinks or args.partitions or args.merge != "auto" \
            or args.consumer != "auto" or (args.workload == "sparse_prefill" and args.rows != 1024):
        return None
    name = f"{kernel}_{args.workload}"
    if args.kv == "bf16" and args.workload in ("sparse", "mtp4", "sparse_prefill"):
        name += "_bf16"
    if (args.kv == "bf16" and args.workload == "dense") or args.v_layout != "plain":
        return None
    if args.kv == "mxfp4":
        name += "_mxfp4"
    if args.workload == "d256" and args.ql != 1:
        name += f"_ql{args.ql}"
    return name


def profiled_traffic(name: Optional[str], kernel: str = "pa_tile"):
    """DRAM bytes per launch from the committed ncu summary profiles/<name>.md,
    if it was taken on the current sources of `kernel`; else None."""
    if name is None:
        return None
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or kernel not in KERNEL_SOURCES:
        return None
    if m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return int(m_bytes.group(1))


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[2:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds: float, local_bytes: int, group=None):
    """Max time and total bytes over ranks (timing only; nothing on the data path)."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized():
        return local_seconds, local_bytes
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(b, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), int(b.item())


def _unit_bytes(w, units):
    """Algorithmic bytes of the sampled (sequence, KV head) units."""
    L = w.ctx_lens.astype(np.int64)
    per_tok = w.row_bytes * 2
    total = 0
    for u in units:
        b = int(u) // w.num_kv_heads
        total += int(L[b]) * per_tok + ((int(L[b]) + w.page_size - 1) // w.page_size) * 4
        total += 2 * w.group * w.query_len * w.head_dim * 2
    return total


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(w, units=CPU_SAMPLE_UNITS, seed=0, threads=1):
    """The oracle, as it is, on a bounded sample of units. threads > 1 runs a
    thread pool over the sampled units, one oracle call per unit (the C oracle
    runs without the GIL); threads == 1 is one call over all of them."""
    import concurrent.futures as cf

    import oracle

    orc = oracle.get()
    U = w.batch * w.num_kv_heads
    rng = np.random.default_rng(seed)
    pick = rng.choice(U, size=min(units, U), replace=False)

    def run(sel):
        mask = np.zeros(U, dtype=np.uint8)
        mask[sel] = 1
        orc.decode(w, unit_mask=mask)

    t0 = time.perf_counter()
    if threads <= 1:
        run(pick)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda u: run([u]), pick))
    dt = time.perf_counter() - t0
    how = "single-threaded" if threads <= 1 else f"a pool of {threads} threads, one unit per task"
    return {"value": _unit_bytes(w, pick) / dt / 1e9, "unit": "GB/s", "cores": max(1, threads), "kind": "oracle",
            "sample": f"{len(pick)} of {U} (sequence, KV head) units of the same workload, "
                      f"{dt:.1f} s, {how}, C in double precision",
            "seconds": dt}


WORKLOADS = {
    "dense": WORKLOAD,
    "tiny": "tiny paged decode: batch 2, 1 KV head, GQA8, head_dim 128, page 16, contexts {37, 100}, FP8 per-tensor",
    "d256": ("packed D256 long-context decode: batch 16, 2 KV heads, GQA8, head_dim 256, page 64, contexts "
             "{8K, 128K} + ragged tails and one empty sequence, FP8 per-token scales"),
    "sparse": ("sparse top-k decode: 64 rows, 16 query heads, 1 KV head, head_dim 128, page 16, 2048 of 131072 "
               "tokens per row, 4096-page pool"),
    "mtp4": ("dense MTP4 verify: batch 32, 4 KV heads, GQA16, head_dim 128, query length 4 causal, page 128, "
             "contexts U[4096, 65536]"),
    "sparse_prefill": ("sparse prefill: one prompt of N rows (--rows, default 1024), 16 query heads, 1 KV head, "
                       "head_dim 128, page 16, row r attends to min(r + 1, 2048) tokens, 4096-page pool"),
    "indexer": ("indexer logits: a 1024-row prompt chunk against 131072 KV tokens (cached prefix + chunk, row r "
                "sees [0, 130049 + r)), 64 heads, head_dim 128, FP8 Q and KV with per-token KV scales, "
                "-inf written outside the windows"),
}


SEQ_LEN = {"indexer": "131072 KV tokens", "dense": "U[1024,8192]", "tiny": "{37,100}", "d256": "{0, 8K+tail, 128K+tail}",
           "sparse": "2048 of 131072", "mtp4": "U[4096,65536]", "sparse_prefill": "min(r + 1, 2048) of r + 1"}
MERGES = {"auto": 0, "direct": 1, "cluster": 2, "last-arriver": 3, "reducer": 4}
CONSUMERS = {"auto": 0, "tile": 1, "tmem": 2}


def workload_name(args) -> str:
    name = WORKLOADS[args.workload]
    if args.kv == "mxfp4":
        name = name.replace("dense FP8 paged decode", "dense MXFP4 paged decode") + \
            ", MXFP4 K/V (E2M1 elements, one E8M0 scale per 32 head dims)"
    elif args.kv == "bf16" and args.workload in ("dense", "mtp4"):
        name = name.replace("dense FP8 paged decode", "dense BF16 paged decode") + ", BF16 K/V"
    if args.v_layout == "transposed":
        name += ", V transposed ([pages, heads, S/8, D, 8])"
    return name


def make_workload(args, rank):
    kv = {"fp8": pw.KV_FP8, "bf16": pw.KV_BF16, "mxfp4": pw.KV_MXFP4}[args.kv]
    if args.kv == "mxfp4" and args.workload not in ("dense", "mtp4"):
        raise SystemExit("--kv mxfp4 applies to the dense and mtp4 workloads")
    if args.v_layout == "transposed" and not (args.kv == "bf16" and args.workload in ("dense", "mtp4")):
        raise SystemExit("--v-layout transposed applies to --kv bf16 on the dense and mtp4 workloads")
    vl = pw.V_TRANSPOSED if args.v_layout == "transposed" else pw.V_PLAIN
    if args.workload == "dense":
        return pw.dense(seed=1002 + rank, page_size=args.page, batch=args.batch or 64, kv_dtype=kv, v_layout=vl)
    if args.workload == "tiny":
        return pw.tiny()
    if args.workload == "d256":
        return pw.d256(query_len=args.ql, window=args.window, with_sinks=args.sinks, batch=args.batch or 16)
    if args.workload == "sparse":
        return pw.sparse(kv_dtype=kv, rows=args.batch or 64)
    if args.workload == "mtp4":
        return pw.mtp4(kv_dtype=kv, batch=args.batch or 32, v_layout=vl)
    if args.workload == "sparse_prefill":
        return pw.sparse_prefill(kv_dtype=kv, rows=args.rows)
    raise ValueError(args.workload)


def run_indexer(args):
    """The indexer-logits line: FP8 tensor-core throughput (TFLOP/s of the
    scores inside the windows) with the same timing protocol as the decode."""
    import torch
    import torch.distributed as dist

    import paged_attention_decode_attn_gb300 as pa

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    w = pw.indexer(seed=1007 + rank, rows=args.batch or 1024)
    flops = w.flops()
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    host = {"q": pin(w.q), "kv": pin(w.kv), "sc": pin(w.kv_scale), "w": pin(w.weights), "ks": pin(w.ks),
            "ke": pin(w.ke)}
    d = {k: v.to(dev) for k, v in host.items()}
    stride = (w.num_kv + 3) // 4 * 4
    logits = torch.empty((w.rows, stride), dtype=torch.float32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def step(on=None):
        pa.pa_mqa_logits(logits, d["q"], d["kv"], d["sc"], d["w"], d["ks"], d["ke"], clean_logits=True,
                         status=status, stream=stream if on is None else on)

    for _ in range(max(3, args.warmup)):
        flush.sum(dtype=torch.int64)
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with Clocks(dev.index) as clk:
        torch.cuda._sleep(int(3e8))
        for i in range(K):
            flush.sum(dtype=torch.int64)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    per_call_ms = np.array([s_.elapsed_time(e) for s_, e in zip(starts, ends)])
    tot_s, tot_flops = aggregate(float(per_call_ms.sum()) / 1000.0, flops * K)
    st = int(status[0].item())
    warm_us = None if args.no_warm else warm_us_per_call(step, torch.cuda.Stream(dev))
    out_host = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = logits.numel() * logits.element_size()
    e2e_steps = args.e2e_steps
    for i in range(e2e_steps + 2):
        if i == 2:
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            t0 = time.perf_counter()
        for k_, v_ in host.items():
            d[k_].copy_(v_, non_blocking=True)
        step()
        out_host.copy_(logits, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s, e2e_flops = aggregate(time.perf_counter() - t0, flops * e2e_steps)
    if rank == 0:
        peaks = {}
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                peaks = json.load(f)
        except (OSError, ValueError):
            pass
        # FP8 dense peak: the measured BF16 burst figure times the nominal FP8/BF16 ratio (2)
        bf16 = float(peaks.get("bf16_tflops", 0) or 0)
        peak, kind = (2.0 * bf16, "measured bf16 burst x 2 (nominal fp8/bf16)") if bf16 > 0 else \
            (2.0 * 1900.0, "fallback bf16 1.9 PFLOP/s x 2")
        per_us = float(np.mean(per_call_ms)) * 1000.0
        achieved = flops / (per_us * 1e-6) / 1e12
        line = {
            "metric": "TFLOP/s of FP8 indexer logits (scores inside the windows, 2 FLOPs per multiply-add)",
            "value": tot_flops / tot_s / 1e12, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": float(np.mean(per_call_ms)), "us_per_call": per_us,
            "us_per_call_median": float(np.median(per_call_ms)) * 1000.0, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 (Q, KV), f32 accumulate and logits",
            "data": "synthetic (seeded pa_workloads.indexer)",
            "config": {"workload": WORKLOADS["indexer"], "global_batch": w.rows * world, "seq_len": SEQ_LEN["indexer"],
                       "heads": w.heads, "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "512 MiB read-only pass before every timed call"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_kind": kind,
                         "traffic": profiled_traffic(None if args.batch else "pa_logits_indexer", "pa_logits"),
                         "flops_per_launch": flops, "kernel": "pa_logits_kernel"},
            "e2e": {"value": e2e_flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": e2e_steps},
            "gpu_launches": K, "clocks": clk.summary(), "device_status": st,
        }
        if warm_us is not None:
            line["us_per_call_warm"] = warm_us
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = pw.dense()
    cores = host_cores()
    vals, secs = [], 0.0
    units = 2 * cores
    for s in range(args.warmup_ref + args.steps_ref):
        r = cpu_baseline(w, units=units, seed=s, threads=cores)
        if s >= args.warmup_ref:
            vals.append(r["value"])
            secs += r["seconds"]
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps_ref, "warmup": args.warmup_ref, "ms_per_step": 1000 * secs / len(vals),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 64, "seq_len": "U[1024,8192]",
                       "parallelism": "replicas", "l2": "cpu"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{units} random units per step of the same workload, a pool of "
                                       f"{cores} threads"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def warm_us_per_call(step, stream, calls=10, replays=5, runs=5, rounds=3):
    """The pages' warm protocol: a CUDA graph of `calls` decodes, replayed
    `replays` times per run; the minimum over `runs` runs, the median over
    `rounds` rounds, in µs per call (no L2 eviction between calls)."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step(stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(calls):
                step(stream)
    torch.cuda.synchronize()
    meds = []
    for _ in range(rounds):
        best = float("inf")
        for _ in range(runs):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                for _ in range(replays):
                    g.replay()
                b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b) * 1000.0 / (replays * calls))
        meds.append(best)
    return float(np.median(meds))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="dense", choices=sorted(WORKLOADS),
                    help="the headline line uses the default dense workload; the others are for profiling")
    ap.add_argument("--v-layout", default="plain", choices=["plain", "transposed"],
                    help="V cache layout (transposed: BF16 caches, dense and mtp4 workloads)")
    ap.add_argument("--kv", default="fp8", choices=["fp8", "bf16", "mxfp4"],
                    help="cache format (dense: fp8, bf16, mxfp4; mtp4: all three; sparse workloads: fp8, bf16)")
    ap.add_argument("--rows", type=int, default=1024, help="sparse_prefill: prompt rows")
    ap.add_argument("--page", type=int, default=16, help="dense: page size (16 is the workload's)")
    ap.add_argument("--batch", type=int, default=0,
                    help="mtp4/d256: batch override (a smaller case for profiler captures; 0 = the workload's)")
    ap.add_argument("--no-warm", action="store_true", help="skip the warm CUDA-graph timing")
    ap.add_argument("--ql", type=int, default=1, help="d256: query length (MTP rows)")
    ap.add_argument("--window", type=int, default=0, help="d256: sliding window (0 = off)")
    ap.add_argument("--sinks", action="store_true", help="d256: per-head sink logits")
    ap.add_argument("--partitions", type=int, default=0, help="plan max_partitions (per-unit schedule)")
    ap.add_argument("--merge", default="auto", choices=sorted(MERGES), help="plan merge mode")
    ap.add_argument("--consumer", default="auto", choices=sorted(CONSUMERS),
                    help="stage consumer: auto, tile (mma.sync) or tmem (tcgen05, 17..64 rows)")
    args = ap.parse_args()
    args.steps_ref = max(1, min(args.steps, 5))
    args.warmup_ref = 1 if args.warmup > 0 else 0
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "indexer":
        return run_indexer(args)

    import torch
    import torch.distributed as dist

    import paged_attention_decode_attn_gb300 as pa

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    w = make_workload(args, rank)
    alg = pw.algorithmic_bytes(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    host = {"q": pin(w.q.view(np.int16)).view(torch.bfloat16), "bt": pin(w.block_table), "ctx": pin(w.ctx_lens)}
    if w.kv_dtype == pw.KV_BF16:
        host["k"] = pin(w.k_cache.view(np.int16)).view(torch.bfloat16)
        host["v"] = pin(w.v_cache.view(np.int16)).view(torch.bfloat16)
    else:
        host["k"], host["v"] = pin(w.k_cache), pin(w.v_cache)
    for name, arr in (("ks", w.k_scale), ("vs", w.v_scale), ("sinks", w.sinks), ("idx", w.topk_idx)):
        if arr is not None:
            host[name] = pin(arr)
    d = {k: v.to(dev) for k, v in host.items()}
    out = torch.empty_like(d["q"])
    fields = dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                  head_dim=w.head_dim, query_len=w.query_len, page_size=w.page_size,
                  max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages,
                  max_context_len=int(w.ctx_lens.max()), kv_dtype=w.kv_dtype, scale_mode=w.scale_mode,
                  causal=int(w.causal), has_sinks=int(w.sinks is not None), sparse_topk=int(w.topk))
    if args.partitions:
        fields.update(schedule=pa.PA_SCHED_PER_UNIT, max_partitions=args.partitions)
    fields["merge_mode"] = MERGES[args.merge]
    fields["consumer"] = CONSUMERS[args.consumer]
    plan = pa.Plan(device=dev, **fields)
    stream = torch.cuda.current_stream(dev)
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        return flush.sum(dtype=torch.int64)

    def step(on=None):
        on = stream if on is None else on
        if w.topk:
            plan.decode_sparse(out, d["q"], d["k"], d["v"], d["bt"], d["ctx"], d["idx"], d.get("ks"), d.get("vs"),
                               d.get("sinks"), stream=on)
        else:
            plan.decode(out, d["q"], d["k"], d["v"], d["bt"], d["ctx"], d.get("ks"), d.get("vs"), w.window,
                        d.get("sinks"), stream=on)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with Clocks(dev.index) as clk:
        # Keep the GPU busy while the host enqueues the timed steps, so that no
        # host-side gap falls between a step's start and end events.
        torch.cuda._sleep(int(3e8))
        for i in range(K):
            flush_l2()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    per_call_ms = np.array([s.elapsed_time(e) for s, e in zip(starts, ends)])
    local_s = float(per_call_ms.sum()) / 1000.0
    tot_s, tot_bytes = aggregate(local_s, alg * K)
    status = plan.device_status()

    warm_us = None if args.no_warm else warm_us_per_call(step, torch.cuda.Stream(dev))

    # end to end through the public API: pinned host inputs -> device, decode, output -> host
    e2e_steps = args.e2e_steps
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out.numel() * out.element_size()
    for i in range(e2e_steps + 2):
        if i == 2:
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            t0 = time.perf_counter()
        for k_, v_ in host.items():
            d[k_].copy_(v_, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_local = time.perf_counter() - t0
    e2e_s, e2e_bytes = aggregate(e2e_local, alg * e2e_steps)

    if rank == 0:
        peak, peak_kind = measured_peak_gbs()
        kernel_name = "pa_mtp_kernel" if plan.info["consumer"] == pa.PA_CONSUMER_TMEM else "pa_tile_kernel"
        per_launch_us = float(np.mean(per_call_ms)) * 1000.0
        achieved = alg / (per_launch_us * 1e-6) / 1e9
        value = tot_bytes / tot_s / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": float(np.mean(per_call_ms)),
            "us_per_call": per_launch_us, "us_per_call_median": float(np.median(per_call_ms)) * 1000.0,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {pw.KV_FP8: "fp8-e4m3", pw.KV_BF16: "bf16", pw.KV_MXFP4: "mxfp4 (e2m1, e8m0 per 32)"}[w.kv_dtype]
                     + " (KV), bf16 (Q/O), f32 accumulate",
            "data": f"synthetic (seeded pa_workloads.{args.workload})",
            "config": {"workload": workload_name(args), "global_batch": w.batch * world,
                       "seq_len": SEQ_LEN[args.workload], "query_len": w.query_len,
                       "window": int(w.window), "sinks": w.sinks is not None,
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "512 MiB read-only pass before every timed call (dense: inputs also larger than L2)",
                       "plan": {k: plan.info[k] for k in ("schedule", "merge_mode", "consumer", "num_partitions", "grid",
                                                         "block_threads", "num_stages", "stage_tokens",
                                                         "ctas_per_sm", "launches_per_call")}},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": profiled_traffic(profile_name(args, kernel_name.replace("_kernel", "")),
                                                     kernel_name.replace("_kernel", "")),
                         "algorithmic_bytes_per_launch": alg, "kernel": kernel_name},
            "e2e": {"value": e2e_bytes / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": e2e_steps},
            "gpu_launches": int(K * plan.info["launches_per_call"]),
            "clocks": clk.summary(),
            "device_status": status,
        }
        if warm_us is not None:
            line["us_per_call_warm"] = warm_us
            line["warm_protocol"] = "10-call CUDA graph x 5 replays, min of 5 runs, median of 3 rounds, no L2 eviction"
        if world == 1 and not args.no_cpu_baseline and args.workload == "dense":
            cores = host_cores()
            # all host cores over every unit of the workload (a few seconds on
            # 16 cores), and one thread over a sample of 64 units
            cb = cpu_baseline(w, units=w.batch * w.num_kv_heads, threads=cores)
            cb.pop("seconds")
            single = cpu_baseline(w, units=64, seed=1)
            single.pop("seconds")
            cb["single_thread"] = single
            line["cpu_baseline"] = cb
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
