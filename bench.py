#!/usr/bin/env python
"""Throughput of the fused FP8 paged MQA-logits + per-row top-k path on GB300.

One step = the fused call over one decode batch (block-table KV gather, FP8
q.K^T on tensor cores, relu-weighted head sum with masks, per-row top-k): the
KV pass and the selection launched as its programmatic dependent, timed
together with CUDA events on the launching stream. The two launches are also
timed apart (pmqa_logits_topk_stages SCORE, then SELECT, with an event
between them) for the kernel roofline. Inputs are synthetic
(synth.config_problem) and resident in HBM; L2 is flushed (256 MB write)
before every timed step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C0..C4] [--all]
    python bench.py --impl reference ...   # the CPU oracle on the same workload

Prints one JSON line (rank 0). Multi-GPU runs (torchrun) are independent
replicas: every rank owns a full copy of the batch, no data-path collective.
"""

from __future__ import annotations

import argparse
import dataclasses
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV tokens scored/sec and achieved HBM GB/s (% of GB300 peak); top-k rows/sec"
# The largest single-GPU workload by realised sum of contexts (1,353,194
# tokens) and the heaviest in compute (next_n 4 x 64 heads per token).
DEFAULT_WORKLOAD = "C3"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--all", action="store_true", default=True,
                    help="also time every other workload, the prefill and the sparse MLA decode (the default)")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline workload alone (no other workloads, no prefill)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--mla", nargs="*", default=None,
                    help="also time the sparse MLA decode workloads (all of them, or the ones "
                         "named) under --headline-only")
    ap.add_argument("--gather-ceiling", action="store_true",
                    help="instead of the step: time the row-gather probe (three issue methods) "
                         "on the rows the KV pass reads on C2 and C3 and the rows the sparse "
                         "MLA decode reads on M1, beside those kernels")
    ap.add_argument("--prefill", action="store_true",
                    help="also time the prefill (non-paged) logits on PF1 (on with --all)")
    args = ap.parse_args(argv)
    if args.headline_only:
        args.all = False
    return args


# ---------------------------------------------------------------- helpers


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, dist, device=None) -> float:
    """Largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device=None) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def read_tensor_peak():
    """Dense fp8 tensor peak (TFLOP/s): the measured bf16 cuBLAS burst figure
    times the nominal fp8 / bf16 ratio of 2, or the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "measured bf16_tflops x 2 (fp8/bf16)"
    except (OSError, KeyError, ValueError):
        return 2.0 * 1900.0, "fallback bf16 1900 TFLOP/s x 2 (fp8/bf16)"


def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources each kernel is built from (under the package's csrc/).
KERNEL_SOURCES = {
    "indexer": ("pmqa_ptx.cuh", "pmqa_main.cuh", "pmqa_kernel.cuh", "pmqa_main_inst.cu",
                "pmqa_select.cuh", "pmqa_api.cu"),
    "prefill": ("pmqa_ptx.cuh", "pmqa_main.cuh", "pmqa_prefill.cuh", "pmqa_prefill_inst.cu",
                "pmqa_api.cu"),
    "mla": ("pmqa_ptx.cuh", "pmqa_mla_ptx.cuh", "pmqa_mla.cu"),
}


def kernel_set(workload: str) -> str:
    return {"P": "prefill", "M": "mla"}.get(workload[:1], "indexer")


def kernel_source_hash(kind: str = "indexer") -> str:
    """Hash of the sources of one kernel family: a counter capture stays
    valid while they are unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_pmqa_gb300", "csrc")
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per launch of the workload's main kernel from a committed
    ncu summary, or None when absent or taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(kernel_set(workload)):
        return None
    return float(rec["dram_bytes_per_launch"])


def valid_positions(prob) -> int:
    """Sum over query rows of the positions the causal window admits."""
    total = 0
    for c in prob.context_lens.tolist():
        for j in range(prob.next_n):
            total += max(0, min(c - prob.next_n + j + 1, c))
    return total


def algorithmic_bytes(prob, k: int, logits_written: bool = False) -> dict:
    """Bytes the fused step must move at minimum: each KV row once (132 B per
    token), the block-table entries, q, weights and lengths, and its outputs."""
    import numpy as np

    ctx = prob.context_lens.astype(np.int64)
    rows = prob.bs * prob.next_n
    parts = {
        "kv": 132 * int(ctx.sum()),
        "block_table": 4 * int(((ctx + prob.block_size - 1) // prob.block_size).sum()),
        "q": int(prob.q.size),
        "weights": 4 * rows * prob.heads,
        "context_lens": 4 * prob.bs,
        "topk_out": 4 * rows * k,
    }
    if logits_written:
        parts["logits"] = 4 * rows * prob.max_model_len
    parts["total"] = sum(parts.values())
    return parts


def score_kernel_bytes(prob) -> dict:
    """Algorithmic bytes of one launch of the KV pass (SCORE stage): every KV
    row of every request once, its table entries, q, weights, lengths, and the
    compact logits it writes for the selection (4 B per admitted position)."""
    import numpy as np

    ctx = prob.context_lens.astype(np.int64)
    rows = prob.bs * prob.next_n
    parts = {
        "kv": 132 * int(ctx.sum()),
        "block_table": 4 * int(((ctx + prob.block_size - 1) // prob.block_size).sum()),
        "q": int(prob.q.size),
        "weights": 4 * rows * prob.heads,
        "context_lens": 4 * prob.bs,
        "compact_logits": 4 * valid_positions(prob),
    }
    parts["total"] = sum(parts.values())
    return parts


def kv_roofline(prob, score_ms: float, step_ms: float, peak: float) -> dict:
    """The KV-stream fractions: 132 B per token of every request, over the KV
    pass's own time (frac) and over the whole fused step (fused_frac), against
    the copy peak. The other bytes the KV pass moves (table entries, q,
    weights, lengths, the compact logits it writes for the selection) are
    reported beside them, not counted."""
    sb = score_kernel_bytes(prob)
    kv = sb["kv"]
    achieved = kv / (score_ms * 1e-3) / 1e9
    fused = kv / (step_ms * 1e-3) / 1e9
    other = {key: v for key, v in sb.items() if key not in ("kv", "total")}
    other["total"] = sum(other.values())
    return {"kv_bytes": kv, "achieved": achieved, "frac": achieved / peak,
            "fused_achieved": fused, "fused_frac": fused / peak, "other_bytes": other}


def cpu_description() -> dict:
    """The host CPU as the oracle sees it: model name, logical cores, the
    affinity mask of this process."""
    import platform

    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model", "processor name") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    try:
        aff = sorted(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        aff = list(range(os.cpu_count() or 1))
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "machine": platform.machine(), "logical_cpus": os.cpu_count(),
            "affinity": _ranges(aff)}


def _ranges(cpus) -> str:
    """[0, 1, 2, 5] -> "0-2,5"."""
    out, i = [], 0
    while i < len(cpus):
        j = i
        while j + 1 < len(cpus) and cpus[j + 1] == cpus[j] + 1:
            j += 1
        out.append(str(cpus[i]) if i == j else f"{cpus[i]}-{cpus[j]}")
        i = j + 1
    return ",".join(out)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.proc = None
        self.enabled = enabled

    def start(self):
        if not self.enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- our arm


def device_problem(prob, device):
    import torch

    return dict(
        q=torch.from_numpy(prob.q).to(device).view(torch.float8_e4m3fn),
        kv=torch.from_numpy(prob.kv).to(device),
        w=torch.from_numpy(prob.weights).to(device),
        ctx=torch.from_numpy(prob.context_lens).to(device),
        bt=torch.from_numpy(prob.block_tables).to(device),
    )


def time_steps(step, steps: int, flush) -> list:
    """Per-step device times (ms) with an L2 flush before each step."""
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        flush()
        e0.record()
        step()
        e1.record()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def time_staged_steps(stages, steps: int, flush):
    """Per-step device times (ms) of a step made of several launches: events
    before, between and after them; returns (step times, per-launch times)."""
    import torch

    n = len(stages)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    for ev in evs:
        flush()
        ev[0].record()
        for i, st in enumerate(stages):
            st()
            ev[i + 1].record()
    torch.cuda.synchronize()
    total = [ev[0].elapsed_time(ev[n]) for ev in evs]
    parts = [[ev[i].elapsed_time(ev[i + 1]) for ev in evs] for i in range(n)]
    return total, parts


def bench_workload(name, args, device, dist, with_e2e: bool, with_paths: bool):
    import torch

    from sparse_attention_indexer_pmqa_gb300 import pmqa
    from synth import config_problem

    prob = config_problem(name)
    k = prob.k
    d = device_problem(prob, device)
    rows = prob.rows
    ws = pmqa.workspace(prob.bs, prob.next_n, prob.max_model_len, k, pmqa.PMQA_OP_LOGITS_TOPK,
                        device)
    idx = torch.empty((rows, k), dtype=torch.int32, device=device)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.zero_()

    args_ = (d["q"], d["kv"], d["w"], d["ctx"], d["bt"], prob.max_model_len, k)

    def step():
        pmqa.pmqa_logits_topk(*args_, idx=idx, ws=ws)

    def stage_score():
        pmqa.pmqa_logits_topk_stages(*args_, pmqa.PMQA_STAGE_SCORE, idx=idx, ws=ws)

    def stage_select():
        pmqa.pmqa_logits_topk_stages(*args_, pmqa.PMQA_STAGE_SELECT, idx=idx, ws=ws)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    times = time_steps(step, args.steps, flush)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t0
    status = pmqa.pmqa_read_device_status(ws)
    if status:
        raise RuntimeError(f"device status {status:#x} during the timed steps")
    # the KV pass (SCORE stage) and the selection (SELECT stage) timed apart
    # for the kernel roofline
    n_k = min(args.steps, 100)
    for _ in range(3):
        stage_score()
        stage_select()
    _, (t_score, t_select) = time_staged_steps([stage_score, stage_select], n_k, flush)
    status = pmqa.pmqa_read_device_status(ws)
    if status:
        raise RuntimeError(f"device status {status:#x} during the stage timings")
    ms = statistics.fmean(times)
    ms_max = max_over_ranks(ms, dist, device)
    out = {"prob": prob, "ms": ms_max, "ms_median": statistics.median(times), "wall_s": wall,
           "times": times, "ms_score": max_over_ranks(statistics.fmean(t_score), dist, device),
           "ms_select": max_over_ranks(statistics.fmean(t_select), dist, device),
           "launches_per_step": 2}

    if with_paths:
        logits = torch.empty((rows, prob.max_model_len), dtype=torch.float32, device=device)
        ws_l = pmqa.workspace(prob.bs, prob.next_n, prob.max_model_len, 0, pmqa.PMQA_OP_LOGITS,
                              device)

        def step_logits():
            pmqa.pmqa_logits(d["q"], d["kv"], d["w"], d["ctx"], d["bt"], prob.max_model_len,
                             out=logits, ws=ws_l)

        def step_topk():
            pmqa.pmqa_topk(logits, d["ctx"], prob.next_n, k, idx=idx, ws=ws)

        n = min(args.steps, 50)
        for _ in range(3):
            step_logits()
            step_topk()
        out["paths_ms"] = {
            "pmqa_logits": statistics.fmean(time_steps(step_logits, n, flush)),
            "pmqa_topk": statistics.fmean(time_steps(step_topk, n, flush)),
            "pmqa_logits_topk (KV pass + selection)": ms,
            "SCORE stage (KV pass)": out["ms_score"],
            "SELECT stage (selection)": out["ms_select"],
        }
        del logits

    if with_e2e:
        host = {key: v.cpu().pin_memory() for key, v in d.items()}
        idx_h = torch.empty((rows, k), dtype=torch.int32).pin_memory()

        def step_e2e():
            for key in d:
                d[key].copy_(host[key], non_blocking=True)
            step()
            idx_h.copy_(idx, non_blocking=True)

        step_e2e()
        torch.cuda.synchronize()
        e_times = time_steps(step_e2e, args.e2e_steps, flush)
        out["e2e_ms"] = max_over_ranks(statistics.fmean(e_times), dist, device)
        out["h2d_bytes"] = sum(v.numel() * v.element_size() for v in host.values())
        out["d2h_bytes"] = idx_h.numel() * idx_h.element_size()
    return out


def prefill_cpu_baseline(p, rows: int = 1024):
    """The prefill oracle, as it stands, on a bounded sample: `rows` query rows
    spread evenly over the workload (rows are independent)."""
    import numpy as np

    import oracle

    oracle.build()
    sel = np.linspace(0, p.m - 1, rows).astype(np.int64)
    sub = dataclasses.replace(p, q=p.q[sel], weights=p.weights[sel], ks=p.ks[sel], ke=p.ke[sel])
    nthreads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.mqa_logits(sub, nthreads=nthreads)
    sec = time.perf_counter() - t0
    return {"value": sub.pairs / sec, "unit": "pairs/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{rows} of {p.m} query rows of {p.name}, evenly spaced ({sub.pairs} pairs), "
                      f"{sec:.2f} s"}


def bench_prefill(name, args, device):
    """Prefill logits (pmqa_mqa_logits) on one prefill workload: every step
    writes the whole [m, n] logits matrix; L2 flushed before each step."""
    import torch

    from sparse_attention_indexer_pmqa_gb300 import pmqa
    from synth import PREFILL_CONFIGS, prefill_config

    p = prefill_config(name)
    q = torch.from_numpy(p.q).to(device).view(torch.float8_e4m3fn)
    k = torch.from_numpy(p.k).to(device).view(torch.float8_e4m3fn)
    sc = torch.from_numpy(p.k_scale).to(device)
    w = torch.from_numpy(p.weights).to(device)
    ks = torch.from_numpy(p.ks).to(device)
    ke = torch.from_numpy(p.ke).to(device)
    out = torch.empty((p.m, p.n), dtype=torch.float32, device=device)
    ws = pmqa.workspace(p.m, 1, p.n, 0, pmqa.PMQA_OP_MQA_LOGITS, device)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.zero_()

    def step():
        pmqa.pmqa_mqa_logits(q, k, sc, w, ks, ke, out=out, ws=ws)

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    times = time_steps(step, min(args.steps, 100), flush)
    status = pmqa.pmqa_read_device_status(ws)
    if status:
        raise RuntimeError(f"device status {status:#x} during the prefill steps")
    ms = statistics.fmean(times)
    pairs = p.pairs
    flops = 2.0 * p.heads * 128 * pairs
    peak, peak_kind = read_tensor_peak()
    tflops = flops / (ms * 1e-3) / 1e12
    return {
        "workload": f"{name}: {PREFILL_CONFIGS[name]['desc']}",
        "ms": ms, "ms_median": statistics.median(times),
        "pairs": pairs, "pairs_per_s": pairs / (ms * 1e-3),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "peak_source": peak_kind,
                     "traffic": measured_traffic(name),
                     "algorithmic_flops_per_launch": flops,
                     "kernel": f"pmqa_prefill_kernel<{p.heads}> (with its prep launch)"},
        "out_gbs": p.m * p.n * 4 / (ms * 1e-3) / 1e9,
        "launches": 2,
    }


def mla_cpu_baseline(p, min_seconds: float = 3.0, max_reps: int = 50):
    """The MLA decode oracle, as it stands, on the whole workload (every query
    row), repeated until at least `min_seconds` have passed."""
    import oracle

    oracle.build()
    nthreads = oracle.default_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.sparse_mla(p, nthreads=nthreads)
        reps += 1
        sec = time.perf_counter() - t0
        if sec >= min_seconds or reps >= max_reps:
            break
    return {"value": reps * p.rows / sec, "unit": "query rows/s", "cores": nthreads,
            "kind": "oracle", "positions_per_s": reps * p.listed / sec,
            "sample": f"all {p.rows} query rows of {p.name} ({p.listed} listed positions), "
                      f"{reps} passes in {sec:.2f} s"}


def bench_mla(name, args, device):
    """Sparse MLA decode (pmqa_sparse_mla_decode) over one workload's listed
    positions: the call (attention kernel + the combining kernel) replayed
    from a CUDA graph; L2 flushed before each step."""
    import torch

    from sparse_attention_indexer_pmqa_gb300 import pmqa
    from synth import MLA_CONFIGS, mla_config

    p = mla_config(name)
    q = torch.from_numpy(p.q.reshape(p.rows, p.heads, -1)).to(device)
    kv = torch.from_numpy(p.kv).to(device)
    idx = torch.from_numpy(p.indices).to(device)
    bt = torch.from_numpy(p.block_tables).to(device)
    out = torch.empty((p.rows, p.heads, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((p.rows, p.heads), dtype=torch.float32, device=device)
    ws = pmqa.mla_workspace(p.rows, device)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.zero_()

    def call():
        pmqa.pmqa_sparse_mla_decode(q, kv, idx, bt, p.next_n, p.q_scale, p.kv_scale, p.sm_scale,
                                    out=out, lse=lse, ws=ws)

    for _ in range(max(args.warmup, 3)):
        flush()
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(3):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    times = time_steps(graph.replay, min(args.steps, 100), flush)
    status = pmqa.pmqa_read_device_status(ws)
    if status:
        raise RuntimeError(f"device status {status:#x} during the MLA decode steps")
    ms = statistics.fmean(times)
    listed = p.listed
    kv_bytes = listed * 576
    other = p.rows * p.heads * 576 + p.indices.size * 4 + p.rows * p.heads * (512 * 2 + 4)
    peak, peak_kind = read_peak()
    achieved = kv_bytes / (ms * 1e-3) / 1e9
    return {
        "workload": f"{name}: {MLA_CONFIGS[name]['desc']}",
        "ms": ms, "ms_median": statistics.median(times), "us": ms * 1e3,
        "rows": p.rows, "listed_positions": listed,
        "rows_per_s": p.rows / (ms * 1e-3), "positions_per_s": listed / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": measured_traffic(name),
                     "algorithmic_bytes_per_launch": kv_bytes,
                     "algorithmic": "576 B latent row per listed position",
                     "other_bytes_per_launch": other,
                     "kernel": "sparse_mla_kernel + sparse_mla_combine_kernel (one call, timed "
                               "whole)"},
        "launches": 2,
    }


def cpu_baseline(prob, min_seconds: float = 10.0, max_reps: int = 60):
    """The oracle, as it stands, on the whole workload (logits + top-k)."""
    import oracle

    oracle.build()
    nthreads = oracle.default_threads()
    reps, t_total = 0, 0.0
    while reps < max_reps and (reps == 0 or t_total < min_seconds):
        t0 = time.perf_counter()
        _, o64, _ = oracle.logits(prob, want64=True, nthreads=nthreads)
        oracle.topk(o64, prob.context_lens, prob.next_n, prob.k, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        reps += 1
        del o64
    per = t_total / reps
    rec = {"value": prob.total_ctx / per, "unit": "tokens/s", "cores": nthreads,
           "kind": "oracle",
           "sample": f"whole {prob.name} batch ({prob.total_ctx} tokens, logits + top-k), "
                     f"{reps} repetition(s), {per:.2f} s each"}
    rec.update(cpu_description())
    rec["single_thread"] = single_thread_baseline()
    return rec


def single_thread_baseline(names=("C0", "C1"), reps: int = 5) -> dict:
    """The oracle on one thread for the single-request workloads: median of
    `reps` whole runs (logits + top-k), in tokens/s."""
    import oracle
    from synth import config_problem

    out = {}
    for name in names:
        prob = config_problem(name)
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            _, o64, _ = oracle.logits(prob, want64=True, nthreads=1)
            oracle.topk(o64, prob.context_lens, prob.next_n, prob.k, nthreads=1)
            ts.append(time.perf_counter() - t0)
        med = statistics.median(ts)
        out[name] = {"value": prob.total_ctx / med, "unit": "tokens/s", "threads": 1,
                     "sample": f"median of {reps} whole runs, {med * 1e3:.1f} ms each"}
    return out


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    import __graft_entry__

    __graft_entry__.build()
    from synth import CONFIGS

    sampler = ClockSampler(local, enabled=not args.no_clocks and rank == 0)
    sampler.start()
    res = bench_workload(args.workload, args, device, dist, with_e2e=True, with_paths=True)
    clocks = sampler.stop()
    prob = res["prob"]
    ms = res["ms"]
    tokens_all = sum_over_ranks(prob.total_ctx, dist, device)
    value = tokens_all / (ms * 1e-3)
    peak, peak_kind = read_peak()
    ab = algorithmic_bytes(prob, prob.k)
    kr = kv_roofline(prob, res["ms_score"], ms, peak)
    traffic = measured_traffic(args.workload)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8e4m3-in/fp32-acc",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {CONFIGS[args.workload]['desc']}",
            "bs": prob.bs, "next_n": prob.next_n, "heads": prob.heads, "head_dim": 128,
            "block_size": prob.block_size, "sum_ctx": prob.total_ctx, "k": prob.k,
            "max_model_len": prob.max_model_len, "seed": 0,
            "l2": "flushed before every timed step (256 MB device write, not timed)",
            "parallelism": f"replicas x{world}",
        },
        "hbm_gbs": ab["total"] / (ms * 1e-3) / 1e9,
        "kv_stream_gbs": ab["kv"] / (ms * 1e-3) / 1e9,
        "topk_rows_per_s": world * prob.rows / (ms * 1e-3),
        "roofline": {
            "bound": "hbm", "achieved": kr["achieved"], "peak": peak, "unit": "GB/s",
            "frac": kr["frac"], "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
            "kernel": f"pmqa_main_kernel<{prob.heads}> (SCORE stage of the fused call)",
            "kernel_ms": res["ms_score"],
            "algorithmic_bytes_per_launch": kr["kv_bytes"],
            "algorithmic": "KV stream, 132 B per token of every request",
            "fused_frac": kr["fused_frac"], "fused_achieved": kr["fused_achieved"],
            "fused_ms": ms,
            "other_bytes_per_launch": kr["other_bytes"],
        },
        "e2e": {
            "value": tokens_all / (res["e2e_ms"] * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": res["h2d_bytes"], "d2h_bytes_per_step": res["d2h_bytes"],
            "note": "every input (q, whole KV pool, weights, lengths, tables) copied from "
                    "pinned host memory and the top-k indices read back, each step",
        },
        "gpu_launches": res["launches_per_step"] * args.steps,
        "paths_ms": res.get("paths_ms"),
        "ms_median": res["ms_median"],
    }
    if clocks:
        line["clocks"] = clocks
    if args.all:
        per = {}
        for wl in CONFIGS:
            if wl == args.workload:
                r = res
            else:
                r = bench_workload(wl, args, device, dist, with_e2e=False, with_paths=True)
            p = r["prob"]
            b = algorithmic_bytes(p, p.k)
            kw = kv_roofline(p, r["ms_score"], r["ms"], peak)
            per[wl] = {"workload": f"{wl}: {CONFIGS[wl]['desc']}", "ms": r["ms"],
                       "sum_ctx": p.total_ctx,
                       "tokens_per_s": p.total_ctx / (r["ms"] * 1e-3),
                       "gbs": b["total"] / (r["ms"] * 1e-3) / 1e9,
                       "score_ms": r["ms_score"], "select_ms": r["ms_select"],
                       "score_kv_gbs": kw["achieved"], "score_frac": kw["frac"],
                       "fused_kv_gbs": kw["fused_achieved"], "fused_frac": kw["fused_frac"],
                       "paths_ms": r.get("paths_ms")}
        line["workloads"] = per
    if args.all or args.prefill:
        line["prefill"] = bench_prefill("PF1", args, device)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            from synth import prefill_config

            line["prefill"]["cpu_baseline"] = prefill_cpu_baseline(prefill_config("PF1"))
    if args.all or args.mla is not None:
        from synth import MLA_CONFIGS

        names = list(MLA_CONFIGS) if args.all or not args.mla else args.mla
        line["sparse_mla_decode"] = {wl: bench_mla(wl, args, device) for wl in names}
        if rank == 0 and world == 1 and not args.no_cpu_baseline and "M1" in names:
            from synth import mla_config

            line["sparse_mla_decode"]["M1"]["cpu_baseline"] = mla_cpu_baseline(mla_config("M1"))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------- gather ceiling

GATHER_METHODS = {0: "ld16 (16-byte loads into registers)",
                  1: "cp.async16 (16-byte cp.async into shared memory)",
                  2: "bulk (one cp.async.bulk per row window)"}


def kv_rows(p):
    """Pool rows the KV pass reads for an indexer problem, in its order: every
    token t < ctx_i of request i through the block table (int32)."""
    import numpy as np

    P = p.block_size
    parts = []
    for i, c in enumerate(p.context_lens):
        t = np.arange(int(c), dtype=np.int64)
        parts.append(p.block_tables[i, t // P].astype(np.int64) * P + t % P)
    return np.concatenate(parts).astype(np.int32)


def mla_rows(p):
    """Pool rows the sparse MLA decode reads for an MLA problem, in its order:
    every listed position (holes skipped) of every query row (int32)."""
    import numpy as np

    req = np.arange(p.rows) // p.next_n
    pos = p.indices.astype(np.int64)
    ok = pos >= 0
    page = p.block_tables[np.repeat(req, p.topk).reshape(p.rows, p.topk),
                          np.where(ok, pos // p.block_size, 0)]
    return (page.astype(np.int64) * p.block_size + pos % p.block_size)[ok].astype(np.int32)


def gather_rows(name):
    """(pool array, int32 rows, row pitch) of a workload: the KV pass's rows
    for C*, the sparse MLA decode's for M*."""
    if name.startswith("M"):
        from synth import mla_config

        p = mla_config(name)
        return p.kv, mla_rows(p), 576
    from synth import config_problem

    p = config_problem(name)
    return p.kv, kv_rows(p), 132


def run_gather_ceiling(args):
    """How fast the GPU reads the same random rows the kernels read, by three
    issue methods (pmqa_gather_probe), beside the kernels' own times on the
    same workloads. One JSON line."""
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__

    __graft_entry__.build()
    from sparse_attention_indexer_pmqa_gb300 import pmqa

    peak, peak_kind = read_peak()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.zero_()

    reps = max(1, min(args.steps, 20))
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    sampler.start()
    res = {}
    for name in ("C2", "C3", "M1"):
        pool_np, rows_np, pitch = gather_rows(name)
        pool = torch.from_numpy(pool_np.reshape(-1)).to(device)
        rows = torch.from_numpy(rows_np).to(device)
        n = rows.numel()
        win = 144 if pitch == 132 else 576
        skipped = int(((rows_np.astype(np.int64) * pitch) // 16 * 16 + win > pool_np.size).sum())
        entry = {"rows": n, "row_bytes": pitch, "window_bytes": win,
                 "row_bytes_total": n * pitch, "rows_skipped_at_pool_end": skipped,
                 "methods": {}}
        xors = {}
        for m, label in GATHER_METHODS.items():
            out = torch.zeros(2, dtype=torch.int32, device=device)

            def call():
                pmqa.pmqa_gather_probe(pool, rows, pitch, m, out=out)

            for _ in range(max(args.warmup, 1)):
                flush()
                call()
            torch.cuda.synchronize()
            out.zero_()
            times = time_steps(call, reps, flush)
            o = out.cpu().tolist()
            # a window that would pass the pool's end (the pool's last row, read
            # as a 144-byte window) is skipped and flagged, nothing else
            if o[0] != (pmqa.PMQA_DEV_BAD_CONTEXT if skipped else 0):
                raise RuntimeError(f"gather probe status {o[0]:#x} on {name}, method {m}")
            xors[m] = o[1] if reps % 2 else None
            ms = statistics.fmean(times)
            entry["methods"][label] = {
                "us": ms * 1e3, "us_median": statistics.median(times) * 1e3,
                "row_gbs": n * pitch / (ms * 1e-3) / 1e9,
                "window_gbs": n * win / (ms * 1e-3) / 1e9,
                "row_frac": n * pitch / (ms * 1e-3) / 1e9 / peak}
        if xors[1] is not None and xors[1] != xors[2]:
            raise RuntimeError(f"cp.async and bulk copies read different bytes on {name}")
        if name.startswith("M"):
            r = bench_mla(name, args, device)
            entry["kernel"] = {"what": "pmqa_sparse_mla_decode (one call)", "us": r["us"],
                               "row_gbs": r["roofline"]["achieved"],
                               "row_frac": r["roofline"]["frac"]}
        else:
            r = bench_workload(name, args, device, None, with_e2e=False, with_paths=False)
            kv_bytes = 132 * r["prob"].total_ctx
            entry["kernel"] = {"what": "KV pass (SCORE stage of pmqa_logits_topk)",
                               "us": r["ms_score"] * 1e3,
                               "row_gbs": kv_bytes / (r["ms_score"] * 1e-3) / 1e9,
                               "row_frac": kv_bytes / (r["ms_score"] * 1e-3) / 1e9 / peak}
        best = max(v["row_gbs"] for v in entry["methods"].values())
        entry["kernel"]["of_best_probe"] = entry["kernel"]["row_gbs"] / best
        res[name] = entry
        del pool, rows
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    line = {"gather_ceiling": res, "peak": peak, "peak_source": f"{peak_kind} hbm_gbs",
            "reps": reps, "l2": "flushed before every timed launch (256 MB device write)",
            "note": "row_gbs counts the row bytes (132 or 576 per row); window_gbs the "
                    "16-byte aligned windows read"}
    if clocks:
        line["clocks"] = clocks
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- reference arm


def run_reference(args):
    """The CPU oracle on the same workload: each step scores one request of the
    batch (its logits rows and their top-k), in request order."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from synth import CONFIGS, Problem, config_problem

    oracle.build()
    prob = config_problem(args.workload)
    nthreads = oracle.default_threads()

    def step(s):
        i = s % prob.bs
        sub = Problem(
            q=np.ascontiguousarray(prob.q[i:i + 1]), kv=prob.kv,
            weights=np.ascontiguousarray(prob.weights[i * prob.next_n:(i + 1) * prob.next_n]),
            context_lens=prob.context_lens[i:i + 1].copy(),
            block_tables=np.ascontiguousarray(prob.block_tables[i:i + 1]), bs=1,
            next_n=prob.next_n, heads=prob.heads, block_size=prob.block_size,
            max_model_len=prob.max_model_len, k=prob.k, name=prob.name)
        _, o64, _ = oracle.logits(sub, want64=True, nthreads=nthreads)
        oracle.topk(o64, sub.context_lens, sub.next_n, sub.k, nthreads=nthreads)
        return int(sub.context_lens[0])

    for s in range(args.warmup):
        step(s)
    tokens, t0 = 0, time.perf_counter()
    for s in range(args.steps):
        tokens += step(args.warmup + s)
    dt = time.perf_counter() - t0
    value = tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {CONFIGS[args.workload]['desc']}",
                   "bs": prob.bs, "next_n": prob.next_n, "heads": prob.heads,
                   "block_size": prob.block_size, "k": prob.k,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                         "sample": "each step: one request of the batch, in order "
                                   "(its logits rows + top-k)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.gather_ceiling:
        run_gather_ceiling(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
