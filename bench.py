#!/usr/bin/env python
"""Benchmark of the block-selection hot path: indexer block scorer + block top-k.

One step = one chained select call (scorer, then top-k) on the deep prompt
workload: 256 queries x 16 indexer heads x head dim 128, bf16 q and kblk
~ N(0,1), fp32 w ~ U(0,1), 520,000 tokens of context (8,125 blocks of 64, the
last one partial), k = 32, KV capacity 524,288 tokens.  Inputs are resident in
HBM; L2 is flushed (a 256 MB write) before every timed step; each step is
timed with CUDA events on the launching stream.

Printed (rank 0, one JSON line): the metric (us per select call, lower is
better), the dominant kernel's roofline against MEASURED_PEAKS.json, the
top-k and decode-window (3 queries, 258,000 tokens) figures, an end-to-end
number through the C ABI with host buffers (H2D of the inputs and D2H of the
ids inside the timed region), SM clocks sampled during the timed region, and
the CPU oracle timed on a bounded sample of the same workload.  The selection
attention over the timed call's ids (64 heads in 4 GQA groups of 16, K and V
caches of 524,288 tokens) is timed beside it, with its own HBM roofline, and
over the decode window's ids; it is not part of the step.  So is the deep
prompt with fp8 e4m3 queries and keys (both select forms and the scorer).

``--impl reference`` times the CPU oracle (the only reference this method has)
on the host cores, each step a bounded sample of the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import inputs  # noqa: E402

METRIC = "us per select call (score+top-k), 256q x 520K tokens"
UNIT = "us/call"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(case):
    n = int(case.n_blocks[0])
    return {
        "workload": f"deep prompt call: {case.nq} queries x {case.n_heads} heads x 128, bf16, "
                    f"{int(case.tokens[0]):,} tokens ({n:,} blocks of 64), k={case.k}, capacity 524,288 tokens",
        "nq": case.nq, "n_heads": case.n_heads, "n_blocks": n, "k": case.k,
        "l2": "flushed before every timed step (256 MB write)",
    }


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 100 ms while active."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd[1:1] = ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- helpers

# The source files each timed kernel is compiled from; a committed DRAM-traffic
# figure is reported only while all of them are unchanged.
KERNEL_SOURCES = {
    "fused": ("scorer_tc.cu", "warp_topk.cuh", "qsa_device.cuh", "tc_ptx.cuh", "sharded.cu"),
    "scorer": ("scorer_tc.cu", "tc_ptx.cuh"),
    "topk": ("topk.cu", "warp_topk.cuh", "qsa_device.cuh"),
    "attention": ("sel_attn.cu", "tc_ptx.cuh", "qsa_device.cuh"),
}


def kernel_source_hash(key: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[key]:
        with open(os.path.join(ROOT, "sparse_attention_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(key)
    if not e or e.get("source_sha") != kernel_source_hash(key):
        return None
    return e.get("dram_bytes_per_launch")


PRIME_CYCLES = 400_000   # ~0.2 ms of GPU sleep queued ahead of each step


def timed_loop(torch, fn, steps, flush, stream, prime=True):
    """Per-step CUDA-event times (ms) of fn(), L2 flushed before each step.

    A short GPU sleep is queued ahead of each step, so the host has enqueued the
    whole step before the GPU reaches its start event: the events time the
    kernels, not the host's launch overhead.  prime=False keeps the host in the
    measurement (end to end).
    """
    times = []
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if prime:
            torch.cuda._sleep(PRIME_CYCLES)
        flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    for s, e in zip(starts, ends):
        times.append(s.elapsed_time(e))
    return times


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest of every rank's value (the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(ms_per_step_max: float, world: int) -> float:
    """Whole-job figure for N replicas: each rank runs one call per step, so the job
    completes `world` calls in the slowest rank's step time."""
    return ms_per_step_max * 1e3 / world


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle on the host cores: each step scores and selects a bounded sample of queries."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    case = inputs.deep_case(2)
    sample_q = args.ref_sample_queries
    sub = slice(0, sample_q)

    def step():
        s = oracle.block_scores(case.q[sub], case.w[sub], case.kblk, case.n_blocks[sub], case.dtype)
        oracle.select(s, case.n_blocks[sub], case.k)

    for _ in range(args.warmup):
        step()
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        t.append(time.perf_counter() - t0)
    per_call_us = statistics.mean(t) * 1e6 * case.nq / sample_q
    cfg = workload_config(case)
    cfg["path"] = "CPU oracle (FP64 scores, full sort), single thread"
    line = {
        "impl": "reference", "metric": METRIC, "value": per_call_us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(t) * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/kblk, U(0,1) w)", "config": cfg,
        "cpu_baseline": {"value": per_call_us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{sample_q} of {case.nq} queries per step, scaled to the full call"},
        "e2e": {"value": per_call_us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- our arm

def cpu_model() -> str:
    """The host CPU's model name (lscpu's, else /proc/cpuinfo's), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(case, target_s=10.0):
    import oracle
    oracle.build()
    per_q = []
    done = 0
    t_start = time.perf_counter()
    while done < case.nq and (time.perf_counter() - t_start) < target_s:
        sl = slice(done, done + 4)
        t0 = time.perf_counter()
        s = oracle.block_scores(case.q[sl], case.w[sl], case.kblk, case.n_blocks[sl], case.dtype)
        oracle.select(s, case.n_blocks[sl], case.k)
        per_q.append((time.perf_counter() - t0) / len(case.n_blocks[sl]))
        done += len(case.n_blocks[sl])
    us = statistics.mean(per_q) * case.nq * 1e6
    return {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
            "host_cores": os.cpu_count(),
            "sample": f"{done} of {case.nq} queries of the same workload (about {target_s:.0f} s), "
                      f"FP64 scores + full sort, single thread, scaled to the full call"}


def cpu_baseline_all_cores(case, target_s=6.0):
    """The same oracle over every host core: threads take 4-query slices (the oracle's C
    calls release the GIL) until the time is up; wall time per query, scaled to the call."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    cores = os.cpu_count() or 1
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t_start = time.perf_counter()

    def worker():
        while time.perf_counter() - t_start < target_s:
            with lock:
                lo = state["next"] % case.nq
                state["next"] += 4
            sl = slice(lo, min(lo + 4, case.nq))
            s = oracle.block_scores(case.q[sl], case.w[sl], case.kblk, case.n_blocks[sl], case.dtype)
            oracle.select(s, case.n_blocks[sl], case.k)
            with lock:
                state["done"] += sl.stop - sl.start

    with ThreadPoolExecutor(cores) as ex:
        for f in [ex.submit(worker) for _ in range(cores)]:
            f.result()
    wall = time.perf_counter() - t_start
    return {"value": wall / state["done"] * case.nq * 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{state['done']} queries of the same workload over {cores} threads in {wall:.1f} s, "
                      f"scaled to the full call"}


def attention_bytes(c) -> float:
    """Algorithmic bytes of one selection-attention call: K and V of every selected
    block of every (query, KV head) (2 x 64 x 128 bf16 = 32 KB), the queries, the
    outputs, the lse, the ids and the context lengths, each read or written once."""
    n_sel = int((c.ids >= 0).sum())
    return (32768.0 * n_sel * c.n_kv_heads + c.nq * c.n_heads * (256.0 + 512.0 + 4.0)
            + 4.0 * c.ids.size + 4.0 * c.nq)


def attention_unique_bytes(c) -> float:
    """K and V bytes of the distinct blocks the whole call selects (every KV head reads
    the same block ids): the traffic if each block were read from HBM once."""
    ids = c.ids[c.ids >= 0]
    return 32768.0 * len(np.unique(ids)) * c.n_kv_heads


def attention_report(acase, adcase, us, us_dec, peaks, peak_src):
    b = attention_bytes(acase)
    gbs = b / (us * 1e-6) / 1e9
    bu = attention_unique_bytes(acase)
    traffic = profiled_traffic("attention")
    bd = attention_bytes(adcase)
    gbs_d = bd / (us_dec * 1e-6) / 1e9
    return {
        "workload": acase.name, "ids": "the deep select call's ids (k = 32)",
        "kernel": "sel_attn_kernel", "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": gbs / peaks["hbm_gbs"], "traffic": profiled_traffic("attention"),
        "per_launch": f"{b:.4g} B (32 KB of K and V per query, KV head and selected block; q, out, lse, ids)",
        "us_per_launch": us, "l2": "flushed before every timed call", "peak_source": f"{peak_src} HBM copy",
        "note": "the algorithmic bytes count one 32 KB block read per (query, KV head, selected block); queries "
                "that select the same block share it through L2, so DRAM moves less",
        "bytes_unique_blocks": bu, "frac_unique_blocks": bu / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
        "dram_frac_from_traffic": None if traffic is None else traffic / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
        "decode": {"workload": adcase.name, "us_per_call": us_dec, "bytes": bd, "gbs": gbs_d,
                   "frac_of_hbm": gbs_d / peaks["hbm_gbs"]},
    }


def us_mean(times_ms):
    """Mean of per-call event times, in us.  The event timer's resolution is coarse on
    this GPU (about 2 us steps), so the mean over many calls is reported, not the
    median, which snaps to the step."""
    return statistics.mean(times_ms) * 1e3


def graph_us_per_call(torch, fns, replays=5):
    """Device time per call of the calls ``fns`` captured in one CUDA graph and replayed
    back to back: no host launch between them and no L2 flush, so a kernel whose inputs
    rotate through more memory than L2 holds still reads them from DRAM.  Events
    around each replay; mean over the replays, divided by the calls."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(replays):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts) * 1e3 / len(fns)


def oracle_scores(case, rows=None):
    """FP64 oracle scores of the case's queries ``rows`` (all by default), over every
    host core (the oracle's C calls release the GIL)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    rows = np.arange(case.nq) if rows is None else np.asarray(rows)
    chunks = [rows[i:i + 8] for i in range(0, len(rows), 8)]
    with ThreadPoolExecutor(os.cpu_count() or 1) as ex:
        parts = list(ex.map(lambda r: oracle.block_scores(case.q[r], case.w[r], case.kblk, case.n_blocks[r],
                                                          case.dtype), chunks))
    return np.concatenate(parts, axis=0)


def parity_report(case, gpu_scores, chained_ids, timed_ids, form):
    """Rules (a)-(c) on a timed workload, through the oracle, outside any timed region:
    (a) the chained call's ids against the oracle's selection over the GPU's own scores,
    (b) the GPU's scores against the FP64 oracle, (c) the timed form's ids against the
    oracle's FP64 selection, with the near-tie counts at the tolerance and at four times
    the observed score error."""
    import oracle
    from oracle import parity
    ref = oracle_scores(case)
    n = case.n_blocks
    err = parity.score_errors(gpu_scores, ref, n)
    a_ids = oracle.select_f32(gpu_scores, n, case.k)
    a_same = int((chained_ids == a_ids).all(1).sum())
    tol = parity.TOL[case.dtype]
    tight = max(4.0 * float(err.max()), 1e-9)
    rc = parity.rule_c(timed_ids, ref, oracle.select(ref, n, case.k), n, case.k, tol, tight)
    rc.pop("failed_ids")
    return {"workload": case.name, "queries": case.nq,
            "rule_a": {"identical_queries": a_same, "pass": a_same == case.nq},
            "rule_b": {"max_normalised_error": float(err.max()), "tol": tol, "pass": bool(err.max() <= tol)},
            "rule_c": dict(rc, form=form, tol=tol, tight_tol=tight, **{"pass": rc["failed"] == 0})}


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from sparse_attention_kv_gb300 import qsa
    from workloads import device
    qsa.load()
    stream = torch.cuda.current_stream()

    case = inputs.deep_case(2)
    q, w, kb, nb = device.to_device(case, dev)
    C = case.max_blocks
    n = int(case.n_blocks[0])
    scores = torch.empty((case.nq, C), dtype=torch.float32, device=dev)
    ids = torch.empty((case.nq, case.k), dtype=torch.int32, device=dev)
    ws = qsa.alloc_workspace(case.nq, C, case.k, device=dev)
    flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.zero_()

    fws = qsa.alloc_workspace(case.nq, C, case.k, fused=True, device=dev)

    def select_chained():
        qsa.select(q, w, kb, nb, case.k, ids, ws, scores=scores, active_blocks=case.active_blocks)

    def select_fused():
        qsa.select(q, w, kb, nb, case.k, ids, fws, fused=True, active_blocks=case.active_blocks)

    def score_only():
        qsa.block_scores(q, w, kb, nb, scores, active_blocks=case.active_blocks, ws=ws)

    def topk_only():
        qsa.block_topk(scores, nb, case.k, ids, ws, active_blocks=case.active_blocks)

    path = qsa.auto_path(case.nq, C, case.active_blocks, case.k)
    topk_launches = 1

    # decode window, 3 queries at 258,000 tokens
    dcase = inputs.decode_case(5)
    dq, dw, dkb, dnb = device.to_device(dcase, dev)
    dscores = torch.empty((dcase.nq, dcase.max_blocks), dtype=torch.float32, device=dev)
    dids = torch.empty((dcase.nq, dcase.k), dtype=torch.int32, device=dev)
    dws = qsa.alloc_workspace(dcase.nq, dcase.max_blocks, dcase.k, device=dev)
    dpath = qsa.auto_path(dcase.nq, dcase.max_blocks, -1, dcase.k)

    dfws = qsa.alloc_workspace(dcase.nq, dcase.max_blocks, dcase.k, fused=True, device=dev)

    def decode_chained():
        qsa.select(dq, dw, dkb, dnb, dcase.k, dids, dws, scores=dscores, active_blocks=-1)

    def decode_fused():
        qsa.select(dq, dw, dkb, dnb, dcase.k, dids, dfws, fused=True, active_blocks=-1)

    # end to end: the step's inputs (q, w, kblk, n_blocks) staged in one pinned host
    # buffer in 256-byte aligned sections, one host-to-device copy, the call on views of
    # the device copy, and the ids read back to pinned host memory
    sections = (q, w, kb, nb)
    offs, total = [], 0
    for t in sections:
        total = (total + 255) // 256 * 256
        offs.append(total)
        total += t.numel() * t.element_size()
    hstage = torch.empty(total, dtype=torch.uint8).pin_memory()
    dstage = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(sections, offs):
        nbytes = t.numel() * t.element_size()
        hstage[o:o + nbytes].copy_(t.cpu().contiguous().view(torch.uint8).reshape(-1))
        views.append(dstage[o:o + nbytes].view(t.dtype).view(t.shape))
    eq_, ew_, ekb_, enb_ = views
    hids = torch.empty_like(ids, device="cpu").pin_memory()

    def e2e_step():
        dstage.copy_(hstage, non_blocking=True)
        if form == "fused":
            qsa.select(eq_, ew_, ekb_, enb_, case.k, ids, fws, fused=True, active_blocks=case.active_blocks)
        else:
            qsa.select(eq_, ew_, ekb_, enb_, case.k, ids, ws, scores=scores, active_blocks=case.active_blocks)
        hids.copy_(ids, non_blocking=True)

    h2d = sum(t.numel() * t.element_size() for t in sections)
    d2h = hids.numel() * hids.element_size()

    # selection attention over the select calls' own ids: 64 heads in 4 GQA groups of 16,
    # K and V caches of the same capacity, contexts of the same length
    select_chained()
    decode_chained()
    torch.cuda.synchronize()
    acase = inputs.deep_attention_case(ids=ids.cpu().numpy())
    a_dev = device.attn_to_device(acase, dev)
    a_out = torch.empty((acase.nq, acase.n_heads, 128), dtype=torch.float32, device=dev)
    a_lse = torch.empty((acase.nq, acase.n_heads), dtype=torch.float32, device=dev)
    adcase = inputs.decode_attention_case(ids=dids.cpu().numpy())
    ad_dev = device.attn_to_device(adcase, dev)
    ad_out = torch.empty((adcase.nq, adcase.n_heads, 128), dtype=torch.float32, device=dev)
    ad_lse = torch.empty((adcase.nq, adcase.n_heads), dtype=torch.float32, device=dev)

    # the prompt call: 256 queries at 131,072 tokens
    pcase = inputs.prompt_case()
    pq, pw, pkb, pnb = device.to_device(pcase, dev)
    pscores = torch.empty((pcase.nq, pcase.max_blocks), dtype=torch.float32, device=dev)
    pids = torch.empty((pcase.nq, pcase.k), dtype=torch.int32, device=dev)
    pws = qsa.alloc_workspace(pcase.nq, pcase.max_blocks, pcase.k, fused=True, device=dev)

    def prompt_chained():
        qsa.select(pq, pw, pkb, pnb, pcase.k, pids, pws, scores=pscores, active_blocks=pcase.active_blocks)

    def prompt_fused():
        qsa.select(pq, pw, pkb, pnb, pcase.k, pids, pws, fused=True, active_blocks=pcase.active_blocks)

    def prompt_score():
        qsa.block_scores(pq, pw, pkb, pnb, pscores, active_blocks=pcase.active_blocks, ws=pws)

    # the deep prompt with fp8 e4m3 queries and keys
    ecase = inputs.deep_e4m3_case()
    eq, ew, ekb, enb = device.to_device(ecase, dev)
    escores = torch.empty((ecase.nq, ecase.max_blocks), dtype=torch.float32, device=dev)
    eids = torch.empty((ecase.nq, ecase.k), dtype=torch.int32, device=dev)
    ews = qsa.alloc_workspace(ecase.nq, ecase.max_blocks, ecase.k, fused=True, device=dev)

    def e4m3_chained():
        qsa.select(eq, ew, ekb, enb, ecase.k, eids, ews, scores=escores, active_blocks=ecase.active_blocks)

    def e4m3_fused():
        qsa.select(eq, ew, ekb, enb, ecase.k, eids, ews, fused=True, active_blocks=ecase.active_blocks)

    def e4m3_score():
        qsa.block_scores(eq, ew, ekb, enb, escores, active_blocks=ecase.active_blocks, ws=ews)

    def attend():
        qsa.select_attention(*a_dev, a_out, a_lse, scale=acase.scale)

    def attend_decode():
        qsa.select_attention(*ad_dev, ad_out, ad_lse, scale=adcase.scale)

    form = "fused"
    if args.profile_steps:
        # a fixed, short sequence of launches for ncu: both forms on both workloads
        for _ in range(args.profile_steps):
            select_chained()
            select_fused()
            decode_chained()
            decode_fused()
            attend()
            attend_decode()
        torch.cuda.synchronize()
        return 0

    # warm-up (also brings the clocks up)
    for _ in range(max(3, args.warmup)):
        flush()
        select_chained()
        select_fused()
        decode_chained()
        decode_fused()
    torch.cuda.synchronize()
    t_end = time.time() + 0.5
    while time.time() < t_end:
        select_fused()
        select_chained()
    torch.cuda.synchronize()
    # qsa_select has two forms (one fused kernel, or scorer then top-k); the faster
    # one on this GPU is the call a user makes, and is the one timed below
    probe = {f: statistics.mean(timed_loop(torch, fn, 30, flush, stream))
             for f, fn in (("fused", select_fused), ("chained", select_chained))}
    form = min(probe, key=probe.get)
    select = select_fused if form == "fused" else select_chained
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    gpu_uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{gpu_uuid}" if gpu_uuid and not str(gpu_uuid).startswith("GPU-") else (
        str(gpu_uuid) if gpu_uuid else None)
    sampler = ClockSampler(gpu_id).start()
    time.sleep(0.25)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_main = timed_loop(torch, select, args.steps, flush, stream)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    reps = max(args.steps, 200)
    t_other = timed_loop(torch, select_chained if form == "fused" else select_fused, reps, flush, stream)
    t_score = timed_loop(torch, score_only, reps, flush, stream)
    t_topk = timed_loop(torch, topk_only, reps, flush, stream)
    t_dec_f = timed_loop(torch, decode_fused, reps, flush, stream)
    t_dec_c = timed_loop(torch, decode_chained, reps, flush, stream)
    t_e2e = timed_loop(torch, e2e_step, args.steps, flush, stream, prime=False)
    t_prompt = {name: timed_loop(torch, fn, reps, flush, stream)
                for name, fn in (("chained", prompt_chained), ("fused", prompt_fused), ("scorer", prompt_score))}
    t_e4m3 = {name: timed_loop(torch, fn, reps, flush, stream)
              for name, fn in (("chained", e4m3_chained), ("fused", e4m3_fused), ("scorer", e4m3_score))}
    def deep_step():
        select()
        attend()

    def decode_step():
        decode_chained()
        attend_decode()

    t_step = {"deep": timed_loop(torch, deep_step, 50, flush, stream),
              "decode": timed_loop(torch, decode_step, reps, flush, stream)}
    t_attn = timed_loop(torch, attend, 50, flush, stream)
    t_attn_dec = timed_loop(torch, attend_decode, reps, flush, stream)
    # every top-k path forced on the same deep and decode scores (cold), and both select
    # forms back to back (warm)
    topk_paths = {}
    for name, pth, cs, sc_, nb_, ids_, ws_, act in (
            ("deep", None, case, scores, nb, ids, ws, case.active_blocks),
            ("decode", None, dcase, dscores, dnb, dids, dws, -1)):
        select_chained() if name == "deep" else decode_chained()
        res = {}
        for pth in (qsa.PATH_WARP, qsa.PATH_SAMPLE, qsa.PATH_REGISTER, qsa.PATH_SPLIT, qsa.PATH_RADIX):
            fn = (lambda p_=pth, c_=cs, s_=sc_, n_=nb_, i_=ids_, w_=ws_, a_=act:
                  qsa.block_topk(s_, n_, c_.k, i_, w_, active_blocks=a_, path=p_))
            try:
                fn()
            except qsa.QSAError:
                continue
            res[qsa.PATH_NAMES[pth]] = us_mean(timed_loop(torch, fn, 100, flush, stream))
        topk_paths[name] = res
    # device time per call with no host launch in between (one CUDA graph of calls back
    # to back): the top-k over 24 copies of the deep scores (200 MB, more than L2 holds,
    # so each call reads its rows from DRAM), the scorer, and both select forms
    select_chained()
    torch.cuda.synchronize()
    rot = [scores.clone() for _ in range(24)]
    graph_us = {
        "topk_deep_rotating_scores": graph_us_per_call(
            torch, [lambda r_=r_: qsa.block_topk(r_, nb, case.k, ids, ws, active_blocks=case.active_blocks)
                    for r_ in rot]),
        "scorer_deep": graph_us_per_call(torch, [score_only] * 20),
        "select_deep_chained": graph_us_per_call(torch, [select_chained] * 20),
        "select_deep_fused": graph_us_per_call(torch, [select_fused] * 20),
        "select_decode_chained": graph_us_per_call(torch, [decode_chained] * 20),
        "select_decode_fused": graph_us_per_call(torch, [decode_fused] * 20)}
    del rot
    clocks = sampler.stop()

    ms_main = max_over_ranks(statistics.mean(t_main), device=dev)
    if rank != 0:
        return 0

    # rules (a)-(c) on the timed workloads through the oracle, outside every timed region
    parity = None
    if not args.no_parity:
        select_chained()
        torch.cuda.synchronize()
        chained_ids = ids.cpu().numpy().copy()
        gpu_scores = scores.cpu().numpy()
        select()
        torch.cuda.synchronize()
        parity = {"deep": parity_report(case, gpu_scores, chained_ids, ids.cpu().numpy(), form)}
        decode_chained()
        torch.cuda.synchronize()
        dch = dids.cpu().numpy().copy()
        dsc = dscores.cpu().numpy()
        decode_fused()
        torch.cuda.synchronize()
        parity["decode"] = parity_report(dcase, dsc, dch, dids.cpu().numpy(), "fused")

    peaks, peak_src = load_peaks()
    us_main = job_us_per_call(ms_main, world)
    us_main_mean = us_mean(t_main)
    us_other = us_mean(t_other)
    us_score = us_mean(t_score)
    us_topk = us_mean(t_topk)
    flops = 2.0 * case.nq * case.n_heads * 128 * n
    topk_bytes = 4.0 * case.nq * n + 4.0 * case.nq * case.k + 4.0 * case.nq
    tflops = flops / (us_score * 1e-6) / 1e12
    gbs = topk_bytes / (us_topk * 1e-6) / 1e9
    scorer_roof = {"kernel": "scorer_tc_kernel<bf16, 16>", "bound": "tensor", "achieved": tflops,
                   "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                   "traffic": profiled_traffic("scorer"),
                   "per_launch": f"{flops:.4g} FLOP (2 x 256 q x 16 h x 128 x {n} blocks)",
                   "us_per_launch": us_score, "peak_source": f"{peak_src} bf16 burst (dense cuBLAS)"}
    topk_roof = {"kernel": f"topk ({qsa.PATH_NAMES[path]} path)", "bound": "hbm", "achieved": gbs,
                 "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                 "traffic": profiled_traffic("topk"), "per_launch": f"{topk_bytes:.4g} B",
                 "us_per_launch": us_topk, "peak_source": f"{peak_src} HBM copy"}
    # the same kernels' fractions by device time alone (graph replays, no launch or event
    # overhead per call; the top-k's rows come from DRAM, the scorer's inputs stay in L2)
    g_topk, g_score = graph_us["topk_deep_rotating_scores"], graph_us["scorer_deep"]
    topk_roof.update(us_per_launch_graph=g_topk,
                     frac_kernel=topk_bytes / (g_topk * 1e-6) / 1e9 / peaks["hbm_gbs"])
    scorer_roof.update(us_per_launch_graph=g_score,
                       frac_kernel=flops / (g_score * 1e-6) / 1e12 / peaks["bf16_tflops"])
    if form == "fused":
        # the fused scorer and its merge: the call's work is the contraction
        ftf = flops / (us_main_mean * 1e-6) / 1e12
        roof = {"kernel": "scorer_tc_kernel<bf16, 16, fused>", "bound": "tensor", "achieved": ftf,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": ftf / peaks["bf16_tflops"],
                "traffic": profiled_traffic("fused"),
                "per_launch": f"{flops:.4g} FLOP (2 x 256 q x 16 h x 128 x {n} blocks), scores kept on chip",
                "us_per_launch": us_main_mean, "peak_source": f"{peak_src} bf16 burst (dense cuBLAS)"}
    else:
        roof = scorer_roof if us_score >= us_topk else topk_roof
    dec_n = int(dcase.n_blocks[0])
    path_bytes = {"deep": topk_bytes, "decode": 4.0 * dcase.nq * dec_n + 4.0 * dcase.nq * dcase.k + 4.0 * dcase.nq}
    topk_path_table = {w_: {p_: {"us": u_, "gbs": path_bytes[w_] / (u_ * 1e-6) / 1e9,
                                 "frac": path_bytes[w_] / (u_ * 1e-6) / 1e9 / peaks["hbm_gbs"]}
                            for p_, u_ in d_.items()}
                       for w_, d_ in topk_paths.items()}
    dec_bytes = 256.0 * dec_n + 4096.0 * dcase.nq + 64.0 * dcase.nq + 8.0 * dcase.nq * dec_n + 4.0 * dcase.nq * dcase.k
    us_dec_f = us_mean(t_dec_f)
    us_dec_c = us_mean(t_dec_c)
    us_dec = min(us_dec_f, us_dec_c)
    us_e2e = statistics.mean(t_e2e) * 1e3
    attn = attention_report(acase, adcase, us_mean(t_attn), us_mean(t_attn_dec),
                            peaks, peak_src)
    # select then attend in one sequence: the attention launches as the top-k's
    # programmatic dependent (the sum of the two calls timed apart is beside it)
    attn["select_then_attend_us"] = {
        "deep": us_mean(t_step["deep"]),
        "deep_parts_sum": us_main_mean + attn["us_per_launch"],
        "decode": us_mean(t_step["decode"]),
        "decode_parts_sum": us_mean(t_dec_c) + attn["decode"]["us_per_call"]}
    p_us = {k_: us_mean(v_) for k_, v_ in t_prompt.items()}
    p_n = int(pcase.n_blocks[0])
    p_flops = 2.0 * pcase.nq * pcase.n_heads * 128 * p_n
    p_tf = p_flops / (p_us["scorer"] * 1e-6) / 1e12
    prompt = {"workload": pcase.name, "select_us": {"chained": p_us["chained"], "fused": p_us["fused"]},
              "scorer": {"kernel": "scorer_tc_kernel<bf16, 16>", "us_per_launch": p_us["scorer"],
                         "achieved": p_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": p_tf / peaks["bf16_tflops"], "per_launch": f"{p_flops:.4g} FLOP"}}
    e_us = {k_: us_mean(v_) for k_, v_ in t_e4m3.items()}
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    e_tf = flops / (e_us["scorer"] * 1e-6) / 1e12
    e4m3 = {"workload": ecase.name, "select_us": {"chained": e_us["chained"], "fused": e_us["fused"]},
            "scorer": {"kernel": "scorer_tc_kernel<e4m3, 16>", "bound": "tensor", "us_per_launch": e_us["scorer"],
                       "achieved": e_tf, "peak": fp8_peak, "unit": "TFLOP/s", "frac": e_tf / fp8_peak,
                       "peak_source": f"{peak_src} bf16 burst x 2 (the nominal fp8 / bf16 dense ratio, 4.5 / 2.25)",
                       "per_launch": f"{flops:.4g} FLOP"},
            "kblk_bytes": 128.0 * ecase.max_blocks}
    line = {
        "metric": METRIC, "value": us_main, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_main, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/kblk, U(0,1) w)",
        "config": dict(workload_config(case), select_form=form,
                       path=("fused select: a tcgen05 scorer that keeps its scores on chip and lists each CTA's "
                              "candidates, then one merge CTA per query as its programmatic dependent" if form == "fused" else
                             f"chained select: tcgen05 scorer, then the {qsa.PATH_NAMES[path]} top-k path "
                             "launched as its programmatic dependent")),
        "selections_per_s": case.nq * world / (ms_main * 1e-3),
        "roofline": roof,
        "forms_us_mean": {form: us_main_mean, ("chained" if form == "fused" else "fused"): us_other},
        "scorer": dict(scorer_roof, frac_of_bf16_peak=scorer_roof["frac"]),
        "topk": dict(topk_roof, path=qsa.PATH_NAMES[path], bytes=topk_bytes, l2="cold (flushed)"),
        "decode_3q_258K": {"us_per_call": us_dec, "form": "fused" if us_dec_f <= us_dec_c else "chained",
                           "fused_us": us_dec_f, "chained_us": us_dec_c,
                           "chained_topk_path": qsa.PATH_NAMES[dpath],
                           "gbs": dec_bytes / (us_dec * 1e-6) / 1e9,
                           "frac_of_hbm": dec_bytes / (us_dec * 1e-6) / 1e9 / peaks["hbm_gbs"]},
        "e2e": {"value": us_e2e, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "form": form},
        "selection_attention": attn,
        "e4m3_keys": e4m3,
        "prompt_256q_131K": prompt,
        "topk_paths_cold": topk_path_table,
        "graph_us_per_call": graph_us,
        "parity": parity,
        "gpu_launches": args.steps * (2 if form == "fused" else 1 + topk_launches),
        "clocks": clocks,
        "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"]},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(case, min(args.cpu_seconds, 6.0))
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true", help="skip the oracle parity report")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-sample-queries", type=int, default=8)
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="only run this many select calls per workload (for ncu); print nothing")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
