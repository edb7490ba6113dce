#!/usr/bin/env python
"""Benchmark of the routed multi-tenant LoRA delta on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one ``lora_delta_fused`` call (the whole hot path: routing, shrink,
expand + fold) on one decode batch of the "decode BGMV qkv" workload: 64 rows,
k_in 4096, output slices (4096, 1024, 1024), 16 adapter slots of rank 16, 10%
unrouted rows.  Inputs are seeded synthetic data already resident in HBM; each
step uses the next of C rotating copies of (pool, x, out, seq_slot) whose total
is more than twice the L2, so the adapter bytes come from HBM.  The K timed
steps are one CUDA graph, timed with CUDA events on the launching stream.

Rank 0 prints one JSON line.  With N > 1 (torchrun) every rank runs its own
batch with the pool replicated (rows are independent: no collective on the
data path), and the slowest rank's time is used.

``--impl reference`` times the CPU oracle (the plain C reference) on the same
workload, on this machine's host cores, rank 0 only.
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

METRIC = "LoRA-delta rows/s; BGMV HBM GB/s and SGMV TFLOP/s as % of GB300 roofline"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# DRAM bytes (read + write) of one launch of the decode step's kernel, from one
# ncu capture of that launch (dram__bytes_read.sum + dram__bytes_write.sum),
# with the hash of the sources it was taken on: reported only while they are
# unchanged, null otherwise.
DECODE_TRAFFIC = {"bytes": 10623232, "sources_sha256_16": "b9fab7ad425dee04"}
DECODE_SOURCES = ("lora_delta_gb300/csrc/bgmv.cuh", "lora_delta_gb300/csrc/bgmv_fused.cuh",
                  "lora_delta_gb300/csrc/common.cuh", "lora_delta_gb300/csrc/api.cu")


def decode_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    ok = h.hexdigest()[:16] == DECODE_TRAFFIC["sources_sha256_16"]
    return DECODE_TRAFFIC["bytes"] if ok else None


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        rows = []
        for ts, line in self.lines:
            if t0 is not None and (ts < t0 or ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl)
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------- the workloads --

def algorithmic_bytes(case, rows_mask=None):
    """HBM bytes the delta must move for one call: each routed slot's A and B
    once (at the padded rank), x of the routed rows, out read + write of the
    routed rows' columns."""
    import numpy as np
    seq = case.seq_slot if rows_mask is None else case.seq_slot[rows_mask]
    routed = (seq >= 0) & (seq < case.max_loras)
    # rows whose slot adapts no slice are untouched: they move nothing
    live = np.array([a is not None and any(a.adapted) for a in case.adapters] + [False])
    routed &= live[np.where(routed, seq, len(case.adapters))]
    slots = np.unique(seq[routed])
    n_routed = int(routed.sum())
    per_slot = 0
    for s in slots:
        ad = case.adapters[s]
        for j, w in enumerate(case.widths):
            if ad is not None and ad.adapted[j]:
                per_slot += case.max_rank * case.k_in * 2 + w * case.max_rank * 2
    cols = sum(case.widths)
    return per_slot + n_routed * case.k_in * 2 + n_routed * cols * 2 * 2


def algorithmic_flops(case):
    seq = case.seq_slot
    routed = int(((seq >= 0) & (seq < case.max_loras)).sum())
    S = len(case.widths)
    return routed * 2 * case.max_rank * (S * case.k_in + sum(case.widths))


def l2_bytes():
    import torch
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 126 * 1024 * 1024


def make_copies(ld, di, case, copies, device):
    """``copies`` independent device copies of (pool, x, out, seq_slot)."""
    import torch
    base = di.linear_to_device(case, device)
    out = []
    for c in range(copies):
        if c == 0:
            pool = base.pool
        else:
            pool = ld.LoraPool(case.k_in, case.widths, case.max_loras, case.max_rank,
                               device=device)
            for j in range(pool.S):
                pool.A[j].copy_(base.pool.A[j])
                pool.B[j].copy_(base.pool.B[j])
            pool.scale_table.copy_(base.pool.scale_table)
            L = case.max_loras
            a_host = [0] * (pool.S * L)
            b_host = [0] * (pool.S * L)
            at = base.pool.a_table.cpu().tolist()
            for j in range(pool.S):
                for s in range(L):
                    if at[j * L + s]:
                        a_host[j * L + s] = pool.A[j][s].data_ptr()
                        b_host[j * L + s] = pool.B[j][s].data_ptr()
            pool.a_table.copy_(torch.tensor(a_host, dtype=torch.int64))
            pool.b_table.copy_(torch.tensor(b_host, dtype=torch.int64))
        out.append(dict(pool=pool, x=base.x.clone(), out=base.out0.clone(),
                        seq=base.seq_slot.clone()))
    torch.cuda.synchronize(device)
    return out


def decode_config(case, world):
    """The workload of one step (the same dict on both arms)."""
    return {"workload": case.name, "rows_per_step": case.n, "k_in": case.k_in,
            "output_slices": list(case.widths), "max_loras": case.max_loras,
            "max_rank": case.max_rank, "unrouted_rows": int((case.seq_slot < 0).sum()),
            "parallelism": f"dp{world} (rows sharded, pool replicated)"}


def run_ours(args, rank, world):
    import numpy as np
    import torch

    import lora_delta_gb300 as ld
    from lora_delta_gb300 import device_inputs as di
    from lora_delta_gb300 import dist as ldist
    from lora_delta_gb300 import inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    ld.lib()
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()

    case = inputs.decode_qkv_case(seed=1235 + 1000 * rank)
    n = case.n
    per_copy = (case.max_loras * sum(case.max_rank * case.k_in * 2 + w * case.max_rank * 2
                                      for w in case.widths)
                + n * case.k_in * 2 + n * case.ld_out * 2 + n * 4)
    copies = max(2, int(np.ceil(2.2 * l2_bytes() / per_copy)))
    bufs = make_copies(ld, di, case, copies, device)
    stream = torch.cuda.Stream(device)
    K, W = args.steps, args.warmup

    def step(k):
        b = bufs[k % copies]
        return lambda: ld.lora_delta_fused(b["out"], b["x"], b["seq"], b["pool"])

    # warm-up: W eager steps (also the first use of every copy)
    with torch.cuda.stream(stream):
        for k in range(max(W, copies)):
            step(k)()
    torch.cuda.synchronize(device)

    # the K timed steps as one CUDA graph
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(K):
            step(k)()
    torch.cuda.synchronize(device)

    sampler = ClockSampler(local)
    sampler.start()
    # untimed pre-roll so that clocks settle and the sampler sees the load
    # (CUDAGraph.replay launches on the current stream: make it `stream`)
    t_pre = time.time()
    n_pre = 0
    with torch.cuda.stream(stream):
        while time.time() - t_pre < 0.4 or n_pre < 1:
            g.replay()
            torch.cuda.synchronize(device)
            n_pre += 1
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ldist.barrier()
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        g.replay()
        ev1.record(stream)
    torch.cuda.synchronize(device)
    t_wall1 = time.time()
    ldist.barrier()
    ms_total = ev0.elapsed_time(ev1)
    sampler.stop()
    clocks = sampler.summary(t_pre, t_wall1)
    ms_total = ldist.max_over_ranks(ms_total, device)
    ms_step = ms_total / K
    total_rows = ldist.sum_over_ranks(n * K, device)
    value = total_rows / (ms_total / 1e3)

    # roofline of the dominant (only) kernel of the step
    abytes = algorithmic_bytes(case)
    achieved = abytes / (ms_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "traffic": decode_traffic(), "peak_source": peak_src,
                "algorithmic_bytes_per_launch": abytes,
                "kernel": "bgmv_fused_kernel<16,LinearTables>"}

    # the data-movement floor of this launch shape: the same bytes, grid,
    # cluster size and programmatic dependent launch, no arithmetic
    floor = decode_floor(ld, bufs, copies, K, stream, device, abytes, hbm_peak, ms_step)

    # eager (no graph) timing of the same K steps, for context
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev2.record(stream)
        for k in range(K):
            step(k)()
        ev3.record(stream)
    torch.cuda.synchronize(device)
    eager_ms = ev2.elapsed_time(ev3) / K

    e2e = run_e2e(ld, di, case, bufs, copies, K, W, device)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init adapters)",
        "config": decode_config(case, world),
        "l2": f"{copies} rotating copies of pool/x/out/seq_slot "
              f"({copies * per_copy / 2**20:.0f} MiB > 2x L2)",
        "timing": "one CUDA graph of K steps, CUDA events on the launching stream",
        "roofline": roofline,
        "decode_floor": floor,
        "eager_ms_per_step": round(eager_ms, 6),
        "e2e": e2e,
        "gpu_launches": K,
        "clocks": clocks,
    }
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(case)
        if not args.no_extra:
            line["other_workloads"] = other_workloads(ld, di, inputs, device, hbm_peak,
                                                      bf16_peak, peak_src)
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_floor(ld, bufs, copies, K, stream, device, abytes, hbm_peak, ms_step):
    """K steps of lora_delta_fused_floor (the fused call's bytes and launch plan,
    no arithmetic) as one CUDA graph on the same rotating buffers."""
    import torch
    step = lambda k: ld.lora_delta_fused_floor(bufs[k % copies]["out"], bufs[k % copies]["x"],
                                               bufs[k % copies]["seq"], bufs[k % copies]["pool"])
    with torch.cuda.stream(stream):
        for k in range(copies):
            step(k)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(K):
            step(k)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / K
    gbs = abytes / (ms / 1e3) / 1e9
    return {"ms_per_step": round(ms, 6), "GB_per_s": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_peak, 4),
            "kernel_frac_of_floor": round(ms / ms_step, 4),
            "what": "lora_delta_fused_floor: the decode step's bytes (A/B shares, x and out "
                    "rows, out written back) with the same grid, cluster size, shared-memory "
                    "plan and programmatic dependent launch, no arithmetic; K steps in one "
                    "CUDA graph on the same rotating buffers"}


def run_e2e(ld, di, case, bufs, copies, K, W, device):
    """The same metric through the public API with host buffers: per step one
    pinned host->device copy of (x, out, seq_slot), the call, and one
    device->host copy of the updated out."""
    import torch
    n = case.n
    x_b, o_b, s_b = n * case.k_in * 2, n * case.ld_out * 2, n * 4
    align = lambda v: (v + 255) // 256 * 256
    total = align(x_b) + align(o_b) + align(s_b)
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    host[:x_b].copy_(bufs[0]["x"].view(torch.uint8).view(-1).cpu())
    host[align(x_b):align(x_b) + o_b].copy_(bufs[0]["out"].view(torch.uint8).view(-1).cpu())
    host[align(x_b) + align(o_b):align(x_b) + align(o_b) + s_b].copy_(
        bufs[0]["seq"].view(torch.uint8).view(-1).cpu())
    host_out = torch.empty(o_b, dtype=torch.uint8).pin_memory()
    dev = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(copies)]
    views = []
    for d in dev:
        x = d[:x_b].view(torch.bfloat16).view(n, case.k_in)
        o = d[align(x_b):align(x_b) + o_b].view(torch.bfloat16).view(n, case.ld_out)
        s = d[align(x_b) + align(o_b):align(x_b) + align(o_b) + s_b].view(torch.int32)
        views.append((d, x, o, s))
    stream = torch.cuda.Stream(device)
    ws = torch.empty(ld.lora_workspace_size(n, len(case.widths), case.max_rank, case.max_loras),
                     dtype=torch.uint8, device=device)

    def step(k):
        d, x, o, s = views[k % copies]
        d.copy_(host, non_blocking=True)
        ld.lora_delta_fused(o, x, s, bufs[k % copies]["pool"], workspace=ws)
        host_out.copy_(d[align(x_b):align(x_b) + o_b], non_blocking=True)

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / K

    with torch.cuda.stream(stream):
        for k in range(max(W, 3)):
            step(k)
    torch.cuda.synchronize(device)
    eager_ms = timed(lambda: [step(k) for k in range(K)])
    # The K steps as one CUDA graph, pipelined the way a serving loop double
    # buffers: step k's host->device copy, call and device->host copy run on
    # three streams in that order, so step k + 1's upload and step k - 1's
    # read-back overlap step k's call.  A device buffer is refilled only after
    # the read-back of the step that used it before.  Every copy stays in the
    # timed region.
    host_outs = [torch.empty(o_b, dtype=torch.uint8).pin_memory() for _ in range(copies)]
    s_up, s_call, s_down = (torch.cuda.Stream(device) for _ in range(3))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fork = torch.cuda.Event()
        fork.record(stream)
        for st in (s_up, s_call, s_down):
            st.wait_event(fork)
        down_done = [None] * K
        for k in range(K):
            d, x, o, s = views[k % copies]
            with torch.cuda.stream(s_up):
                if k >= copies:
                    s_up.wait_event(down_done[k - copies])
                d.copy_(host, non_blocking=True)
                up = torch.cuda.Event()
                up.record(s_up)
            with torch.cuda.stream(s_call):
                s_call.wait_event(up)
                ld.lora_delta_fused(o, x, s, bufs[k % copies]["pool"], workspace=ws)
                called = torch.cuda.Event()
                called.record(s_call)
            with torch.cuda.stream(s_down):
                s_down.wait_event(called)
                host_outs[k % copies].copy_(d[align(x_b):align(x_b) + o_b], non_blocking=True)
                down_done[k] = torch.cuda.Event()
                down_done[k].record(s_down)
        for st in (s_up, s_call, s_down):
            stream.wait_stream(st)
    torch.cuda.synchronize(device)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(device)
    ms = timed(g.replay)
    return {"value": round(n / (ms / 1e3), 1), "unit": "rows/s", "ms_per_step": round(ms, 6),
            "h2d_bytes_per_step": total, "d2h_bytes_per_step": o_b,
            "path": "one CUDA graph of the K steps, each: pinned host -> device copy of "
                    "(x, out, seq_slot), lora_delta_fused, device -> pinned host copy of out; "
                    "steps pipelined over three streams (upload / call / read-back)",
            "eager": {"value": round(n / (eager_ms / 1e3), 1), "ms_per_step": round(eager_ms, 6),
                      "path": "the same steps one after another on one stream, from Python"}}


def cpu_baseline(case, budget_s: float = 10.0):
    """The CPU oracle as it stands, on this machine's host cores."""
    import numpy as np

    import oracle
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, case.max_loras,
                             case.max_rank)
    out = case.out0.copy()
    oracle.delta(out, case.x, case.seq_slot, pool)  # untimed first call
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.delta(out, case.x, case.seq_slot, pool)
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= 2000:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": round(reps * case.n / dt, 1), "unit": "rows/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} repetitions of the full {case.n}-row decode batch "
                      f"({dt:.1f} s, OpenMP over rows, {cores} threads)"}


def rotation(set_bytes: int) -> int:
    """Copies of a workload's buffers whose total passes twice the L2 (at least 1)."""
    import math
    return max(1, math.ceil(2.2 * l2_bytes() / max(1, set_bytes)))


def other_workloads(ld, di, inputs, device, hbm_peak, bf16_peak, peak_src, only=None, reps=20,
                    warm=3):
    """The other workloads of the path, each timed on its own (not the headline).

    Each is timed with CUDA events over ``reps`` calls on one stream after
    ``warm`` warm-up calls.  Where one call's buffers are smaller than twice the
    L2, the calls rotate over enough independent copies of all of them (inputs,
    adapters, outputs) that the total passes twice the L2, so the bytes come from
    HBM; the copy count goes into each result."""
    import numpy as np
    import torch
    res = {}
    stream = torch.cuda.Stream(device)
    rep_default, warm_default = max(20, reps), max(3, warm)

    def timed(fns, reps=rep_default, warm=warm_default):
        fns = fns if isinstance(fns, (list, tuple)) else [fns]
        with torch.cuda.stream(stream):
            for i in range(max(warm, len(fns))):
                fns[i % len(fns)]()
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(reps):
                fns[i % len(fns)]()
            e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / reps

    # prefill SGMV gate_up (8192 rows)
    if only in (None, "prefill"):
        _prefill(ld, di, inputs, device, hbm_peak, bf16_peak, timed, res)
    if only in (None, "skewed"):
        _skewed(ld, di, inputs, device, hbm_peak, timed, res)
    if only in (None, "fold"):
        _fold(ld, di, inputs, device, hbm_peak, timed, res)
    if only in (None, "moe"):
        _moe(ld, di, inputs, device, hbm_peak, timed, res)
    if only in (None, "moe_inplace"):
        _moe_inplace(ld, di, inputs, device, hbm_peak, timed, res)
    res["peak_source"] = peak_src
    return res


def _prefill(ld, di, inputs, device, hbm_peak, bf16_peak, timed, res):
    import torch
    case = inputs.prefill_gate_up_case()
    ab, fl = algorithmic_bytes(case), algorithmic_flops(case)
    ds = [di.linear_to_device(case, device) for _ in range(rotation(ab))]
    ws = torch.empty(ld.lora_workspace_size(case.n, len(case.widths), case.max_rank,
                                         case.max_loras), dtype=torch.uint8, device=device)
    ms = timed([lambda d=d: ld.lora_delta_fused(d.out0, d.x, d.seq_slot, d.pool, workspace=ws)
                for d in ds])
    gbs, tfs = ab / (ms / 1e3) / 1e9, fl / (ms / 1e3) / 1e12
    attain = min(bf16_peak, fl / ab * hbm_peak / 1e3)
    res["prefill_gate_up"] = {"rows_per_s": round(case.n / (ms / 1e3), 1), "ms": round(ms, 4),
                              "GB_per_s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                              "TFLOP_per_s": round(tfs, 2),
                              "tensor_frac": round(tfs / bf16_peak, 5),
                              "attainable_TFLOP_per_s": round(attain, 1),
                              "roofline_frac": round(tfs / attain, 4),
                              "launches_per_call": 5, "copies": len(ds)}
    del ds, ws
    torch.cuda.empty_cache()


def _skewed(ld, di, inputs, device, hbm_peak, timed, res):
    import torch
    # skewed many-adapter decode: both projections per step
    c1, c2 = inputs.skewed_case(0), inputs.skewed_case(1)
    ab = algorithmic_bytes(c1) + algorithmic_bytes(c2)
    ds = [(di.linear_to_device(c1, device), di.linear_to_device(c2, device))
          for _ in range(rotation(ab))]
    ws = torch.empty(max(ld.lora_workspace_size(c.n, 1, c.max_rank, c.max_loras) for c in (c1, c2)),
                     dtype=torch.uint8, device=device)
    ms = timed([lambda d1=d1, d2=d2: (
        ld.lora_delta_fused(d1.out0, d1.x, d1.seq_slot, d1.pool, workspace=ws),
        ld.lora_delta_fused(d2.out0, d2.x, d2.seq_slot, d2.pool, workspace=ws)) for d1, d2 in ds])
    res["skewed_decode"] = {"rows_per_s": round(c1.n / (ms / 1e3), 1), "ms": round(ms, 4),
                            "GB_per_s": round(ab / (ms / 1e3) / 1e9, 1),
                            "hbm_frac": round(ab / (ms / 1e3) / 1e9 / hbm_peak, 4),
                            "launches_per_call": 10, "copies": len(ds)}
    del ds, ws
    torch.cuda.empty_cache()


def _fold(ld, di, inputs, device, hbm_peak, timed, res):
    import torch
    # expert-sorted MoE fold (w13): 2048 tokens x top-8 of 64 experts, one
    # adapter per expert (10% unadapted), rows grouped by device offsets
    case, offsets = inputs.expert_sorted_case()
    ab = algorithmic_bytes(case)
    ds = [di.linear_to_device(case, device) for _ in range(rotation(ab))]
    off = torch.from_numpy(offsets).to(device)
    ws = torch.empty(ld.lora_workspace_size(case.n, 1, case.max_rank, case.max_loras),
                     dtype=torch.uint8, device=device)
    ms = timed([lambda d=d: ld.lora_delta_segmented(d.out0, d.x, off, d.pool, workspace=ws)
                for d in ds])
    gbs = ab / (ms / 1e3) / 1e9
    res["moe_expert_fold_w13"] = {"rows_per_s": round(case.n / (ms / 1e3), 1), "ms": round(ms, 4),
                                  "GB_per_s": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                                  "launches_per_call": 5, "copies": len(ds)}
    del ds, ws
    torch.cuda.empty_cache()


def _moe_keys(case):
    import numpy as np
    valid = case.lora_ids >= 0
    return valid, {(int(l), int(e)) for t in np.flatnonzero(valid)
                   for l, e in zip([case.lora_ids[t]] * case.top_k, case.topk_ids[t])}


def _moe(ld, di, inputs, device, hbm_peak, timed, res):
    import torch
    # MoE FC1 (regular and shared-A / fused-B)
    for shared in (False, True):
        mc = inputs.moe_case(shared_a=shared)
        valid, keys = _moe_keys(mc)
        pairs = int(valid.sum()) * mc.top_k
        n_a = 1 if shared else 2
        bank = len(keys) * (n_a * mc.rank * mc.H * 2 + 2 * mc.I * mc.rank * 2)
        ab = bank + mc.T * mc.top_k * 2 * mc.I * 2 + int(valid.sum()) * mc.H * 2
        sets = []
        for _ in range(rotation(ab)):
            dm = di.moe_to_device(mc, device)
            out = torch.empty(mc.T, mc.top_k, 2 * mc.I, dtype=torch.bfloat16, device=device)
            sets.append((dm, out))
        ws = torch.empty(ld.lora_moe_workspace_size(mc.T, mc.top_k, mc.E, mc.L, mc.rank, shared),
                         dtype=torch.uint8, device=device)
        ms = timed([lambda dm=dm, out=out: ld.lora_moe_fc1_delta(
            out, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b, shared, dm.topk_ids,
            dm.lora_ids, mc.E, mc.I, mc.rank, mc.L, mc.scale, workspace=ws) for dm, out in sets])
        res["moe_fc1_" + ("shared" if shared else "regular")] = {
            "pairs_per_s": round(mc.T * mc.top_k / (ms / 1e3), 1), "ms": round(ms, 4),
            "routed_pairs": pairs, "GB_per_s": round(ab / (ms / 1e3) / 1e9, 1),
            "hbm_frac": round(ab / (ms / 1e3) / 1e9 / hbm_peak, 4), "launches_per_call": 3,
            "copies": len(sets)}
        del sets, ws
        torch.cuda.empty_cache()


def _moe_inplace(ld, di, inputs, device, hbm_peak, timed, res):
    import torch
    # in-place MoE deltas on either side of the activation, FC1's routing:
    # w13 (gate/up, regular banks) into intermediate_cache1, w2 (down, with
    # routing weights) into intermediate_cache3 from per-pair activations
    mc = inputs.moe_case()
    c2 = inputs.moe_w2_case()
    for name, case in (("moe_w13_inplace", mc), ("moe_w2_inplace_weighted", c2)):
        valid, keys = _moe_keys(case)
        pairs = int(valid.sum()) * case.top_k
        if name == "moe_w13_inplace":
            bank = len(keys) * (2 * mc.rank * mc.H * 2 + 2 * mc.I * mc.rank * 2)
            ab = bank + pairs * 2 * mc.I * 2 * 2 + int(valid.sum()) * mc.H * 2
            y0 = inputs.moe_y0(mc.seed, (mc.T, mc.top_k, 2 * mc.I))
            ws = torch.empty(ld.lora_moe_workspace_size(mc.T, mc.top_k, mc.E, mc.L, mc.rank,
                                                        False), dtype=torch.uint8, device=device)
            fns = []
            for _ in range(rotation(ab)):
                dm, y = di.moe_to_device(case, device), di.bf16(y0, device)
                fns.append(lambda dm=dm, y=y: ld.lora_moe_w13_delta(
                    y, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b, False, dm.topk_ids,
                    dm.lora_ids, mc.E, mc.I, mc.rank, mc.L, mc.scale, workspace=ws))
        else:
            bank = len(keys) * (case.rank * case.I * 2 + case.H * case.rank * 2)
            ab = bank + pairs * case.H * 2 * 2 + pairs * case.I * 2
            ws = torch.empty(ld.lora_moe_workspace_size(case.T, case.top_k, case.E, case.L,
                                                        case.rank, True),
                             dtype=torch.uint8, device=device)
            fns = []
            for _ in range(rotation(ab)):
                dm, y = di.moe_to_device(case, device), di.bf16(case.y0, device)
                wts = torch.from_numpy(case.topk_weights).to(device)
                fns.append(lambda dm=dm, y=y, wts=wts: ld.lora_moe_w2_delta(
                    y, dm.x, dm.w_ptr_a, dm.stride_a, dm.w_ptr_b, dm.stride_b, dm.topk_ids,
                    dm.lora_ids, case.E, case.H, case.rank, case.L, case.scale,
                    topk_weights=wts, workspace=ws))
        ms = timed(fns)
        res[name] = {"pairs_per_s": round(case.T * case.top_k / (ms / 1e3), 1),
                     "ms": round(ms, 4), "routed_pairs": pairs,
                     "GB_per_s": round(ab / (ms / 1e3) / 1e9, 1),
                     "hbm_frac": round(ab / (ms / 1e3) / 1e9 / hbm_peak, 4),
                     "launches_per_call": 3, "copies": len(fns)}
        del fns, ws
        torch.cuda.empty_cache()


# ---------------------------------------------------------- reference arm --

def run_reference(args, rank, world):
    """The CPU oracle on the same workload (rank 0 only), bounded per step."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from lora_delta_gb300 import inputs
    case = inputs.decode_qkv_case()
    pool = oracle.build_pool(case.adapters, case.k_in, case.widths, case.max_loras,
                             case.max_rank)
    out = case.out0.copy()
    t0 = time.perf_counter()
    oracle.delta(out, case.x, case.seq_slot, pool)
    t_full = time.perf_counter() - t0
    K, W = args.steps, args.warmup
    budget = 60.0
    rows = int(np.clip(case.n * budget / max(1e-9, (K + W) * t_full), 1, case.n))
    x, seq, o = case.x[:rows].copy(), case.seq_slot[:rows].copy(), case.out0[:rows].copy()
    for _ in range(W):
        oracle.delta(o, x, seq, pool)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle.delta(o, x, seq, pool)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    value = rows * K / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "rows/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(dt / K * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; random-init adapters)",
            "config": decode_config(case, world),
            "cpu_baseline": {"value": round(value, 1), "unit": "rows/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"first {rows} rows of the {case.n}-row decode batch "
                                       f"per step ({K} steps after {W} warm-up steps)"},
            "e2e": {"value": round(value, 1), "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (prefill, skewed, MoE)")
    ap.add_argument("--only", choices=["prefill", "skewed", "moe", "fold", "moe_inplace"], default=None,
                    help="time one of the other workloads alone and print its numbers "
                         "(for profiling captures; not the benchmark line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from lora_delta_gb300 import dist as ldist
    rank, world = ldist.init()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.only:
        import torch
        import lora_delta_gb300 as ld
        from lora_delta_gb300 import device_inputs as di
        from lora_delta_gb300 import inputs
        device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(device)
        hbm_peak, bf16_peak, _, peak_src = load_peaks()
        res = other_workloads(ld, di, inputs, device, hbm_peak, bf16_peak, peak_src,
                              only=args.only, reps=args.steps, warm=args.warmup)
        print(json.dumps(res), flush=True)
    else:
        run_ours(args, rank, world)


if __name__ == "__main__":
    main()
