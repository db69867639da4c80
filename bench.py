"""Benchmark: GQA decode KV-read GB/s (% of GB300 HBM peak) and us/call.

One step = one full pass of the decode hot path (stage 1 split-KV kernel and
stage 2 log-sum-exp combine, one prepared launch) over one batch of synthetic
inputs already resident in HBM; the K steps run back to back between two
events.  The split kernel's own duration (the roofline's) comes from a second
loop of K launches of stage 1 alone, each bracketed by events.  The headline workload is the long-context bf16 case
(batch 8, 32 q / 8 KV heads, head_dim 128, capacity = length = 131072: 4.3 GB
of KV per step, far larger than the 129 MB L2, so no flush is needed between
steps).  Every workload's us/call and GB/s are reported in ``per_config``
(cold L2: a 512 MB buffer is written and a 1 GB one read before each timed
call, so the L2 holds none of the inputs and no dirty lines).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4]
  python bench.py --impl reference ...   # the FP64 CPU oracle, same metric
  python bench.py --sweep                # + the automatic plan over SWEEP_SHAPES, cold
  python bench.py --read-ceiling         # + the read rate of the same data movement without arithmetic

GB/s counts algorithmic bytes: sum_b len_b x (4096 B fp16/bf16 | 2048 B e4m3)
of K+V, plus q, out and the lengths; workspace traffic is not counted.
With N > 1 (torchrun) every rank runs its own replica of the workload on its
own GPU (the work items are independent; there is no data-path collective),
the step time is the max over ranks and ``value`` sums all ranks' bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GQA decode KV-read GB/s (% of GB300 HBM peak) and µs/call per config"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "split_kv_traffic.json")
KERNEL_SOURCES = ["gqa_decode_attention_sm_gb300/csrc/kernels/common.cuh",
                  "gqa_decode_attention_sm_gb300/csrc/kernels/split_kv_mma.cuh"]


# ------------------------------------------------------------------ helpers


def code_tokens(text: str) -> str:
    """C++ source with comments removed and whitespace collapsed (string and
    character literals kept): what the compiler sees, so that a comment edit
    leaves the hash below, and the traffic capture keyed to it, in place."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the split kernel's code (comments and layout ignored)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def traffic_per_launch(workload_index: int):
    """DRAM bytes per split-kernel launch of this workload from the committed
    ncu summary, and how they were obtained, if the summary was taken on the
    current kernel source; else (None, None).  The capture may be of a
    smaller case of the same kernel (one batch row), scaled to the full
    workload by the units processed; the summary states the factor."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, None
    if d.get("source_hash") != kernel_source_hash() or d.get("workload") != workload_index:
        return None, None
    return d.get("dram_bytes_per_launch"), d.get("note")


def bytes_per_token(kv_dtype: str) -> int:
    """KV bytes per (token, batch row), all 8 KV heads, K and V."""
    if kv_dtype == "e4m3":
        return 2048
    if kv_dtype == "i8":  # int8 codes plus one bf16 scale per (plane, KV head) row
        return 2048 + 2 * 8 * 2
    return 4096


def algorithmic_bytes(w, lens_list) -> int:
    """KV bytes below the lengths, plus q and out (q_len query tokens each) and the lengths."""
    return sum(lens_list) * bytes_per_token(w.kv_dtype) + 2 * w.batch * w.q_len * 32 * 128 * 2 + 4 * w.batch


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (read-only)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout: float = 10.0):
        """Block until nvidia-smi has printed its first sample (or timeout):
        its start-up (NVML initialisation, over a second on a fresh machine)
        must not overlap a timed region."""
        t_end = time.time() + timeout
        while self.proc is not None and not self.samples and time.time() < t_end:
            if self.proc.poll() is not None:
                break
            time.sleep(0.02)
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = [s for t, s in self.samples if t0 <= t <= t1]
        window = "timed region"
        if len(rows) < 3:  # a short timed region: widen to the samples around it
            rows = [s for t, s in self.samples if t0 - 1.0 <= t <= t1 + 1.0]
            window = "timed region +/- 1 s"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "window": window,
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                                   default=None)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------- CPU baseline


def host_batch_row(t, b):
    """Bit patterns of batch row b (q, kv, length) copied to the host."""
    from gqa_decode_attention_sm_gb300.inputs import bits
    return bits(t["q"][b:b + 1]), bits(t["kv"][b:b + 1]), t["lens"][b:b + 1].cpu().numpy()


def oracle_rows(t, host, rows, threads):
    """Time the oracle on query-head `rows` of one host batch row.

    Returns (seconds, KV bytes those rows stand for: len x bytes_per_token / 32
    per row, the same accounting as the GPU metric)."""
    import oracle
    w = t["workload"]
    fmt = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3}
    qb, kvb, lens = host
    t0 = time.perf_counter()
    oracle.gqa_decode(qb, fmt[w.q_dtype], kvb, fmt[w.kv_dtype], lens, q_scale=t["q_scale"],
                      k_scale=t["k_scale"], v_scale=t["v_scale"], rows=rows, threads=threads)
    secs = time.perf_counter() - t0
    per_token = 2048 if w.kv_dtype == "e4m3" else 4096
    return secs, int(lens[0]) * per_token * len(rows) // 32


# ------------------------------------------------------------------- arms


def run_reference(args):
    """The oracle as it stands, timed on the host cores (the reference arm)."""
    import oracle
    from gqa_decode_attention_sm_gb300 import inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    oracle.build()
    w = inputs.WORKLOADS[args.workload]
    # one batch row of the workload, generated on the CPU with the same recipe
    t = inputs.make(inputs.with_(w, batch=1), "cpu")
    host = host_batch_row(t, 0)
    threads = oracle.default_threads()
    rows = list(range(min(32, threads)))  # one query-head row per core per step
    times, nb = [], 0
    for i in range(args.warmup + args.steps):
        secs, nb = oracle_rows(t, host, rows, threads)
        if i >= args.warmup:
            times.append(secs)
    mean = sum(times) / len(times)
    gbs = nb / mean / 1e9
    sample = (f"{len(rows)} query-head rows (length {int(host[2][0])}) of one batch row of "
              f"'{w.name}' per step, FP64, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * mean, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "capacity": w.capacity,
                       "kv_dtype": w.kv_dtype, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def near_host_cpus(dev):
    """The group of this process's CPUs whose freshly pinned host memory the
    GPU reads fastest.  Pinned pages land on the NUMA node of the CPU that
    first touches them, and a virtual machine may report one node for CPUs
    that sit on different sockets (on one GB300 machine: 211 GB/s host-to-device
    from 1 GiB buffers pinned on CPUs 0-7, 88 GB/s from CPUs 8-15; 64 MiB
    buffers copied at full rate from either).  Tries each half of the allowed
    CPUs with a 1 GiB buffer; returns (cpus, GB/s per group)."""
    import torch
    allowed = sorted(os.sched_getaffinity(0))
    if len(allowed) < 2:
        return set(allowed), {}
    half = len(allowed) // 2
    groups = [set(allowed[:half]), set(allowed[half:])]
    rates = {}
    try:
        for grp in groups:
            os.sched_setaffinity(0, grp)
            h = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
            h.fill_(1)
            d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
            d.copy_(h, non_blocking=True)
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(4):
                d.copy_(h, non_blocking=True)
            b.record()
            torch.cuda.synchronize(dev)
            rates[f"{min(grp)}-{max(grp)}"] = round(4 * (1 << 30) / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
            del h, d
    finally:
        os.sched_setaffinity(0, set(allowed))
    best = max(range(len(groups)), key=lambda i: list(rates.values())[i])
    return groups[best], rates


def call_samples(fn, n, flush=None, stream=None):
    """us of `fn` on each of n calls, each bracketed by CUDA events (flush outside)."""
    import torch
    res = []
    for _ in range(n):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        res.append(a.elapsed_time(b) * 1e3)
    return sorted(res)


def time_calls(fn, n, flush=None, stream=None):
    """Median us of `fn` over n calls, each bracketed by CUDA events (flush outside)."""
    res = call_samples(fn, n, flush, stream)
    return res[len(res) // 2]


def timer_resolution_us(samples):
    """(The event timer's resolution as seen in the samples: the smallest gap
    between two distinct values; the share of samples equal to the median).
    The timer resolves 32 ns, but a cold call's event interval on this GPU
    mostly lands on whole multiples of 2.048 us (most samples of the small
    workloads are exactly 8.192 or 10.24 us), so their medians cannot show
    changes below that step: cold_graph_us measures those calls instead."""
    vals = sorted(set(round(x, 4) for x in samples))
    gaps = [round(b - a, 3) for a, b in zip(vals, vals[1:]) if b - a > 1e-3]
    med = sorted(samples)[len(samples) // 2]
    at_median = sum(1 for x in samples if abs(x - med) < 1e-4) / len(samples)
    return (min(gaps) if gaps else None), round(at_median, 3)


def cold_graph_us(fn, flush, calls=40, reps=7):
    """us per cold call below the event timer's step: one CUDA graph of
    `calls` x (flush, fn) and one of `calls` x flush, each replayed `reps`
    times between two events; the median difference over `calls`.  The
    calls run as a graph does (no launch from the host between them)."""
    import torch
    graphs = []
    for with_call in (True, False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                flush()
                if with_call:
                    fn()
        graphs.append(g)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    times = {True: [], False: []}
    for _ in range(reps):
        for g, key in zip(graphs, (True, False)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            b.synchronize()
            times[key].append(a.elapsed_time(b) * 1e3)
    med = lambda v: sorted(v)[len(v) // 2]  # noqa: E731
    return (med(times[True]) - med(times[False])) / calls


def sdpa_context(t, w, n, flush):
    """Context only: torch SDPA (enable_gqa=True, default backend) on the same
    GPU inputs, K and V copied out contiguously beforehand (untimed); ragged
    lengths become a boolean mask over the capacity."""
    import math
    import torch
    F = torch.nn.functional
    q = t["q"].unsqueeze(2)  # [B, 32, 1, 128]
    k = t["kv"][:, 0].contiguous()  # [B, 8, C, 128]
    v = t["kv"][:, 1].contiguous()
    mask = None
    if not (w.len_lo == w.len_hi == w.capacity):
        pos = torch.arange(w.capacity, device=q.device)
        mask = (pos[None, :] < t["lens"][:, None].long())[:, None, None, :]
    scale = t["q_scale"] / math.sqrt(128.0)

    def fn():
        F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale, enable_gqa=True)

    try:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        us = time_calls(fn, n, flush=flush)
    except Exception as e:  # an SDPA backend without this shape or dtype
        return {"unavailable": f"{type(e).__name__}: {str(e)[:120]}"}
    row = {"us_per_call": round(us, 2),
           "note": "torch SDPA, enable_gqa=True, default backend, contiguous K/V copies; context only"}
    if mask is not None:
        row["note"] += "; boolean mask over the capacity (slots past a length may hold NaN: timing only)"
    return row


def oracle_config(t, w, nbytes, reps):
    """The oracle (all host cores) on a sample of the workload: every batch row
    for small batches, else the first few (all 32 query heads each); CPU GB/s
    and the µs a whole call would take at that rate."""
    import oracle
    threads = oracle.default_threads()
    rows_b = w.batch if w.batch * w.capacity <= 32 * 8192 else (1 if w.index == 4 else 4)
    hosts = [host_batch_row(t, b) for b in range(rows_b)]
    best = None
    for _ in range(reps):
        secs = sb = 0
        for host in hosts:
            s_, b_ = oracle_rows(t, host, list(range(32)), threads)
            secs, sb = secs + s_, sb + b_
        best = secs if best is None else min(best, secs)
    gbs = sb / best / 1e9
    return {"GBps": round(gbs, 3), "us_per_call": round(nbytes / gbs / 1e3, 1), "cores": threads,
            "sample": f"{rows_b} of {w.batch} batch rows, best of {reps}" + ("" if rows_b == w.batch else
                                                                             "; us_per_call scaled by bytes")}


L2_COLD = "cold (512 MB written, then 1 GB read, before each call)"


def make_cold_flush(dev):
    """The flush run before every cold call."""
    import torch
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean_buf = torch.ones(256 << 20, dtype=torch.float32, device=dev)  # 1 GB

    def flush():
        # Write a buffer larger than L2 (cold for the inputs), then read another
        # one so the L2 holds clean lines: the timed call should not pay for
        # writing back the flush's dirty lines.  The read is 1 GB (8x L2): after
        # a 256 MB read some dirty lines were still resident, and the timed
        # call paid for writing them back (per-CTA timelines on GB300: a wider
        # tail, +6 us on workload 3, +13 us on workload 4; 512 MB or more, or no
        # write at all, removed it).
        flush_buf.fill_(1)
        clean_buf.max()

    return flush


# Shapes away from the five workloads, for the automatic plan (split count,
# balanced schedule or one piece per CTA, cluster merge): (KV format, batch,
# capacity).  Each runs with every length = capacity and, from batch 8 on,
# with lengths U[capacity / 4, capacity].
SWEEP_SHAPES = (
    ("bf16", 1, 4096), ("bf16", 1, 32768), ("bf16", 4, 16384), ("bf16", 8, 4096), ("bf16", 8, 32768),
    ("bf16", 64, 4096), ("bf16", 64, 32768), ("bf16", 256, 4096), ("bf16", 16, 131072), ("bf16", 1024, 1024),
    ("bf16", 4, 8192), ("e4m3", 1, 32768), ("e4m3", 8, 4096), ("e4m3", 8, 8192), ("e4m3", 16, 32768),
    ("e4m3", 128, 8192), ("e4m3", 256, 16384), ("e4m3", 4, 262144), ("i8", 1, 32768), ("i8", 8, 4096),
    ("i8", 16, 32768), ("i8", 128, 8192),
)


def planner_sweep(dev, peak, gq, inputs, quick=False):
    """Cold us per call and the fraction of the peak over SWEEP_SHAPES, each
    through prepare/launch with the automatic split count."""
    import torch
    from gqa_decode_attention_sm_gb300 import api as gapi
    flush = make_cold_flush(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rows = []
    for n, (kv, B, C) in enumerate(SWEEP_SHAPES):
        for ragged in ((False, True) if B >= 8 else (False,)):
            w = inputs.custom(B, C, C // 4 if ragged else C, C, kv_dtype=kv, kv_std=2.0 if kv == "e4m3" else 1.0,
                              index=700 + n)
            t = inputs.make(w, dev)
            out = torch.empty_like(t["q"])
            fp8 = kv == "e4m3"
            tensors = {"Q": t["q"], "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]}
            if t["kv_scales"] is not None:
                tensors["KV_SCALES"] = t["kv_scales"]
            p = gq.prepare(tensors, q_scale=t["q_scale"], k_scale=t["k_scale"] if fp8 else None,
                           v_scale=t["v_scale"] if fp8 else None)
            nbytes = algorithmic_bytes(w, t["lens"].cpu().tolist())
            for _ in range(3):
                gq.launch(p)
            torch.cuda.synchronize()
            us = time_calls(lambda: gq.launch(p), 5 if quick else 20, flush=flush)
            timing = "events"
            if us < 100.0:  # a few event steps (2.048 us each): the difference of two CUDA graphs instead
                us = cold_graph_us(lambda: gq.launch(p), flush, calls=10 if quick else 40, reps=3 if quick else 7)
                timing = "graph difference"
            rows.append({"timing": timing, "kv": kv, "batch": B, "capacity": C, "lengths": f"U[{C // 4},{C}]" if ragged else "capacity",
                         "splits": p.num_splits, "kernels": gapi.launch_count(B, C, p.kv_format, 1, p.num_splits, sms),
                         "us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                         "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "alg_bytes": nbytes})
            del t, out, p, tensors
            torch.cuda.empty_cache()
    return rows


def warm_graph_us(fn, calls=20, reps=10):
    """us per call of `fn` with warm L2, launched from one CUDA graph of
    `calls` back-to-back calls (median over `reps` replays)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    return time_calls(g.replay, reps) / calls


def append_rows(dev, gq, inputs, flush, quick=False):
    """The step before decode (RMS norm + RoPE of each request's new token,
    its K and V written into the cache at a device-side slot), alone and as
    a serving step with the decode that follows, both launched from one CUDA
    graph; over workloads 4 and 5.  Each call rewrites the last slot below
    the length, so every call writes the same bytes."""
    import torch
    rows = {}
    for key, w in (("4-append-decode", inputs.WORKLOADS[4]), ("5-append-decode", inputs.WORKLOADS[5])):
        t = inputs.make(w, dev)
        B = w.batch
        g = torch.Generator(device=dev)
        g.manual_seed(4242)

        def rnd(*shape, scale=1.0, base=0.0):
            return (base + scale * torch.randn(shape, generator=g, device=dev)).to(torch.bfloat16)

        qp, kp, vp = rnd(B, 32, 128), rnd(B, 8, 128), rnd(B, 8, 128)
        wq, wk = rnd(128, scale=0.1, base=1.0), rnd(128, scale=0.1, base=1.0)
        slots = (t["lens"] - 1).contiguous()
        pos = slots.clone()
        fp8 = w.kv_dtype == "e4m3"
        ks, vs = (t["k_scale"], t["v_scale"]) if fp8 else (1.0, 1.0)
        q_out = torch.empty(B, 32, 128, dtype=torch.bfloat16, device=dev)
        out = torch.empty_like(q_out)
        hdr = torch.zeros(256, dtype=torch.uint8, device=dev)
        tensors = {"Q": q_out, "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]}
        p = gq.prepare(tensors, q_scale=t["q_scale"], k_scale=ks if fp8 else None, v_scale=vs if fp8 else None)

        def append():
            gq.append_kv(qp, kp, vp, wq, wk, pos, slots, t["kv"], q_out=q_out, k_scale=ks, v_scale=vs,
                         kv_scales=t["kv_scales"], workspace=hdr)

        def step():
            append()
            gq.launch(p)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        n = 5 if quick else 20
        rows[key] = {
            "append_us_cold": round(cold_graph_us(append, flush, calls=10 if quick else 40, reps=3 if quick else 7), 3),
            "append_us_warm_graph": round(warm_graph_us(append, calls=n), 3),
            "step_us_warm_graph": round(warm_graph_us(step, calls=n), 2),
            "decode_us_warm_graph": round(warm_graph_us(lambda: gq.launch(p), calls=n), 2),
            "batch": B, "kv": w.kv_dtype,
            "note": (f"append (norm + RoPE + K/V write, {B} requests) alone, cold (graph difference) and warm "
                     "(in a CUDA graph); a serving step = append then decode over the full cache, in a CUDA "
                     "graph, next to the decode alone"),
        }
        del t, out, p, tensors
        torch.cuda.empty_cache()
    return rows


def per_config_table(dev, peak, gq, inputs, quick=False, cpu=True):
    import torch
    flush = make_cold_flush(dev)
    table = {}
    cases = dict(inputs.WORKLOADS)
    # beyond the five workloads: an int8 cache (one bf16 scale per row) with workload 5's shape
    cases["5-int8"] = inputs.custom(64, 32768, 16384, 32768, kv_dtype="i8", index=5)
    for idx, w in cases.items():
        t = inputs.make(w, dev)
        out = torch.empty_like(t["q"])
        fp8 = w.kv_dtype == "e4m3"
        tensors = {"Q": t["q"], "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]}
        if t["kv_scales"] is not None:
            tensors["KV_SCALES"] = t["kv_scales"]
        p = gq.prepare(tensors, q_scale=t["q_scale"], k_scale=t["k_scale"] if fp8 else None,
                       v_scale=t["v_scale"] if fp8 else None)
        nbytes = algorithmic_bytes(w, t["lens"].cpu().tolist())
        for _ in range(3):
            gq.launch(p)
        torch.cuda.synchronize()
        n = 5 if quick else (20 if w.capacity * w.batch > 1 << 20 else 50)
        samples = call_samples(lambda: gq.launch(p), n, flush=flush)
        us = samples[len(samples) // 2]
        row = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
               "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "alg_bytes": nbytes,
               "splits": p.num_splits, "l2": L2_COLD,
               "us_per_call_mean": round(sum(samples) / len(samples), 3)}
        row["timer_resolution_us"], row["samples_at_median"] = timer_resolution_us(samples)
        if w.batch * w.capacity <= 1 << 12:
            # the latency-bound sizes take a few event steps: also time them
            # below the step, as the difference of two CUDA graphs
            cg = cold_graph_us(lambda: gq.launch(p), flush, calls=10 if quick else 40, reps=3 if quick else 7)
            row["us_per_call_cold_graph"] = round(cg, 3)
            row["event_samples_us"] = [round(x, 3) for x in samples]
            row["cold_graph_note"] = ("(graph of 40 x [flush, call] - graph of 40 x flush) / 40, median of 7 "
                                      "replays each: cold L2, launched from a graph; resolution ~0.1 us")
        if w.kv_dtype == "i8":
            row["note"] = "int8 codes + bf16 row scales, workload 5 shape (not one of the five workloads)"
        if w.kv_dtype in ("f16", "bf16"):
            row["torch_sdpa"] = sdpa_context(t, w, n, flush)
        if cpu and w.kv_dtype != "i8":
            row["oracle_cpu"] = oracle_config(t, w, nbytes, 3 if idx in (1, 2, 3) else 1)
        if w.batch * w.capacity <= 1 << 12:
            # warm L2, device time: 20 calls back to back inside one CUDA graph
            reps = 20
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(reps):
                    gq.launch(p)
            g.replay()
            torch.cuda.synchronize()
            row["us_per_call_warm_l2_graph"] = round(time_calls(g.replay, 10) / reps, 2)
        table[str(idx)] = row
        del t, out, p
        torch.cuda.empty_cache()
    # a 2-token verify window (two queries per request read the cache once):
    # over workload 4, and over the ragged workload 3 (the balanced schedule)
    # verify windows (T query tokens per request read the cache once): 2
    # tokens over workloads 3-5, and 3 and 4 tokens over the 8-bit caches of
    # workload 5's shape (e4m3, and int8 with bf16 row scales)
    i8_w5 = inputs.custom(64, 32768, 16384, 32768, kv_dtype="i8", index=5)
    window_rows = [(f"{i}-window2", inputs.with_(inputs.WORKLOADS[i], q_len=2), n) for i, n in (
        (4, "workload 4 with a 2-token verify window (q_len 2, causal within the window)"),
        (3, "workload 3 (ragged, NaN tail) with a 2-token verify window"),
        (5, "workload 5 (e4m3 KV) with a 2-token verify window"))]
    window_rows += [(f"5-window{T}", inputs.with_(inputs.WORKLOADS[5], q_len=T),
                     f"workload 5 (e4m3 KV) with a {T}-token verify window") for T in (3, 4)]
    window_rows += [(f"5-int8-window{T}", inputs.with_(i8_w5, q_len=T),
                     f"int8 cache + bf16 row scales (workload 5 shape) with a {T}-token verify window")
                    for T in (3, 4)]
    made = {}
    for key, w, note in window_rows:
        base = (w.index, w.kv_dtype)
        if base not in made:  # one cache per shape and format; the windows differ in q only
            made.clear()
            torch.cuda.empty_cache()
            made[base] = inputs.make(inputs.with_(w, q_len=1), dev)
        t = dict(made[base])
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed + 1)
        t["q"] = torch.randn((w.batch, w.q_len, 32, 128), generator=g, device=dev,
                             dtype=torch.float32).to(torch.float16 if w.q_dtype == "f16" else torch.bfloat16)
        out = torch.empty_like(t["q"])
        fp8 = w.kv_dtype == "e4m3"
        fmt = {"f16": 0, "bf16": 1, "e4m3": 2, "i8": 3}[w.kv_dtype]
        S = gq.plan(w.batch, w.capacity, fmt, dev)
        ws = torch.zeros(gq.workspace_size(w.batch * w.q_len, w.capacity, S), dtype=torch.uint8, device=dev)
        scales = {"k_scale": t["k_scale"], "v_scale": t["v_scale"]} if fp8 else {}

        def window():
            gq.gqa_decode_verify(t["q"], t["kv"], t["lens"], out=out, num_splits=S, workspace=ws,
                                 kv_scales=t["kv_scales"], **scales)

        for _ in range(3):
            window()
        torch.cuda.synchronize()
        nbytes = algorithmic_bytes(w, t["lens"].cpu().tolist())  # q and out of every query token
        us = time_calls(window, 5 if quick else 20, flush=flush)
        table[key] = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                      "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "alg_bytes": nbytes,
                      "splits": S, "l2": L2_COLD,
                      "note": note}
        del t, out, ws
    made.clear()
    torch.cuda.empty_cache()

    # a paged cache: workload 4 scattered over a shuffled pool of 256-token pages
    w = inputs.WORKLOADS[4]
    t = inputs.make(w, dev)
    pt = inputs.paginate(t, 256, extra_pages=8)
    del t["kv"]
    out = torch.empty_like(pt["q"])
    S = gq.plan(w.batch, w.capacity, 1, dev)
    ws = torch.zeros(gq.workspace_size(w.batch, w.capacity, S), dtype=torch.uint8, device=dev)

    def paged():
        gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"], out=out, num_splits=S,
                            workspace=ws)

    for _ in range(3):
        paged()
    torch.cuda.synchronize()
    nbytes = algorithmic_bytes(w, pt["lens"].cpu().tolist())
    us = time_calls(paged, 5 if quick else 20, flush=flush)
    table["4-paged"] = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                        "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "alg_bytes": nbytes, "splits": S,
                        "l2": L2_COLD,
                        "note": "workload 4 in a shuffled pool of 256-token pages (block table)"}
    del t, pt, out, ws
    torch.cuda.empty_cache()

    # an int8 cache (codes + bf16 row scales, workload 5 shape) in 256-token pages
    w = inputs.custom(64, 32768, 16384, 32768, kv_dtype="i8", index=5)
    t = inputs.make(w, dev)
    pt = inputs.paginate(t, 256, extra_pages=8)
    del t["kv"], t["kv_scales"]
    out = torch.empty_like(pt["q"])
    S = gq.plan(w.batch, w.capacity, 3, dev)
    ws = torch.zeros(gq.workspace_size(w.batch, w.capacity, S), dtype=torch.uint8, device=dev)

    def paged_i8():
        gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"], out=out, num_splits=S,
                            workspace=ws, kv_scales=pt["kv_scale_pages"])

    for _ in range(3):
        paged_i8()
    torch.cuda.synchronize()
    nbytes = algorithmic_bytes(w, pt["lens"].cpu().tolist())
    us = time_calls(paged_i8, 5 if quick else 20, flush=flush)
    table["5-int8-paged"] = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                             "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "alg_bytes": nbytes, "splits": S,
                             "l2": L2_COLD,
                             "note": "int8 codes + bf16 row scales (workload 5 shape) in shuffled 256-token pages"}
    del t, pt, out, ws
    torch.cuda.empty_cache()

    # the append step, alone and followed by the decode (a serving step)
    table.update(append_rows(dev, gq, inputs, flush, quick=quick))

    # one long request: bf16, batch 1, 131072 tokens (all parallelism from splitting the row)
    w = inputs.custom(1, 131072, 131072, kv_dtype="bf16", index=4)
    t = inputs.make(w, dev)
    out = torch.empty_like(t["q"])
    p = gq.prepare({"Q": t["q"], "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]}, q_scale=1.0)

    def long_one():
        gq.launch(p)

    for _ in range(3):
        long_one()
    torch.cuda.synchronize()
    nbytes = algorithmic_bytes(w, t["lens"].cpu().tolist())
    us = time_calls(long_one, 5 if quick else 20, flush=flush)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(20):
        long_one()
    b.record()
    torch.cuda.synchronize()
    table["bf16-1x131072"] = {"us_per_call": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                              "frac_of_peak": round(nbytes / us / 1e3 / peak, 4), "alg_bytes": nbytes,
                              "splits": p.num_splits, "l2": L2_COLD,
                              "us_per_call_back_to_back": round(a.elapsed_time(b) / 20 * 1e3, 2),
                              "note": "one long request: batch 1, 131072 bf16 tokens"}
    return table


def run_gpu(args):
    import numpy as np
    import torch

    from gqa_decode_attention_sm_gb300 import build as gbuild
    import gqa_decode_attention_sm_gb300 as gq
    from gqa_decode_attention_sm_gb300 import api as gapi
    from gqa_decode_attention_sm_gb300 import inputs

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)  # before the process group, so NCCL binds this rank's GPU
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0:
        gbuild.build()
    barrier(world)

    peak, peak_kind = measured_peak()
    w = inputs.WORKLOADS[args.workload]
    if args.batch:
        w = inputs.with_(w, batch=args.batch)
    if args.kv_dtype:
        eight = args.kv_dtype in ("e4m3", "i8")
        w = inputs.with_(w, kv_dtype=args.kv_dtype, q_dtype="bf16" if eight else args.kv_dtype,
                         name=f"{w.name} with {args.kv_dtype} KV")
    T = args.q_len
    if T > 1:
        w = inputs.with_(w, q_len=T, name=f"{w.name} with a {T}-token verify window")
    t = inputs.make(w, dev, seed=w.seed + 7919 * rank)
    lens_list = t["lens"].cpu().tolist()
    fp8 = w.kv_dtype == "e4m3"
    out = torch.empty_like(t["q"])
    kvf = {"f16": gapi.KV_F16, "bf16": gapi.KV_BF16, "e4m3": gapi.KV_E4M3, "i8": gapi.KV_I8}[w.kv_dtype]
    def make_step(d, o):
        """One decode step over the device inputs d (q, kv, lens, kv_scales)
        into o through the public API; returns (step, prepared or None)."""
        if T == 1:
            tensors = {"Q": d["q"], "KV": d["kv"], "O": o, "sequence_lengths": d["lens"]}
            if d["kv_scales"] is not None:
                tensors["KV_SCALES"] = d["kv_scales"]
            pp = gq.prepare(tensors, q_scale=t["q_scale"], k_scale=t["k_scale"] if fp8 else None,
                            v_scale=t["v_scale"] if fp8 else None)
            return (lambda: gq.launch(pp)), pp
        # a verify window: both stages through gqa_decode_verify, one workspace
        ws = torch.zeros(gq.workspace_size(w.batch * T, w.capacity, num_splits), dtype=torch.uint8, device=dev)
        kw = {"k_scale": t["k_scale"], "v_scale": t["v_scale"]} if fp8 else {}
        if d["kv_scales"] is not None:
            kw["kv_scales"] = d["kv_scales"]
        return (lambda: gq.gqa_decode_verify(d["q"], d["kv"], d["lens"], q_scale=t["q_scale"], out=o,
                                             num_splits=num_splits, workspace=ws, **kw)), None

    if T > 1:
        num_splits = gq.plan(w.batch, w.capacity, kvf, dev)
    step, p = make_step(t, out)
    if T == 1:
        num_splits, splits_eff = p.num_splits, p.splits_effective
    else:
        splits_eff = gapi.split_geometry(w.capacity, num_splits, kvf)[1]
    # kernels per step, by the library's own rule (one when the splits merge on chip)
    launches_per_step = gapi.launch_count(w.batch, w.capacity, kvf, T, num_splits,
                                          torch.cuda.get_device_properties(dev).multi_processor_count)
    nbytes = algorithmic_bytes(w, lens_list)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local).start().wait_first()
    time.sleep(0.3)
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    # the steps back to back, events only at the ends: an event recorded
    # between the two kernels would stop the combine from being scheduled
    # during the split kernel's tail (programmatic dependent launch)
    start.record(stream)
    for _ in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    # the dominant kernel's own duration: the split kernel alone, each launch
    # bracketed by events (stage 1 alone takes no int8 cache and no window:
    # there, the step)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        if w.kv_dtype == "i8" or T > 1:
            step()
        else:
            gq.split_stage(p)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall1 = time.time()
    time.sleep(0.3)
    clocks.stop()

    total_ms = start.elapsed_time(end)
    split_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    total_ms = max_over_ranks(total_ms, world, dev)
    all_bytes = sum_over_ranks(float(nbytes), world, dev)
    ms_per_step = total_ms / K
    value = all_bytes / (ms_per_step * 1e-3) / 1e9

    # end to end through the public API with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e:
        # host buffers on the CPUs (and so the memory) nearest the GPU, as a
        # serving process bound to the GPU's NUMA node would have them
        all_cpus = os.sched_getaffinity(0)
        cpus, h2d_probe = near_host_cpus(dev)

        # the step's inputs: q, the cache (with its int8 row scales) and the lengths
        in_keys = ("q", "kv", "lens") + (("kv_scales",) if t["kv_scales"] is not None else ())

        def pin_inputs(grp):
            """Pinned host copies of the step's inputs (in_keys, then out),
            first touched (and so placed) from the CPUs grp; returns them and
            the GB/s of one full-size host-to-device copy of the cache."""
            os.sched_setaffinity(0, grp)
            try:
                bufs = [torch.empty(t[k].shape, dtype=t[k].dtype, pin_memory=True).copy_(t[k]) for k in in_keys]
                bufs.append(torch.empty(out.shape, dtype=out.dtype, pin_memory=True).zero_())
            finally:
                os.sched_setaffinity(0, all_cpus)  # the oracle below uses every core
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            t["kv"].copy_(bufs[1], non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize(dev)
            return bufs, round(bufs[1].numel() * bufs[1].element_size() / (a.elapsed_time(b) * 1e-3) / 1e9, 1)

        # The 1 GiB probe can miss how a multi-GB buffer is placed: check the
        # real buffers and, well short of the probe, try the other CPU group.
        hbufs, full_rate = pin_inputs(cpus)
        full_rates = {f"{min(cpus)}-{max(cpus)}": full_rate}
        others = [set(c) for c in ([sorted(all_cpus)[:len(all_cpus) // 2], sorted(all_cpus)[len(all_cpus) // 2:]]
                                   if len(all_cpus) > 1 else []) if set(c) != set(cpus)]
        if h2d_probe and others and full_rate < 0.85 * max(h2d_probe.values()):
            first = cpus
            del hbufs
            hbufs, alt_rate = pin_inputs(others[0])
            full_rates[f"{min(others[0])}-{max(others[0])}"] = alt_rate
            cpus = others[0]
            if alt_rate < full_rate:
                del hbufs
                hbufs, _ = pin_inputs(first)
                cpus = first
        hin, hout = dict(zip(in_keys, hbufs[:-1])), hbufs[-1]
        t["kv"].copy_(hin["kv"], non_blocking=True)  # the device cache holds what the host copy holds
        torch.cuda.synchronize(dev)
        ke = max(2, min(K, args.e2e_steps))
        # Two device sets of the inputs and the output, used by turns: the
        # host-to-device copies of step k + 1 (on a copy stream) overlap the
        # decode of step k.  Each step still copies all its inputs in and its
        # result out; a set is refilled only after its previous decode and
        # read-back are done.  A verify window keeps one set (its steps then
        # run one after another): with two, its steps measured slower (28.3
        # against 20.8 ms at workload 5's shape with 2 tokens).
        sets = [(t, out, step)]
        if T == 1:
            d2 = {k: torch.empty_like(t[k]) for k in in_keys}
            d2.setdefault("kv_scales", None)
            out2 = torch.empty_like(out)
            sets.append((d2, out2, make_step(d2, out2)[0]))
        cs = torch.cuda.Stream(dev)
        nset = len(sets)
        copied = [torch.cuda.Event() for _ in sets]
        freed = [torch.cuda.Event() for _ in sets]
        for ev_ in freed:
            ev_.record(stream)

        def e2e_steps(n, start_ev):
            cs.wait_event(start_ev)  # no copy before the region starts
            for k in range(n):
                d, o, st = sets[k % nset]
                with torch.cuda.stream(cs):
                    cs.wait_event(freed[k % nset])
                    for key in in_keys:
                        d[key].copy_(hin[key], non_blocking=True)
                    copied[k % nset].record(cs)
                stream.wait_event(copied[k % nset])
                st()
                hout.copy_(o, non_blocking=True)
                freed[k % nset].record(stream)

        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_steps(2, a)  # both sets once, untimed
        torch.cuda.synchronize(dev)
        barrier(world)
        a.record(stream)
        e2e_steps(ke, a)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a.elapsed_time(b) / ke, world, dev)
        h2d = sum(b.numel() * b.element_size() for b in hin.values())
        e2e = {"value": round(all_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 3), "steps": ke, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hout.numel() * hout.element_size(),
               "path": "pinned host " + "/".join(in_keys) + " -> H2D -> " +
                       ("gqa_decode_prepared/fp8kv/int8kv" if T == 1 else "gqa_decode_verify") + " -> D2H out",
               "overlap": ("two device input sets: step k+1's H2D (copy stream) overlaps step k's decode"
                           if nset == 2 else "none: one device input set, steps one after another"),
               "host_cpus": f"{min(cpus)}-{max(cpus)}", "h2d_probe_GBps": h2d_probe,
               "h2d_full_size_GBps": full_rates}
        del hbufs, hin, hout, sets

    achieved = nbytes / (split_ms * 1e-3) / 1e9
    # the committed capture is of the workload as defined (no batch or KV override)
    traffic, traffic_note = (traffic_per_launch(args.workload) if not (args.batch or args.kv_dtype or T > 1)
                             else (None, None))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "capacity": w.capacity, "kv_dtype": w.kv_dtype,
                   "q_dtype": w.q_dtype, "q_len": T, "lengths": f"U[{w.len_lo},{w.len_hi}]" if w.len_lo != w.len_hi
                   else w.len_lo, "num_splits": num_splits, "splits_effective": splits_eff,
                   "alg_bytes_per_step_per_gpu": nbytes,
                   "l2": f"inputs ({nbytes / 1e9:.2f} GB) larger than L2 (129 MB); no flush between steps"
                   if nbytes > 2 * 129e6 else "inputs smaller than 2x L2: steps run warm",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "us_per_call": round(ms_per_step * 1e3, 2),
                   "frac_of_peak": round(value / world / peak, 4)},
        "roofline": {"bound": "hbm", "kernel": "split_kv_mma_kernel", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs (copy, burst)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "frac_of_nominal_7900": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "traffic_note": traffic_note, "kernel_ms": round(split_ms, 4),
                     "alg_bytes_per_launch": nbytes},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks.summary(wall0, wall1),
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline and T == 1:
        import oracle
        oracle.build()
        threads = oracle.default_threads()
        secs, sb, nrows = 0.0, 0, 0
        for b in range(min(w.batch, args.cpu_batch_rows)):
            host = host_batch_row(t, b)
            s_, b_ = oracle_rows(t, host, list(range(32)), threads)
            secs, sb, nrows = secs + s_, sb + b_, nrows + 32
        line["cpu_baseline"] = {"value": round(sb / secs / 1e9, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "seconds": round(secs, 2),
                                "sample": f"{nrows} query-head rows ({nrows // 32} batch rows) of "
                                          f"'{w.name}', FP64, {threads} threads; {sb} KV bytes"}
    if rank == 0 and not args.no_per_config:
        line["per_config"] = per_config_table(dev, peak, gq, inputs, quick=args.quick,
                                              cpu=not args.no_cpu_baseline)
    if rank == 0 and world == 1 and args.read_ceiling:
        line["read_ceiling"] = read_ceiling(achieved)
    if rank == 0 and args.sweep:
        line["sweep"] = {"l2": L2_COLD, "rows": planner_sweep(dev, peak, gq, inputs, quick=args.quick)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def read_ceiling(achieved):
    """Context for the roofline: the read rate this GPU reaches with the split
    kernel's data movement alone (bench_read_ceiling.cu: contiguous runs of a
    4.3 GB buffer streamed through a shared-memory ring by 1-D bulk copies, no
    arithmetic), built with nvcc for sm_103a and run in a child process after
    the timed region.  Adds the split kernel's GB/s as a fraction of the best."""
    import subprocess
    from gqa_decode_attention_sm_gb300 import build as gbuild
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "read_ceiling")
    subprocess.run([gbuild.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe,
                    os.path.join(ROOT, "bench_read_ceiling.cu")], check=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    d = json.loads(run.stdout.strip().splitlines()[-1])
    if run.returncode != 0 or "best_GBps" not in d:
        raise RuntimeError(f"read-ceiling probe failed: {run.stdout[-300:]} {run.stderr[-300:]}")
    d["split_kernel_GBps"] = round(achieved, 1)
    d["split_kernel_frac_of_best"] = round(achieved / d["best_GBps"], 4)
    return d


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--kv-dtype", choices=["f16", "bf16", "e4m3", "i8"], default=None,
                    help="override the workload's KV format (8-bit formats take a bf16 query)")
    ap.add_argument("--q-len", type=int, default=1, choices=[1, 2, 3, 4],
                    help="query tokens per request: above 1 the step is a verify window (gqa_decode_verify)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-batch-rows", type=int, default=4,
                    help="batch rows (all 32 query heads each) in the oracle CPU-baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="also time SWEEP_SHAPES (batch x capacity x KV format, uniform and ragged lengths) "
                         "with the automatic plan, cold, and report them under 'sweep'")
    ap.add_argument("--read-ceiling", action="store_true",
                    help="also build and run bench_read_ceiling.cu (the read rate of the split kernel's data "
                         "movement without arithmetic) and report the split kernel as a fraction of it")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
