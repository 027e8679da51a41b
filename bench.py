"""Benchmark of the exact per-row top-k transform on GB300 (one JSON line on stdout).

Workload (the 128k-context decode sweep of the indexer top-k): B=256 rows of
c4_len=32768 fp32 scores, N(0,1) plus one N(0, sigma=4) offset per row, full
seq_lens, k=1024, paged output (page_size=64, a random page permutation per row).
One step is one call of topk_transform_paged over the batch.

Timing: W untimed warm-up steps, then exactly K steps replayed from a CUDA graph
whose nodes cycle through R input sets that together exceed 4x the L2 size, so
every step reads its scores from HBM; CUDA events on the launching stream bracket
the K steps, with a device synchronise (and, under torchrun, a barrier) on both
sides; the slowest rank's time counts. nvidia-smi samples the clocks meanwhile.

Also reported: the roofline of the kernel (algorithmic bytes per launch over its
average launch time, against the measured HBM copy bandwidth), the end-to-end
rate through the same public call with pinned host buffers and the copies inside
the timed region, the CPU oracle's rate on the host cores (a baseline only), and
a sweep over the other batch sizes and the raw form.

``--impl reference`` times the CPU oracle instead, on the same workload and
metric; each step processes one row per host core.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "top-k rows/sec & scored Gelem/s at c4_len=32768,k=1024 (1 GB300); % HBM roofline"
C4_LEN, K_TOP, PAGE_SIZE = 32768, 1024, 64
KERNEL_NAME = "topk_rows_kernel"
KERNEL_SRC = os.path.join(ROOT, "sparse_attention_indexer_sm_gb300", "csrc", "topk_select.cu")
PROFILE = os.path.join(ROOT, "profiles", "topk_rows_kernel_paged_b256_n32768.md")
L2_FACTOR = 4
REFERENCE_BUDGET_S = 120.0  # the reference arm's timed steps fit about this many seconds


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=256)
    ap.add_argument("--form", choices=["paged", "raw"], default="paged")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=11,
                    help="timed windows of exactly --steps calls; the median is reported")
    ap.add_argument("--profile-workload", default=None, metavar="NAME",
                    help="only run --warmup then --steps plain calls of one workload (for ncu "
                         "captures; nothing is timed): " + ", ".join(PROFILE_WORKLOADS))
    return ap.parse_args()


PROFILE_WORKLOADS = ("c1", "c2-8192", "c2-32768", "c3-b<B>-paged", "c3-b<B>-raw", "c4-banded",
                     "c4-narrow", "c4-subnormal", "c5-b<B>", "window-causal", "window-w8192")


def named_workload(name: str):
    """The workload a --profile-workload name stands for (the sweep's configurations)."""
    if name == "c1":
        return workloads.config1()
    if name.startswith("c2-"):
        return workloads.config2(int(name[3:]))
    if name.startswith("c3-b"):
        b, form = name[4:].split("-")
        return workloads.config3(int(b), form)
    if name.startswith("c4-"):
        return workloads.config4(name[3:])
    if name.startswith("c5-b"):
        return workloads.config5(int(name[4:]))
    if name == "window-causal":
        return workloads.prefill_windows(4096, C4_LEN, window=None)
    if name == "window-w8192":
        return workloads.prefill_windows(4096, C4_LEN, window=8192)
    raise SystemExit(f"unknown workload {name!r}; one of: " + ", ".join(PROFILE_WORKLOADS))


def run_profile_workload(args):
    """--warmup then --steps plain calls of one workload on rotating input sets (inputs
    beyond L2 as in the timed runs), for a profiler to capture; prints one line."""
    import torch
    import sparse_attention_indexer_sm_gb300 as pkg
    w = named_workload(args.profile_workload)
    dev = torch.device("cuda:0")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = w.scores.nbytes + w.seq_lens.nbytes + (w.page_table.nbytes if w.form == "paged" else 0)
    n_sets = max(2, min(64, math.ceil(L2_FACTOR * l2 / set_bytes)))
    sets = device_sets(w, n_sets, dev, torch)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            call(pkg, w, sets[i % n_sets], stream)
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_workload": args.profile_workload, "name": w.name,
                      "calls": args.warmup + args.steps, "input_sets": n_sets}), flush=True)


def algorithmic_bytes(batch: int, L: int, k: int, form: str, page_size: int = PAGE_SIZE) -> int:
    """Bytes the method must move per call: scores read once, seq_len, the k output
    slots, and (paged) one page-table entry per distinct page that can hold a winner."""
    per_row = 4 * L + 4 + 4 * k
    if form == "paged":
        per_row += 4 * min(k, (L + page_size - 1) // page_size)
    elif form == "ragged":
        per_row += 4
    return batch * per_row


def workload_bytes(w, page_size: int = PAGE_SIZE) -> int:
    """algorithmic_bytes for any workload: per row 4 L_b + 4 + 4 k, plus the page-table
    entries (paged) or the row start / window start (ragged, window)."""
    total = 4 * w.scored_elements + w.batch * (4 + 4 * w.k)
    if w.form == "paged":
        L = np.clip(w.seq_lens.astype(np.int64), 0, w.scores.shape[1])
        total += int((4 * np.minimum(w.k, (L + page_size - 1) // page_size)).sum())
    elif w.form in ("ragged", "window"):
        total += 4 * w.batch
    return int(total)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def source_sha() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(batch: int, form: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload and the kernel source has not changed since."""
    if batch != 256 or form != "paged":
        return None
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            key, _, v = line.strip()[2:].partition(":")
            vals[key.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != source_sha():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"topk_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t_start: float, t_end: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except OSError:
            pass
        finally:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows]
        mx = [float(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


# --------------------------------------------------------------------------- our arm

def max_over_ranks(secs: float, dist, device) -> float:
    """The slowest rank's time (rows shard across ranks with no data exchange;
    this timing reduction is the only collective)."""
    import torch
    t = torch.tensor([secs], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(batch: int, form: str, rank: int):
    """Rank r's own rows: the same shapes, its own seed (weak scaling)."""
    return workloads.config3(batch, form, seed=workloads.BASE_SEED + 2 + 1000 * rank)


def device_sets(w, n_sets, dev, torch):
    """n_sets device copies of one workload (distinct buffers, identical bits)."""
    s_host = torch.from_numpy(w.scores)
    sets = []
    for _ in range(n_sets):
        d = {"scores": s_host.to(dev), "seq": torch.from_numpy(w.seq_lens).to(dev),
             "out": torch.empty((w.batch, w.k), dtype=torch.int32, device=dev)}
        if w.form == "paged":
            d["pt"] = torch.from_numpy(w.page_table).to(dev)
        if w.form in ("window", "ragged"):
            d["starts"] = torch.from_numpy(w.row_starts).to(dev)
        sets.append(d)
    return sets


def call(pkg, w, d, stream):
    if w.form == "paged":
        pkg.topk_transform_paged(d["scores"], d["seq"], d["pt"], w.page_size, w.k, out=d["out"],
                                 stream=stream)
    elif w.form == "window":
        pkg.topk_transform_window(d["scores"], d["starts"], d["seq"], w.k,
                                  max_row_len_hint=w.max_row_len, out=d["out"], stream=stream)
    elif w.form == "ragged":
        pkg.topk_transform_ragged(d["scores"], d["starts"], d["seq"], w.k,
                                  max_row_len_hint=w.max_row_len, out=d["out"], stream=stream)
    else:
        pkg.topk_transform_raw(d["scores"], d["seq"], w.k, out=d["out"], stream=stream)


def time_steps(pkg, w, steps, warmup, dev, torch, l2_bytes, dist=None, repeats=1):
    """Time exactly `steps` calls, `repeats` times over. The calls cycle through R input
    sets that together exceed L2_FACTOR x L2 (l2_bytes = 0: two sets, L2-hot); they are
    replayed from two CUDA graphs, one over all R sets and one over the first
    steps % R, so each timed window is exactly `steps` graph-launched calls. Each window
    is bracketed by a device synchronise (and, under torchrun, a barrier) on both sides,
    with CUDA events on the launching stream. Returns (seconds of each window, the
    slowest rank's under torchrun; wall-clock span of the windows; R)."""
    set_bytes = w.scores.nbytes + w.seq_lens.nbytes + (w.page_table.nbytes if w.form == "paged" else 0)
    n_sets = max(2, min(4096, math.ceil(L2_FACTOR * l2_bytes / set_bytes)))
    sets = device_sets(w, n_sets, dev, torch)
    stream = torch.cuda.Stream(dev)
    full, rest = divmod(steps, n_sets)
    graphs = []
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 1)):  # untimed warm-up steps
            call(pkg, w, sets[i % n_sets], stream)
        stream.synchronize()
        for n, reps in ((n_sets, full), (rest, 1)):
            if n == 0 or reps == 0:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for d in sets[:n]:
                    call(pkg, w, d, stream)
            g.replay()  # one untimed replay
            graphs.append((g, reps))
        stream.synchronize()
    windows = []
    t0 = time.time()
    for _ in range(repeats):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            start.record(stream)
            for g, reps in graphs:
                for _ in range(reps):
                    g.replay()
            end.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        secs = start.elapsed_time(end) / 1e3
        windows.append(max_over_ranks(secs, dist, dev) if dist is not None else secs)
    t1 = time.time()
    del graphs, sets
    torch.cuda.empty_cache()
    return windows, (t0, t1), n_sets


def window_stats(windows, steps):
    """Median, min and max microseconds per call over the timed windows."""
    us = sorted(x / steps * 1e6 for x in windows)
    return {"windows": len(us), "us_per_call_median": statistics.median(us),
            "us_per_call_min": us[0], "us_per_call_max": us[-1]}


def time_grouped(pkg, ws, steps, dev, torch, l2_bytes):
    """The problems ws as one grouped call and as separate calls, each step on its
    own rotating input set (CUDA graph replay); returns (grouped s, separate s)."""
    set_bytes = sum(w.scores.nbytes + w.seq_lens.nbytes
                    + (w.page_table.nbytes if w.form == "paged" else 0) for w in ws)
    n_sets = max(2, min(1024, math.ceil(L2_FACTOR * l2_bytes / set_bytes)))
    sets = [[device_sets(w, 1, dev, torch)[0] for w in ws] for _ in range(n_sets)]

    def grouped(ds):
        probs = []
        for w, d in zip(ws, ds):
            q = {"form": w.form, "k": w.k, "scores": d["scores"], "seq_lens": d["seq"],
                 "out": d["out"]}
            if w.form == "paged":
                q["page_table"], q["page_size"] = d["pt"], w.page_size
            probs.append(q)
        return probs

    probs = [grouped(ds) for ds in sets]
    stream = torch.cuda.Stream(dev)
    result = []
    for mode in ("grouped", "separate"):
        with torch.cuda.stream(stream):
            def one(i):
                if mode == "grouped":
                    pkg.topk_transform_grouped(probs[i], stream=stream)
                else:
                    for w, d in zip(ws, sets[i]):
                        call(pkg, w, d, stream)
            for i in range(n_sets):
                one(i)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(n_sets):
                    one(i)
            graph.replay()
            stream.synchronize()
            reps = max(1, steps // n_sets)
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for _ in range(reps):
                graph.replay()
            end.record(stream)
            end.synchronize()
            result.append(start.elapsed_time(end) / 1e3 / (reps * n_sets))
            del graph
    del sets, probs
    torch.cuda.empty_cache()
    return tuple(result)


def time_e2e(pkg, w, steps, dev, torch):
    """Same call with pinned host inputs: H2D of scores/seq_lens/page_table, the
    kernel, D2H of the result, every step, inside the timed region."""
    stream = torch.cuda.Stream(dev)
    h_scores = torch.from_numpy(w.scores).pin_memory()
    h_seq = torch.from_numpy(w.seq_lens).pin_memory()
    h_pt = torch.from_numpy(w.page_table).pin_memory() if w.form == "paged" else None
    h_out = torch.empty((w.batch, w.k), dtype=torch.int32).pin_memory()
    d = {"scores": torch.empty_like(h_scores, device=dev), "seq": torch.empty_like(h_seq, device=dev),
         "out": torch.empty((w.batch, w.k), dtype=torch.int32, device=dev)}
    if h_pt is not None:
        d["pt"] = torch.empty_like(h_pt, device=dev)

    def step():
        d["scores"].copy_(h_scores, non_blocking=True)
        d["seq"].copy_(h_seq, non_blocking=True)
        if h_pt is not None:
            d["pt"].copy_(h_pt, non_blocking=True)
        call(pkg, w, d, stream)
        h_out.copy_(d["out"], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        stream.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        end.synchronize()
    secs = start.elapsed_time(end) / 1e3
    h2d = h_scores.numel() * 4 + h_seq.numel() * 4 + (h_pt.numel() * 4 if h_pt is not None else 0)
    d2h = h_out.numel() * 4
    return secs, h2d, d2h


def isolated_latency(pkg, w, dev, torch, l2_bytes, calls: int = 200):
    """Device time of one call issued by itself: a spin kernel (torch.cuda._sleep) keeps
    the stream busy while the host enqueues an event, the call and an event, so the
    events bracket only the device's start of the call after the spin and the call
    itself, not the binding's host work. Inputs rotate as in time_steps. Returns the
    median and 10th/90th percentiles in microseconds."""
    set_bytes = w.scores.nbytes + w.seq_lens.nbytes + (w.page_table.nbytes if w.form == "paged" else 0)
    n_sets = max(2, min(64, math.ceil(L2_FACTOR * l2_bytes / set_bytes)))
    sets = device_sets(w, n_sets, dev, torch)
    stream = torch.cuda.Stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    us = []
    with torch.cuda.stream(stream):
        for i in range(calls + 10):
            torch.cuda._sleep(100000)  # about 50 us of device time
            e0.record(stream)
            call(pkg, w, sets[i % n_sets], stream)
            e1.record(stream)
            e1.synchronize()
            if i >= 10:  # warm-up calls first
                us.append(e0.elapsed_time(e1) * 1e3)
    del sets
    torch.cuda.empty_cache()
    us.sort()
    return {"batch": w.batch, "form": w.form,
            "workload": f"isolated call, B={w.batch} (stream idle before it)",
            "us_median": statistics.median(us), "us_p10": us[len(us) // 10],
            "us_p90": us[(9 * len(us)) // 10], "calls": calls, "input_sets": n_sets}


def cpu_baseline(w, seconds: float = 1.5):
    """The oracle as it stands, on every host core, over whole batches of the same
    workload until about `seconds` of wall time (a bounded sample)."""
    import oracle
    o = oracle.default()
    cores = o.usable_cores()
    rows, t0 = 0, time.perf_counter()
    while True:
        o.run(w, threads=cores)
        rows += w.batch
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    # the same oracle on one core, over the workload's first 32 rows at a time
    n1 = min(32, w.batch)
    part = workloads.Workload(w.name, w.form, w.k, w.scores[:n1], w.seq_lens[:n1],
                              w.page_table[:n1] if w.page_table is not None else None, w.page_size)
    rows1, t1 = 0, time.perf_counter()
    while True:
        o.run(part, threads=1)
        rows1 += n1
        el1 = time.perf_counter() - t1
        if el1 >= seconds / 3:
            break
    return {"value": rows / el, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows} rows ({rows // w.batch} full batches of the bench workload), "
                      f"{el:.2f} s wall on {cores} threads",
            "single_core_value": rows1 / el1,
            "single_core_sample": f"{rows1} rows ({n1} rows of the bench workload at a time), "
                                  f"{el1:.2f} s wall on 1 thread"}


def workload_for(batch: int, form: str):
    return workloads.config3(batch, form)


def describe(w) -> str:
    return (f"topk_transform_{w.form} B={w.batch} c4_len={C4_LEN} k={w.k}"
            + (f" page_size={w.page_size}" if w.form == "paged" else "")
            + " decode scores N(0,1)+N(0,4) row offset, full seq_lens")


def run_ours(args):
    import torch
    import sparse_attention_indexer_sm_gb300 as pkg

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as td
        td.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = td
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkg.load_library()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    peak, peak_kind = peaks()

    w = rank_workload(args.batch, args.form, rank)
    with ClockSampler(local) as clk:
        windows, (t0, t1), n_sets = time_steps(pkg, w, args.steps, args.warmup, dev, torch, l2,
                                               dist, repeats=args.repeats)
        clocks = clk.summary(t0, t1)
    secs = statistics.median(windows)  # each window: exactly K steps, slowest rank's time
    launches = args.steps
    per_call = secs / args.steps
    rows_per_s = world * w.batch * args.steps / secs
    gelem = world * w.scored_elements * args.steps / secs / 1e9
    alg = algorithmic_bytes(w.batch, C4_LEN, w.k, w.form)
    achieved = alg / per_call / 1e9
    traffic = profiled_traffic(w.batch, w.form)

    e2e_steps = max(20, min(args.steps, 400))
    if dist is not None:
        dist.barrier()
    e_secs, h2d, d2h = time_e2e(pkg, w, e2e_steps, dev, torch)
    if dist is not None:  # the whole job's end-to-end rate: the slowest rank decides
        e_secs = max_over_ranks(e_secs, dist, dev)

    result = {
        "metric": METRIC,
        "value": rows_per_s,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": per_call * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": describe(w), "batch_per_gpu": w.batch, "c4_len": C4_LEN,
                   "k": w.k, "form": w.form, "page_size": w.page_size,
                   "l2": f"inputs larger than L2: {n_sets} rotating input sets, "
                         f"{n_sets * w.scores.nbytes / 1e6:.0f} MB >= {L2_FACTOR}x L2 ({l2 / 1e6:.0f} MB)",
                   "timing": "CUDA graph replay, CUDA events on the launching stream",
                   "parallelism": f"rows sharded, {world} GPU(s), no collective"},
        "scored_gelem_per_s": gelem,
        "us_per_call": per_call * 1e6,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
                     "frac_of_nominal_8TBps": achieved / 8000.0, "kernel": KERNEL_NAME},
        "e2e": {"value": world * w.batch * e2e_steps / e_secs, "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": e_secs / e2e_steps * 1e3},
        "clocks": clocks,
        "repeats": window_stats(windows, args.steps),
        "gpu_launches": launches,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0 and world == 1 and not args.no_sweep:
        sweep = []

        def line(ws, steps, label=None, l2_bytes=l2, alg_bytes=None, repeats=5):
            """One sweep entry: `repeats` windows of exactly `steps` calls, median and spread."""
            win, _, ns = time_steps(pkg, ws, steps, 5, dev, torch, l2_bytes, repeats=repeats)
            st = window_stats(win, steps)
            pc = st["us_per_call_median"] / 1e6
            ab = alg_bytes if alg_bytes is not None else workload_bytes(ws)
            entry = {"batch": ws.batch, "form": ws.form}
            if label is not None:
                entry["workload"] = label
            entry.update({"us_per_call": pc * 1e6, "us_per_call_min": st["us_per_call_min"],
                          "us_per_call_max": st["us_per_call_max"], "windows": st["windows"],
                          "rows_per_s": ws.batch / pc,
                          "scored_gelem_per_s": ws.scored_elements / pc / 1e9,
                          "gbs": ab / pc / 1e9, "frac": ab / pc / 1e9 / peak, "input_sets": ns})
            return entry

        for (b, form) in ((1, "paged"), (8, "paged"), (64, "paged"), (128, "paged"),
                          (256, "paged"), (256, "raw"), (64, "raw")):
            if (b, form) == (w.batch, w.form):
                continue
            ws = workload_for(b, form)
            sweep.append(line(ws, 4000 if b >= 64 else 8000,
                              alg_bytes=algorithmic_bytes(b, C4_LEN, ws.k, form)))
        # the other configurations of the workload table, each timed the same way
        others = [("C1", workloads.config1()), ("C2 c4_len=8192", workloads.config2(8192)),
                  ("C2 c4_len=32768", workloads.config2(32768))]
        others += [(f"C4 {dist}", workloads.config4(dist)) for dist in ("banded", "narrow", "subnormal")]
        others += [(f"C5 B={b}", workloads.config5(b)) for b in (1, 2, 4)]
        for label, ws in others:
            sweep.append(line(ws, 2000, label=f"{label}: {ws.name}"))
        # prefill-shaped window rows: 4096 queries over a 32768-key context, causal and
        # with a sliding window of 8192 keys
        for window in (None, 8192):
            ws = workloads.prefill_windows(4096, C4_LEN, window=window)
            sweep.append(line(ws, 200, label=ws.name))
        # several independent problems per step: four C3 paged batches of 64 rows, as
        # one grouped call (one launch) and as four calls
        ws4 = [workloads.config3(64, seed=workloads.BASE_SEED + 2 + 1000 * i) for i in range(4)]
        tg, tsep = time_grouped(pkg, ws4, 2000, dev, torch, l2)
        ab = sum(workload_bytes(w) for w in ws4)
        sweep.append({"batch": 256, "form": "grouped", "workload": "4 x paged B=64 c4_len=32768 k=1024",
                      "us_per_call": tg * 1e6, "us_per_call_separate": tsep * 1e6,
                      "gbs": ab / tg / 1e9, "frac": ab / tg / 1e9 / peak})
        # labelled extras, never the headline (a failure here leaves the line intact): the
        # headline workload with its inputs hot in L2 (two input sets replayed), and the
        # device time of single calls issued with the stream otherwise idle
        try:
            e = line(w, 4000, label="headline, L2-hot", l2_bytes=0, alg_bytes=alg)
            e["l2"] = f"hot: {e['input_sets']} input sets replayed"
            sweep.append(e)
        except Exception as exc:  # noqa: BLE001
            sweep.append({"workload": "headline, L2-hot", "error": repr(exc)})
        for b in (1, 64, 256):
            try:
                sweep.append(isolated_latency(pkg, workload_for(b, "paged"), dev, torch, l2))
            except Exception as exc:  # noqa: BLE001
                sweep.append({"workload": f"isolated call, B={b}", "error": repr(exc)})
        result["sweep"] = sweep
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    o = oracle.default()
    cores = o.usable_cores()
    w = workload_for(args.batch, args.form)

    def part(n):
        return workloads.Workload(w.name, w.form, w.k, w.scores[:n], w.seq_lens[:n],
                                  None if w.page_table is None else w.page_table[:n], w.page_size)

    # one step: `rows_per_step` rows of the workload, one per thread (all host cores);
    # the warm-up steps time a step, and the sample shrinks (down to one row on one
    # thread) until the K timed steps fit REFERENCE_BUDGET_S
    rows_per_step = min(cores, w.batch)
    sub = part(rows_per_step)
    for i in range(max(args.warmup, 1)):
        t = time.perf_counter()
        o.run(sub, threads=rows_per_step)
        step = time.perf_counter() - t
        if args.steps * step > REFERENCE_BUDGET_S and rows_per_step > 1:
            rows_per_step = max(1, int(rows_per_step * REFERENCE_BUDGET_S / (args.steps * step)))
            sub = part(rows_per_step)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.run(sub, threads=rows_per_step)
    secs = time.perf_counter() - t0
    cores = rows_per_step
    value = rows_per_step * args.steps / secs
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": describe(w), "batch_per_gpu": w.batch, "c4_len": C4_LEN, "k": w.k,
                   "form": w.form, "page_size": w.page_size},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {rows_per_step} rows of the workload, one per thread"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.profile_workload is not None:
        run_profile_workload(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
