"""Benchmark: deterministic exact ragged top-k on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]
                    [--page-size P] [--op topk|stats|indexer]

A step is one call of the whole hot path (one launch of the library over one
batch of rows).  The default workload is the decode batch: 64 rows with
lengths uniform in [4096, 131072], lightning-indexer scores, k = 2048.  The
timed region replays the K launches from CUDA graphs over rotating input
copies whose total exceeds 3x the L2 size, so every step reads cold scores
from HBM.  Rank 0 prints one JSON line.  With the default workload the same
run also times the other k = 2048 workload, the prefill chunk (16384 causal
rows), and the two reported workloads (long rows, adversarial ties) by the
same method, and reports them under "also" (--no-also skips them).

--page-size P times the page-table transform (topk_ragged_paged) and
--op stats the tie / plateau statistics op (topk_ragged_stats) on the same
workload, in the same way.  --op indexer times the indexer + top-k chain
(topk_ragged_indexer: the tensor-core indexer scores from bf16 queries and
keys, then the selection) on the decode or prefill shape.

--impl reference times the CPU oracle (the plain per-row sort the library is
checked against) on the host cores, on a bounded sample of rows per step.
Under torchrun with N > 1 every rank runs its own replica of the workload
(rows are independent, nothing is exchanged); only the timing is reduced.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ragged exact top-k rows/s and achieved HBM GB/s (k=2048) vs roofline"
METRIC_STATS = "ragged tie/plateau statistics rows/s and achieved HBM GB/s (k=2048) vs roofline"
METRIC_INDEXER = "lightning-indexer scores + exact top-k rows/s (k=2048) vs roofline"
STATS_FIELDS = 6   # 32-bit fields of one topk_row_stats
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SRC = os.path.join(ROOT, "sparse_attention_deterministic_gb300", "csrc", "topk_ragged.cu")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0        # GB300 HBM3e, as specified
NOMINAL_BF16_TFLOPS = 2250.0    # dense bf16 tensor throughput, as specified
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--config", default="decode",
                   choices=["tiny", "decode", "prefill", "adversarial", "long"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=500)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-also", action="store_true",
                   help="with the default decode workload, skip the prefill, long and adversarial records under 'also'")
    p.add_argument("--page-size", type=int, default=0,
                   help="write KV-cache slots through random per-row page tables of this "
                        "page size (topk_ragged_paged); 0: plain indices")
    p.add_argument("--op", default="topk", choices=["topk", "stats", "indexer"],
                   help="topk: the selection; stats: per-row tie/plateau statistics; "
                        "indexer: indexer scores on the tensor cores, then the selection")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, world: int) -> float:
    """The slowest rank's time: the job's steps end when every rank's do."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ms_per_step: float, world: int) -> float:
    """Units per second over all ranks (weak scaling: each rank runs the
    same workload on its own GPU, with no exchange between ranks)."""
    return world * units_per_rank / (ms_per_step / 1e3)


def algorithmic_bytes(total_len: int, B: int, k: int) -> int:
    """One read of every score, the index writes and the row metadata."""
    return 4 * total_len + 4 * B * k + 8 * B


def algorithmic_bytes_stats(total_len: int, B: int) -> int:
    """One read of every score, the row metadata and the statistics written."""
    return 4 * total_len + 8 * B + 4 * STATS_FIELDS * B


def kernel_source_sha() -> str:
    """Hash of every kernel source file (csrc/*.cu, *.cuh, in name order)."""
    h = hashlib.sha256()
    csrc = os.path.dirname(KERNEL_SRC)
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(workload)
    if not entry or entry.get("kernel_source_sha") != kernel_source_sha():
        return None
    return entry.get("dram_bytes_per_launch")


def hbm_peak():
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        # The samples go to a temporary file (or BENCH_CLOCKS_DIR); their
        # summary goes into the JSON line.
        out_dir = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        os.makedirs(out_dir, exist_ok=True)
        self.path = os.path.join(out_dir, f"clocks_gpu{self.index}_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: the top half by power draw
        order = sorted(range(len(sm)), key=lambda i: power[i])
        loaded = [sm[i] for i in order[len(order) // 2:]] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- #
# CPU oracle arm (also the cpu_baseline key of our arm).
# --------------------------------------------------------------------------- #

def time_oracle(w, seconds: float, rows_per_call=None, max_calls=None, op="topk", max_threads=None):
    """Run the oracle on row samples of the workload for about `seconds`.
    Returns (rows/s, elements/s, threads, description)."""
    import numpy as np

    import oracle

    s, st, ln = w.numpy()
    B = len(st)
    cores = len(os.sched_getaffinity(0))
    rows_per_call = B if rows_per_call is None else max(1, min(B, rows_per_call))
    threads = max(1, min(cores, rows_per_call, max_threads or cores))
    rows = elems = calls = 0
    cursor = 0
    t0 = time.perf_counter()
    while True:
        sel = (np.arange(cursor, cursor + rows_per_call) % B)
        cursor = (cursor + rows_per_call) % B
        if op == "stats":
            threads = 1
            oracle.row_stats(s, st[sel], ln[sel], w.k)
        else:
            oracle.topk_ragged(s, st[sel], ln[sel], w.k, w.offset_mode, n_threads=threads,
                               with_values=False)
        rows += rows_per_call
        elems += int(ln[sel].clip(min=0).sum())
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_calls is not None and calls >= max_calls):
            break
    desc = (f"{calls} oracle call(s) of {rows_per_call} row(s) of the {w.name} workload "
            f"({rows} rows, {elems} scores) in {el:.2f} s on {threads} host thread(s)")
    return rows / el, elems / el, threads, desc


def run_reference_indexer(args):
    import workloads as W
    w = W.INDEXER[args.config](device="cpu")
    ln = w.lengths.numpy()
    t0 = time.perf_counter()
    indexer_reference_sample(w, [0])
    per_row = time.perf_counter() - t0
    rows_per_step = max(1, min(w.B, int(120.0 / max(1, args.steps + args.warmup) / max(per_row, 1e-9))))
    cursor = 0

    def step():
        nonlocal cursor
        rows = [(cursor + j) % w.B for j in range(rows_per_step)]
        cursor = (cursor + rows_per_step) % w.B
        indexer_reference_sample(w, rows)
        return int(ln[rows].sum())

    for _ in range(args.warmup):
        step()
    elems = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        elems += step()
    el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC_INDEXER, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 scores; u32 select",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "k": w.k, "op": "indexer",
                                        "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} row(s) per step, rows cycled in order; {elems} keys "
                                   f"in {el:.2f} s"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference(args, rank):
    import workloads as W

    if rank != 0:
        return
    if args.op == "indexer":
        run_reference_indexer(args)
        return
    w = W.make(args.config, device="cpu") if args.config in ("tiny", "adversarial") else None
    if w is None:
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        w = W.make(args.config, device=dev).to("cpu")
    import numpy as np

    import oracle
    s, st, ln = w.numpy()
    cores = len(os.sched_getaffinity(0))
    # Calibrate one row's single-thread cost over the length mix, then size
    # every step so the whole run ends in about two minutes.
    stats = args.op == "stats"

    def run_oracle(sel, n_threads):
        if stats:   # a Python loop over rows: one thread
            oracle.row_stats(s, st[sel], ln[sel], w.k)
        else:
            oracle.topk_ragged(s, st[sel], ln[sel], w.k, w.offset_mode, n_threads=n_threads,
                               with_values=False)

    probe = np.linspace(0, w.B - 1, num=min(w.B, 8)).astype(np.int64)
    t0 = time.perf_counter()
    run_oracle(probe, 1)
    per_row_s = (time.perf_counter() - t0) / len(probe)
    budget_s = 120.0 / max(1, args.steps + args.warmup)
    par = 1 if stats else cores
    rows_per_step = max(1, min(w.B, int(budget_s / max(per_row_s, 1e-9) * par)))
    threads = 1 if stats else max(1, min(cores, rows_per_step))
    cursor = 0

    def step():
        nonlocal cursor
        sel = np.arange(cursor, cursor + rows_per_step) % w.B
        cursor = (cursor + rows_per_step) % w.B
        run_oracle(sel, threads)
        return int(ln[sel].clip(min=0).sum())

    for _ in range(args.warmup):
        step()
    elems = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        elems += step()
    el = time.perf_counter() - t0
    rows = rows_per_step * args.steps
    value = rows / el
    line = {
        "impl": "reference", "metric": METRIC_STATS if stats else METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "k": w.k, "sum_len": w.total_len(),
                   "offset_mode": w.offset_mode, "rows_per_step": rows_per_step, "op": args.op},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} row(s) of the {w.name} workload per step, "
                                   f"rows cycled in order; {elems} scores in {el:.2f} s"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "elements_per_s": elems / el,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# Our arm.
# --------------------------------------------------------------------------- #

def measure(args, w, device, local, world, op="topk", page_size=0):
    """Time one workload on this rank: cold-L2 graph replays of K launches
    (the headline), warm L2, the end-to-end public call from pinned host
    buffers, parity against the oracle and byte identity of the timed
    launches.  Returns a dict of the measurements."""
    import numpy as np
    import torch

    import oracle
    import sparse_attention_deterministic_gb300 as pkg

    B, k, total = w.B, w.k, w.total_len()
    stats = op == "stats"
    out_cols = STATS_FIELDS if stats else k
    in_bytes = w.scores.numel() * 4 + 8 * B
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    n_copies = max(2, math.ceil(3 * l2 / in_bytes) + 1)
    copies = [w.scores.clone() for _ in range(n_copies)]
    outs = [torch.empty((B, out_cols), dtype=torch.int32, device=device) for _ in range(n_copies)]
    stream = torch.cuda.Stream(device)
    info = ({"kernel": "topk_stats_kernel", "grid": B, "cluster": 1, "launches": 1 if B else 0}
            if stats else pkg.launch_info(w.scores.numel(), B, k, device))

    # The page-table transform: random per-row page tables (the row-start
    # offset has no meaning there, so the mode keeps only its other bits).
    page_table, mode = None, w.offset_mode
    if page_size > 0:
        n_pages = -(-int(w.lengths.max()) // page_size)
        g = torch.Generator().manual_seed(1234)
        page_table = torch.stack([torch.randperm(4 * n_pages, generator=g)[:n_pages] for _ in range(B)]
                                 ).to(torch.int32).to(device)
        mode = w.offset_mode & ~pkg.TOPK_OFFSET_ROW_START

    def call(scores, starts, lengths, out, s=None):
        if stats:
            pkg.topk_ragged_stats(scores, starts, lengths, k, out=out, stream=s)
        else:
            pkg.topk_ragged(scores, starts, lengths, k, mode, out_idx=out, stream=s,
                            page_table=page_table, page_size=max(page_size, 1))

    def launch(i, s=stream):
        call(copies[i], w.row_starts, w.lengths, outs[i], s)

    # Parity guard: the timed configuration must match the oracle on this input.
    with torch.cuda.stream(stream):
        launch(0)
    stream.synchronize()
    s_np, st_np, ln_np = w.numpy()
    if stats:
        ref = oracle.row_stats(s_np, st_np, ln_np, k)[0].view(np.int32)
    else:
        ref, _, _ = oracle.topk_ragged(s_np, st_np, ln_np, k, mode,
                                       n_threads=len(os.sched_getaffinity(0)), with_values=False)
    if page_table is not None:
        ref = oracle.paged_slots(ref, page_table.cpu().numpy(), page_size)
    parity = bool(np.array_equal(outs[0].cpu().numpy(), ref))
    if pkg.device_status(device) != 0:
        parity = False

    # CUDA graphs: one with a launch per input copy, one for the remainder.
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                launch(i % n_copies, torch.cuda.current_stream())
        return g

    full = capture(n_copies)
    rem_n = args.steps % n_copies
    rem = capture(rem_n) if rem_n else None
    reps = args.steps // n_copies

    with ClockSampler(local) as clocks:
        # warm-up (untimed): W launches, then ~1 s of replays so the clock
        # samples cover a loaded GPU.
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                launch(i % n_copies)
        stream.synchronize()
        t_end = time.perf_counter() + 1.0
        with torch.cuda.stream(stream):   # replay() launches on the current stream
            while time.perf_counter() < t_end:
                full.replay()
                stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                full.replay()
            if rem is not None:
                rem.replay()
            ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_per_step = ms / args.steps
    # Every timed launch read an identical copy of the inputs, so their
    # outputs must agree byte for byte.
    torch.cuda.synchronize(device)
    repeats_identical = all(torch.equal(outs[i], outs[0]) for i in range(1, n_copies))

    # Warm L2: the same launches over a single input copy (it stays in L2
    # when it fits), for comparison with the cold-L2 number above.
    n_warm = 16
    g_warm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=stream):
        for _ in range(n_warm):
            launch(0, torch.cuda.current_stream())
    warm_reps = max(1, min(args.steps, 2000) // n_warm)
    with torch.cuda.stream(stream):
        g_warm.replay()
        ew0, ew1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ew0.record(stream)
        for _ in range(warm_reps):
            g_warm.replay()
        ew1.record(stream)
    ew1.synchronize()
    warm_ms = max_over_ranks(ew0.elapsed_time(ew1), world) / (warm_reps * n_warm)

    # End to end through the public API with host buffers: pinned H2D of the
    # step's scores and metadata, the call, D2H of the indices.
    h_scores = w.scores.cpu().pin_memory()
    h_starts = w.row_starts.cpu().pin_memory()
    h_lengths = w.lengths.cpu().pin_memory()
    h_out = torch.empty((B, out_cols), dtype=torch.int32).pin_memory()
    d_scores = torch.empty_like(w.scores)
    d_starts = torch.empty_like(w.row_starts)
    d_lengths = torch.empty_like(w.lengths)
    d_out = torch.empty((B, out_cols), dtype=torch.int32, device=device)

    def e2e_step():
        d_scores.copy_(h_scores, non_blocking=True)
        d_starts.copy_(h_starts, non_blocking=True)
        d_lengths.copy_(h_lengths, non_blocking=True)
        call(d_scores, d_starts, d_lengths, d_out)
        h_out.copy_(d_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(5):
            e2e_step()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.e2e_steps
    e2e_parity = bool(np.array_equal(h_out.numpy(), ref))

    peak, peak_kind = hbm_peak()
    alg = algorithmic_bytes_stats(total, B) if stats else algorithmic_bytes(total, B, k)
    achieved = alg / (ms_per_step * 1e-3) / 1e9
    return {
        "B": B, "k": k, "total": total, "mode": mode, "info": info, "parity": parity,
        "repeats_identical": repeats_identical, "n_copies": n_copies, "in_bytes": in_bytes, "l2": l2,
        "ms_per_step": ms_per_step, "warm_ms": warm_ms, "e2e_ms": e2e_ms, "e2e_parity": e2e_parity,
        "h2d": h_scores.numel() * 4 + 8 * B, "d2h": B * out_cols * 4, "alg": alg, "achieved": achieved,
        "peak": peak, "peak_kind": peak_kind, "clocks": clocks.summary(),
        "traffic": stored_traffic(w.name + (":stats" if stats else "")),
    }


def roofline_of(m):
    return {"bound": "hbm", "achieved": m["achieved"], "peak": m["peak"], "unit": "GB/s",
            "frac": m["achieved"] / m["peak"], "peak_kind": m["peak_kind"],
            "frac_of_nominal": m["achieved"] / NOMINAL_HBM_GBS, "traffic": m["traffic"],
            "algorithmic_bytes_per_launch": m["alg"]}


ALSO_WORKLOADS = ("prefill", "long", "adversarial")


def also_record(args, name: str, device, local, world) -> dict:
    """One workload timed like the headline, as a record under "also"."""
    import workloads as W
    wa = W.make(name, device=device)
    ma = measure(args, wa, device, local, world)
    return {
        "workload": name, "B": ma["B"], "k": ma["k"], "sum_len": ma["total"],
        "offset_mode": ma["mode"], "ms_per_step": ma["ms_per_step"],
        "value": whole_job_rate(ma["B"], ma["ms_per_step"], world), "unit": "rows/s",
        "elements_per_s": whole_job_rate(ma["total"], ma["ms_per_step"], world),
        "achieved_gbs": ma["achieved"], "roofline": roofline_of(ma), "launch": ma["info"],
        "parity_vs_oracle": ma["parity"], "timed_launches_identical": ma["repeats_identical"],
        "warm_l2": {"ms_per_step": ma["warm_ms"], "achieved_gbs": ma["alg"] / (ma["warm_ms"] * 1e-3) / 1e9},
        "e2e": {"value": whole_job_rate(ma["B"], ma["e2e_ms"], world), "unit": "rows/s",
                "h2d_bytes_per_step": ma["h2d"], "d2h_bytes_per_step": ma["d2h"],
                "ms_per_step": ma["e2e_ms"], "parity_vs_oracle": ma["e2e_parity"]},
        "l2": f"{ma['n_copies']} rotating input copies ({ma['n_copies'] * ma['in_bytes'] / 1e6:.0f} MB"
              f" > 3x L2 {ma['l2'] / 1e6:.0f} MB): cold scores every step",
        "gpu_launches": args.steps * ma["info"]["launches"],
        "clocks": ma["clocks"],
    }


def run_ours(args, rank, world, local):
    import torch

    import sparse_attention_deterministic_gb300 as pkg
    import workloads as W

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    pkg.build()
    pkg.init(device)

    stats = args.op == "stats"
    if stats and args.page_size > 0:
        raise SystemExit("--page-size applies to --op topk")
    w = W.make(args.config, device=device)
    m = measure(args, w, device, local, world, op=args.op, page_size=args.page_size)
    # The second k = 2048 workload, prefill, and the two reported ones (long
    # rows, adversarial ties), in the same run and by the same method, beside
    # the decode headline.
    also = None
    if args.config == "decode" and args.op == "topk" and args.page_size == 0 and not args.no_also:
        also = {name: also_record(args, name, device, local, world) for name in ALSO_WORKLOADS}

    if rank != 0:
        return
    B, total = m["B"], m["total"]
    ms_per_step = m["ms_per_step"]
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        rps, eps, threads, desc = time_oracle(w.to("cpu"), args.cpu_seconds, op=args.op)
        rps1, _, _, desc1 = time_oracle(w.to("cpu"), args.cpu_seconds / 3, op=args.op, max_threads=1)
        cpu = {"value": rps, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": desc, "elements_per_s": eps,
               "single_thread": {"value": rps1, "unit": "rows/s", "sample": desc1}}
    line = {
        "metric": METRIC_STATS if stats else METRIC, "value": whole_job_rate(B, ms_per_step, world),
        "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": args.config, "B": B, "k": m["k"], "sum_len": total,
                   "offset_mode": m["mode"], "page_size": args.page_size, "op": args.op, "scores": "fp32",
                   "l2": f"{m['n_copies']} rotating input copies ({m['n_copies'] * m['in_bytes'] / 1e6:.0f} MB"
                         f" > 3x L2 {m['l2'] / 1e6:.0f} MB): cold scores every step",
                   "timing": "CUDA events around graph replays of K launches on one stream",
                   "launch": m["info"], "parity_vs_oracle": m["parity"],
                   "timed_launches_identical": m["repeats_identical"]},
        "elements_per_s": whole_job_rate(total, ms_per_step, world),
        "warm_l2": {"ms_per_step": m["warm_ms"], "value": whole_job_rate(B, m["warm_ms"], world),
                    "unit": "rows/s", "achieved_gbs": m["alg"] / (m["warm_ms"] * 1e-3) / 1e9},
        "achieved_gbs": m["achieved"],
        "roofline": roofline_of(m),
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(B, m["e2e_ms"], world), "unit": "rows/s",
                "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"], "ms_per_step": m["e2e_ms"],
                "parity_vs_oracle": m["e2e_parity"]},
        "gpu_launches": args.steps * m["info"]["launches"],
        "clocks": m["clocks"],
    }
    if also is not None:
        line["also"] = also
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# The indexer + top-k chain.
# --------------------------------------------------------------------------- #

def indexer_bytes_flops(w) -> tuple[int, int]:
    """Algorithmic bytes of the score kernel (every key row read once, the
    queries, weights, shifts and metadata, the score writes) and its flops."""
    B = w.B
    nbytes = (256 * w.unique_key_rows() + 2 * 64 * 128 * B + 4 * 64 * B + 4 * B + 12 * B + 4 * w.n_scores)
    return nbytes, 2 * 64 * 128 * w.n_scores


def indexer_reference_sample(w, rows, bound=False):
    """The oracle's indexer scores and selection for a list of rows; with
    bound, also each score's error-bound magnitude (scale * sum_h w_h
    sum_d |q_hd k_td| + sum_h w_h |x_h|), of which 2^-16 bounds the fp32 path."""
    import numpy as np

    import oracle
    q = w.q[rows].float().cpu().numpy()
    wt = w.w[rows].cpu().numpy()
    b = w.bias[rows].cpu().numpy()
    ln = w.lengths[rows].cpu().numpy()
    ks = w.key_starts[rows].cpu().numpy()
    lo, hi = int(ks.min()), int((ks + ln).max())
    keys = w.keys[lo:hi].float().cpu().numpy()
    ss = np.zeros(len(rows), dtype=np.int64)
    ss[1:] = np.cumsum(ln)[:-1]
    s, _ = oracle.indexer_scores(q, wt, b, keys, ks - lo, ln, ss, int(ln.sum()), w.scale)
    oracle.topk_ragged(s.astype(np.float32), ss, ln, w.k, 0, with_values=False)
    if not bound:
        return s, ss
    mag = np.zeros_like(s)
    for j in range(len(rows)):
        kj = keys[ks[j] - lo:ks[j] - lo + ln[j]].astype(np.float64)
        x = w.scale * (kj @ q[j].astype(np.float64).T) + b[j]
        mag[ss[j]:ss[j] + ln[j]] = (w.scale * (np.abs(kj) @ np.abs(q[j].astype(np.float64)).T) @ wt[j]
                                    + np.abs(x) @ wt[j])
    return s, ss, mag


def run_indexer(args, rank, world, local):
    import numpy as np
    import torch

    import oracle
    import sparse_attention_deterministic_gb300 as pkg
    import workloads as W

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    pkg.build()
    pkg.init(device)
    if args.config not in W.INDEXER:
        raise SystemExit("--op indexer takes --config decode or prefill")
    w = W.INDEXER[args.config](device=device)
    B, k = w.B, w.k
    scores = torch.zeros(w.n_scores, dtype=torch.float32, device=device)
    out = torch.empty((B, k), dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device)
    args_t = (w.q, w.w, w.keys, w.key_starts, w.lengths, w.score_starts)

    def chain(s=None):
        pkg.topk_ragged_indexer(*args_t, k=k, bias=w.bias, scale=w.scale, scores=scores, out_idx=out, stream=s)

    def scores_only(s=None):
        pkg.indexer_scores(*args_t, bias=w.bias, scale=w.scale, out=scores, stream=s)

    # Parity guard: the selection over the GPU's scores is the oracle's, and
    # sampled rows' scores are within the fp32 bound of the oracle's float64.
    with torch.cuda.stream(stream):
        chain(stream)
    stream.synchronize()
    s_np = scores.cpu().numpy()
    ln_np, ss_np = w.lengths.cpu().numpy(), w.score_starts.cpu().numpy()
    ref_idx, _, _ = oracle.topk_ragged(s_np, ss_np, ln_np, k, 0, n_threads=len(os.sched_getaffinity(0)),
                                       with_values=False)
    parity = bool(np.array_equal(out.cpu().numpy(), ref_idx)) and pkg.device_status(device) == 0
    sample = [0, B // 2, B - 1]
    ref_s, ref_ss, mag = indexer_reference_sample(w, sample, bound=True)
    worst = 0.0
    for j, i in enumerate(sample):
        L, a = int(ln_np[i]), int(ss_np[i])
        got = s_np[a:a + L].astype(np.float64)
        r0 = ref_ss[j]
        err = np.abs(got - ref_s[r0:r0 + L]) / (2.0 ** -16 * mag[r0:r0 + L] + 1e-30)
        worst = max(worst, float(err.max()))
    scores_parity = worst <= 1.0

    n_graph = 16
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n_graph):
            chain(torch.cuda.current_stream())
    reps = max(1, args.steps // n_graph)
    steps = reps * n_graph

    def timed(fn_replay, n):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(n):
                fn_replay()
            ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1)

    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                chain(stream)
            g.replay()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        ms = timed(g.replay, reps)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        # the dominant kernel alone, same stream
        with torch.cuda.stream(stream):
            for _ in range(3):
                scores_only(stream)
        ms_scores = timed(lambda: scores_only(stream), n_graph * 4) / (n_graph * 4)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / steps
    value = whole_job_rate(B, ms_per_step, world)

    # End to end with host inputs: H2D of queries, weights, shifts, keys and
    # metadata, the chain, D2H of the indices.
    host = [t.cpu().pin_memory() for t in (w.q, w.w, w.bias, w.keys, w.key_starts, w.lengths, w.score_starts)]
    dev_t = [torch.empty_like(t) for t in (w.q, w.w, w.bias, w.keys, w.key_starts, w.lengths, w.score_starts)]
    h_out = torch.empty((B, k), dtype=torch.int32).pin_memory()

    def e2e_step():
        for d, h in zip(dev_t, host):
            d.copy_(h, non_blocking=True)
        pkg.topk_ragged_indexer(dev_t[0], dev_t[1], dev_t[3], dev_t[4], dev_t[5], dev_t[6], k=k, bias=dev_t[2],
                                scale=w.scale, scores=scores, out_idx=out)
        h_out.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        e1.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.e2e_steps
    e2e_parity = bool(np.array_equal(h_out.numpy(), ref_idx))

    if rank != 0:
        return
    nbytes, flops = indexer_bytes_flops(w)
    hbm, hbm_kind = hbm_peak()
    bf16 = json.load(open(PEAKS_PATH)).get("bf16_tflops") if os.path.exists(PEAKS_PATH) else None
    bf16_kind = "measured" if bf16 else "fallback"
    bf16 = bf16 or 1900.0
    t_hbm, t_tensor = nbytes / (hbm * 1e9), flops / (bf16 * 1e12)
    if t_hbm >= t_tensor:
        achieved = nbytes / (ms_scores * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_kind": hbm_kind, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_launch": nbytes}
    else:
        achieved = flops / (ms_scores * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                "frac": achieved / bf16, "peak_kind": bf16_kind + " (dense bf16, burst)",
                "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS, "algorithmic_flops_per_launch": flops}
    roof.update({"kernel": "indexer_scores_kernel", "kernel_ms": ms_scores,
                 "traffic": stored_traffic(w.name)})
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        t0 = time.perf_counter()
        rows_done = elems = 0
        i = 0
        while time.perf_counter() - t0 < args.cpu_seconds:
            indexer_reference_sample(w, [i % B])
            rows_done += 1
            elems += int(ln_np[i % B])
            i += 1
        el = time.perf_counter() - t0
        cpu = {"value": rows_done / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
               "sample": f"{rows_done} row(s) of the {w.name} workload, one per oracle call (float64 scores, "
                         f"then the selection): {elems} keys in {el:.2f} s"}
    line = {
        "metric": METRIC_INDEXER, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x bf16 -> f32; u32 select", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "k": k, "sum_len": w.n_scores, "key_rows": w.unique_key_rows(),
                   "op": "indexer", "l2": f"keys {w.keys.numel() * 2 / 1e6:.0f} MB, queries "
                                         f"{w.q.numel() * 2 / 1e6:.0f} MB: inputs larger than L2"
                                         if w.keys.numel() * 2 > 3 * 129e6 else
                                         "keys shared by every row stay in L2; queries stream",
                   "timing": "CUDA events around graph replays of 16 chained calls on one stream",
                   "parity_vs_oracle": parity, "scores_within_bound": scores_parity,
                   "scores_worst_err_over_bound": worst},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(B, e2e_ms, world), "unit": "rows/s",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
                "d2h_bytes_per_step": B * k * 4, "ms_per_step": e2e_ms, "parity_vs_oracle": e2e_parity},
        "gpu_launches": 2 * steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.op == "indexer":
        run_indexer(args, rank, world, local)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
