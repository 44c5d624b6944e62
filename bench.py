#!/usr/bin/env python
"""Benchmark of the table-batched embedding-bag (TBE) hot path on GB300.

One step = one forward (pooled gather) + one backward (sort, segment,
short/long-run reduce) over one batch of the mid-size skewed workload:
T=8 fp16 tables of 100,000 rows, D=128, B=2048, Poisson(20) bag lengths,
Zipf(1.05) ids, fp16 output, fp32 output gradients.  Four index batches are
generated once, kept resident on the device and rotated; the 129 MB L2 is
flushed (a 256 MB write, then a 256 MB read of another buffer) before every
timed step, outside its events.

Metric: effective bytes per second -- every lookup's row (forward) and every
lookup's output-gradient slice (backward) counted, plus indices, offsets,
outputs and the unique-row gradients written; see effective_bytes().

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the
operator has no exchange step); rank 0 prints the whole-job line.  ``--impl reference`` times the CPU oracle on the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TBE fwd/bwd effective HBM GB/s & M lookups/s (% of 8 TB/s peak)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = "mid_skewed"
WORKLOAD_DESC = ("TBE mid-size skewed: T=8 fp16 tables x 100000 rows, D=128, B=2048, bag lengths "
                 "Poisson(20) (one empty bag per table), ids Zipf(1.05) through a per-table permutation, "
                 "fp16 output, fp32 grad_out; forward + backward (row gradients)")
N_BATCHES = 4
INDEX_BYTES = 8  # width of ids and offsets in the byte accounting (--index-bits)
IDX_NP = {8: np.int64, 4: np.int32}
DT_NAMES = {0: "f32", 1: "f16", 2: "bf16"}
OPT_LR, OPT_EPS = 0.01, 1e-8  # exact row-wise Adagrad step timed beside the headline
FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--B", type=int, default=None, help="batch size override (profiling of smaller cases)")
    ap.add_argument("--only", choices=["both", "fwd", "bwd"], default="both")
    ap.add_argument("--path", choices=["auto", "gather", "histogram"], default="auto")
    ap.add_argument("--hist-variant", choices=["fp16", "bf16", "weighted", "tables4", "all"], default="fp16",
                    help="tables of the histogram sweep")
    ap.add_argument("--index-bits", type=int, choices=[64, 32], default=64,
                    help="width of ids and offsets (32: the *_i32 entry points)")
    ap.add_argument("--tuning", default=None,
                    help='JSON object of tbe_tuning fields to set first, e.g. \'{"long_run_threshold": 256}\'')
    ap.add_argument("--sweep", choices=["backward", "histogram"], default=None,
                    help="tuning sweeps: backward = long-run threshold x chunk on the run-length band, mid-size and "
                         "backward-skew workloads; histogram = histogram path against the gather path over mean bag "
                         "length x table rows; one JSON line per point")
    ap.add_argument("--profile", action="store_true",
                    help="plain launch loop for a profiler: --warmup then --steps eager steps, one JSON line")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def effective_bytes(p, unique_per_table):
    """Algorithmic bytes of one forward and one backward (no dedup credit).

    FWD = sum_i (D_t*s_w + 8 + 4*weighted) + (T*B+1)*8 + B*sumD*s_out
    BWD = sum_i (4*D_t + 8 + 4*weighted) + (T*B+1)*8 + sum_t U_t*(8 + 4*D_t)
    """
    from tbe_inputs import ELEM_BYTES

    lens = np.diff(p.offsets).reshape(p.T, p.B).sum(axis=1).astype(np.int64)  # lookups per table
    sw = np.array([ELEM_BYTES[int(d)] for d in p.weights_dtype], np.int64)
    D = p.D.astype(np.int64)
    w = (p.table_weighted.astype(np.int64) if p.per_sample_weights is not None else np.zeros(p.T, np.int64))
    s_out = ELEM_BYTES[int(p.out_dtype)]
    ib = INDEX_BYTES
    offs = (p.T * p.B + 1) * ib
    fwd = int(np.sum(lens * (D * sw + ib + 4 * w)) + offs + p.B * int(D.sum()) * s_out)
    U = np.asarray(unique_per_table, np.int64)
    bwd = int(np.sum(lens * (4 * D + ib + 4 * w)) + offs + np.sum(U * (8 + 4 * D)))
    return fwd, bwd


def compulsory_bytes(p, unique_per_table):
    """Bytes one forward and one backward cannot avoid: every distinct row
    (forward) and every output-gradient row (backward) once, plus indices,
    weights, offsets and outputs.

    FWD_c = sum_t U_t*D_t*s_w + 8*N + 4*N_weighted + (T*B+1)*8 + B*sumD*s_out
    BWD_c = 8*N + 4*N_weighted + (T*B+1)*8 + 4*B*sumD + sum_t U_t*(8 + 4*D_t)
    """
    from tbe_inputs import ELEM_BYTES

    lens = np.diff(p.offsets).reshape(p.T, p.B).sum(axis=1).astype(np.int64)
    sw = np.array([ELEM_BYTES[int(d)] for d in p.weights_dtype], np.int64)
    D = p.D.astype(np.int64)
    w = (p.table_weighted.astype(np.int64) if p.per_sample_weights is not None else np.zeros(p.T, np.int64))
    U = np.asarray(unique_per_table, np.int64)
    ids = int(np.sum(lens * (INDEX_BYTES + 4 * w)))
    offs = (p.T * p.B + 1) * INDEX_BYTES
    sumD = int(D.sum())
    fwd = int(np.sum(U * D * sw)) + ids + offs + p.B * sumD * ELEM_BYTES[int(p.out_dtype)]
    bwd = ids + offs + 4 * p.B * sumD + int(np.sum(U * (8 + 4 * D)))
    return fwd, bwd


def optimizer_bytes(p, unique_per_table):
    """Algorithmic bytes of one exact row-wise Adagrad step: per distinct row
    its id (8), its gradient (4 D), its weights read and written (2 D x the
    table's element size) and its momentum read and written (8); plus the
    per-table counts."""
    from tbe_inputs import ELEM_BYTES

    U = np.asarray(unique_per_table, np.int64)
    D = p.D.astype(np.int64)
    sw = np.array([ELEM_BYTES[int(d)] for d in p.weights_dtype], np.int64)
    return int(np.sum(U * (8 + 4 * D + 2 * sw * D + 8))) + 8 * (p.T + 1)


def kernel_bytes(p, U_total):
    """Algorithmic bytes of each backward kernel for one launch (the
    forward gather's are the forward's effective bytes)."""
    N = p.N
    D = int(p.D[0])
    tb = p.T * p.B
    return {
        "bwd_linearize": INDEX_BYTES * (N + tb + 1) + 4 * N + 4 * N,
        "bwd_sort_pass": 16 * N,
        "bwd_rle": 4 * N + 12 * U_total,
        "bwd_classify": 4 * U_total,
        "bwd_reduce": N * (4 * D + 4 + 4) + U_total * (8 + 4 + 4 * D),
    }


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, r in rows for k in range(4) if r[k].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


class L2Flush:
    """Evicts the 129 MB L2 between steps: a 256 MB write, then a 256 MB read
    of another buffer so that the write's dirty lines are written back
    before the step starts (the step then sees a cold, clean L2)."""

    def __init__(self, dev):
        import torch

        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, k):
        import torch

        self.w.fill_(float(k))
        torch.sum(self.r, dim=0, out=self.acc)


def spread(ms):
    """Mean, median and 90th percentile of a list of times (microseconds)."""
    a = 1e3 * np.asarray(ms, np.float64)
    return dict(mean_us=float(a.mean()), median_us=float(np.median(a)), p90_us=float(np.percentile(a, 90)))


def apply_tuning(tbe, spec):
    """Sets the tbe_tuning fields named in the JSON object `spec` (None: the
    library's defaults) and returns the tuning in effect."""
    if spec:
        tbe.set_tuning(**json.loads(spec))
    return tbe.get_tuning()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def traffic_from_profiles(kernel, workload=WORKLOAD):
    """DRAM bytes per launch measured by ncu for `kernel`, if the committed
    record (profiles/dram_traffic.json) was taken from the current source of
    that kernel."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    srcs = {"fwd_gather": "tbe_forward.cu", "bwd_reduce": "tbe_backward.cu",
            "bwd_sort_pass": "tbe_backward.cu", "fwd_histogram": "tbe_histogram.cu",
            "exact_update": "tbe_optimizer.cu"}
    src = srcs.get(kernel)
    if src is None:
        return None
    h = hashlib.sha256(open(os.path.join(ROOT, "table_embedding_bags_gb300", "csrc", src), "rb").read()).hexdigest()[:16]
    with open(path) as f:
        entries = json.load(f)["entries"]
    for e in entries:
        if e["kernel"] == kernel and e["src_sha"] == h and e["workload"] == workload:
            return float(e["bytes_per_launch"])
    return None


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_profile(args):
    """Eager steps of one workload for a profiler (no graphs, no timing hygiene)."""
    import torch

    import table_embedding_bags_gb300 as tbe
    from tbe_inputs import make_config, materialize_weights

    tbe.load_library()
    apply_tuning(tbe, args.tuning)
    p = make_config(args.workload, B=args.B, with_grad=args.only != "fwd")
    plan = tbe.Plan.from_problem(p)
    ind = torch.from_numpy(p.indices.astype(IDX_NP[INDEX_BYTES])).cuda()
    off = torch.from_numpy(p.offsets.astype(IDX_NP[INDEX_BYTES])).cuda()
    psw = None if p.per_sample_weights is None else torch.from_numpy(p.per_sample_weights).cuda()
    path = {"auto": tbe.TBE_PATH_AUTO, "gather": tbe.TBE_PATH_GATHER, "histogram": tbe.TBE_PATH_HISTOGRAM}[args.path]
    w = materialize_weights(p, device="cuda") if args.only != "bwd" else None
    G = torch.from_numpy(p.grad_out).cuda() if args.only != "fwd" else None
    bufs = tbe.BackwardBuffers(plan, p.B, p.N) if args.only != "fwd" else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = None
    for k in range(args.warmup + args.steps):
        if k == args.warmup:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        if args.only != "bwd":
            tbe.tbe_forward(plan, w, ind, off, p.B, psw, dev_status=status, path=path)
        if args.only != "fwd":
            tbe.tbe_backward(plan, G, ind, off, p.B, psw, bufs=bufs, dev_status=status,
                             want_run_starts=False, want_sorted_positions=False)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return dict(profile=True, workload=args.workload, B=p.B, N=p.N, only=args.only, path=args.path,
                steps=args.steps, wall_ms_per_step=1e3 * (time.perf_counter() - t0) / max(args.steps, 1))


# ---------------------------------------------------------------------------
# tuning sweeps
# ---------------------------------------------------------------------------

SWEEP_BWD_WORKLOADS = ["band_short", "band_mid", "band_long", "mid_skewed", "bwd_skew"]
SWEEP_TAU = [16, 32, 64, 128, 256]
SWEEP_CHUNK = [64, 128, 256]
SWEEP_HIST_ROWS = [8, 16, 32, 64]
SWEEP_HIST_LEN = [4, 8, 16, 32, 48, 64, 128, 256, 512]
SWEEP_HIST_LOOKUPS = 4 << 20  # lookups per histogram-sweep batch (B = this / mean length)


def time_replays(torch, fn, flush, reps, warm=2):
    """Captures fn() in a CUDA graph and times `reps` replays, each after an
    L2 flush, with CUDA events; returns (median, mean) in microseconds."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for k in range(warm):
        flush(k)
        g.replay()
    torch.cuda.synchronize()
    us = []
    for k in range(reps):
        flush(k)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        us.append(1e3 * e0.elapsed_time(e1))
    return float(np.median(us)), float(np.mean(us))


def sweep_backward(args, tbe, torch, flush):
    """Backward time over long-run threshold x chunk (plus the defaults)."""
    from tbe_inputs import make_config

    default = tbe.get_tuning()
    names = [args.workload] if args.workload != WORKLOAD else SWEEP_BWD_WORKLOADS
    for name in names:
        p = make_config(name, batch=0, B=args.B)
        plan = tbe.Plan.from_problem(p)
        ind, off = torch.from_numpy(p.indices).cuda(), torch.from_numpy(p.offsets).cuda()
        G = torch.from_numpy(p.grad_out).cuda()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        points = [(default["long_run_threshold"], default["long_chunk"])]
        points += [(tau, ch) for tau in SWEEP_TAU for ch in SWEEP_CHUNK]
        for tau, ch in points:
            tbe.set_tuning(**dict(default, long_run_threshold=tau, long_chunk=ch))
            bufs = tbe.BackwardBuffers(plan, p.B, p.N)

            def fn():
                tbe.tbe_backward(plan, G, ind, off, p.B, None, bufs=bufs, dev_status=status,
                                 want_run_starts=False, want_sorted_positions=False)

            med, mean = time_replays(torch, fn, flush, args.steps)
            assert int(status.item()) == 0, f"device status {int(status.item())}"
            U = int(bufs.unique_count[-1].item())
            print(json.dumps(dict(sweep="backward", workload=name, N=p.N, U=U, long_run_threshold=tau,
                                  long_chunk=ch, default=(tau, ch) == points[0], median_us=round(med, 2),
                                  mean_us=round(mean, 2))), flush=True)
            del bufs
    tbe.set_tuning(**default)


HIST_VARIANTS = {  # name: (table dtype, tables, weighted)
    "fp16": ("fp16", 1, False), "bf16": ("bf16", 1, False), "weighted": ("fp16", 1, True),
    "tables4": ("fp16", 4, False),
}


def sweep_histogram(args, tbe, torch, flush):
    """Forward time of the histogram path and of the gather path on T tables
    of `rows` x 128 with bag lengths U{L/2 .. 3L/2} and uniform ids; the
    variant fixes the table dtype, T and whether lookups carry per-sample
    weights."""
    from tbe_inputs import DT_BF16, DT_F16, DT_F32, make_problem, materialize_weights

    names = list(HIST_VARIANTS) if args.hist_variant == "all" else [args.hist_variant]
    for name in names:
        dt_name, T, weighted = HIST_VARIANTS[name]
        dt = DT_F16 if dt_name == "fp16" else DT_BF16
        rows_list = SWEEP_HIST_ROWS if name == "fp16" else [16, 64]
        for rows in rows_list:
            for L in SWEEP_HIST_LEN:
                B = int(min(262144, max(1024, SWEEP_HIST_LOOKUPS // (L * T))))
                rng = np.random.default_rng([rows, L, T])
                lens = rng.integers(max(1, L // 2), L + L // 2 + 1, size=(T, B))
                ids = [rng.integers(0, rows, size=int(lens[t].sum())) for t in range(T)]
                psw = rng.random(int(lens.sum())).astype(np.float32) if weighted else None
                p = make_problem(T, B, rows=[rows] * T, D=[128] * T, weights_dtype=[dt] * T, out_dtype=DT_F32,
                                 lengths=lens, ids=ids, psw=psw, seed=rows * 1000 + L)
                w = materialize_weights(p, device="cuda")
                plan = tbe.Plan.from_problem(p)
                ind = torch.from_numpy(p.indices.astype(IDX_NP[INDEX_BYTES])).cuda()
                off = torch.from_numpy(p.offsets.astype(IDX_NP[INDEX_BYTES])).cuda()
                d_psw = torch.from_numpy(psw).cuda() if weighted else None
                out = torch.empty((B, 128 * T), dtype=torch.float32, device="cuda")
                status = torch.zeros(1, dtype=torch.int32, device="cuda")
                res = {}
                for path, code in (("histogram", tbe.TBE_PATH_HISTOGRAM), ("gather", tbe.TBE_PATH_GATHER)):
                    def fn(code=code):
                        tbe.tbe_forward(plan, w, ind, off, B, d_psw, out=out, dev_status=status, path=code)

                    res[path] = time_replays(torch, fn, flush, args.steps)[0]
                assert int(status.item()) == 0, f"device status {int(status.item())}"
                print(json.dumps(dict(sweep="histogram", variant=name, rows=rows, T=T, mean_bag=L, B=B, N=p.N,
                                      index_bits=8 * INDEX_BYTES, histogram_us=round(res["histogram"], 2),
                                      gather_us=round(res["gather"], 2),
                                      faster="histogram" if res["histogram"] < res["gather"] else "gather")),
                      flush=True)


def run_sweep(args):
    import torch

    import table_embedding_bags_gb300 as tbe

    tbe.load_library()
    torch.cuda.set_device(0)
    apply_tuning(tbe, args.tuning)
    flush = L2Flush(torch.device("cuda", 0))
    if args.sweep == "backward":
        sweep_backward(args, tbe, torch, flush)
    else:
        sweep_histogram(args, tbe, torch, flush)


def run_ours(args, world, rank, local):
    import torch

    import table_embedding_bags_gb300 as tbe
    from tbe_inputs import make_config, materialize_weights

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tbe.load_library()
    tuning = apply_tuning(tbe, args.tuning)
    probs = [make_config(args.workload, batch=k, B=args.B) for k in range(N_BATCHES)]
    p0 = probs[0]
    weights = materialize_weights(p0, device=dev)
    plan = tbe.Plan.from_problem(p0, device=dev)
    nmax = max(p.N for p in probs)
    bufs = tbe.BackwardBuffers(plan, p0.B, nmax, device=dev)
    out = torch.empty((p0.B, p0.total_D), dtype=torch.float16 if p0.out_dtype == 1 else torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dev_in = []
    for p in probs:
        dev_in.append(dict(indices=torch.from_numpy(p.indices.astype(IDX_NP[INDEX_BYTES])).to(dev),
                           offsets=torch.from_numpy(p.offsets.astype(IDX_NP[INDEX_BYTES])).to(dev),
                           grad=torch.from_numpy(p.grad_out).to(dev),
                           psw=None if p.per_sample_weights is None else torch.from_numpy(p.per_sample_weights).to(dev)))
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    tbe.trace_enable(True)
    path = {"auto": tbe.TBE_PATH_AUTO, "gather": tbe.TBE_PATH_GATHER, "histogram": tbe.TBE_PATH_HISTOGRAM}[args.path]

    def step(k):
        d = dev_in[k % N_BATCHES]
        tbe.tbe_forward(plan, weights, d["indices"], d["offsets"], p0.B, d["psw"], out=out, dev_status=status,
                        path=path)
        tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p0.B, d["psw"], bufs=bufs,
                         dev_status=status, want_run_starts=False, want_sorted_positions=False)

    for k in range(args.warmup):
        flush(k)
        step(k)
    torch.cuda.synchronize()
    # unique rows per table of every batch (for the effective bytes)
    uniq = []
    for k in range(N_BATCHES):
        step(k)
        torch.cuda.synchronize()
        uc = bufs.unique_count.cpu().numpy()
        uniq.append(np.diff(uc))
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # CUDA graphs per index batch, so no host launch gap enters the events:
    # the headline loop replays one graph holding the whole step (forward then
    # backward, no stage events, so the backward's kernels keep their
    # programmatic overlap); a second loop replays separate forward and
    # backward graphs for the forward/backward split; a third replays
    # backward graphs with an event after every kernel for the per-kernel
    # roofline.
    def capture(traced):
        tbe.trace_enable(traced)
        out_graphs = []
        for k in range(N_BATCHES):
            d = dev_in[k]
            gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(gf):
                tbe.tbe_forward(plan, weights, d["indices"], d["offsets"], p0.B, d["psw"], out=out, dev_status=status,
                                path=path)
            with torch.cuda.graph(gb):
                tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p0.B, d["psw"], bufs=bufs,
                                 dev_status=status, want_run_starts=False, want_sorted_positions=False)
            out_graphs.append((gf, gb))
        return out_graphs

    def capture_steps():
        tbe.trace_enable(False)
        out_graphs = []
        for k in range(N_BATCHES):
            d = dev_in[k]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                tbe.tbe_forward(plan, weights, d["indices"], d["offsets"], p0.B, d["psw"], out=out, dev_status=status,
                                path=path)
                tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p0.B, d["psw"], bufs=bufs,
                                 dev_status=status, want_run_starts=False, want_sorted_positions=False)
            out_graphs.append(g)
        return out_graphs

    step_graphs = capture_steps()

    # the same step with the backward's index stages (tbe_backward_index: no
    # grad_out needed) on a second stream beside the forward, and the
    # reduction (tbe_backward_reduce) after both
    obufs = tbe.BackwardBuffers(plan, p0.B, nmax, device=dev)
    side = torch.cuda.Stream(device=dev)

    def capture_overlap():
        tbe.trace_enable(False)
        out_graphs = []
        for k in range(N_BATCHES):
            d = dev_in[k]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cur = torch.cuda.current_stream()
                side.wait_stream(cur)
                with torch.cuda.stream(side):
                    tbe.tbe_backward_index(plan, d["indices"], d["offsets"], p0.B, d["psw"], bufs=obufs,
                                           dev_status=status, want_run_starts=False, want_sorted_positions=False,
                                           stream=side)
                tbe.tbe_forward(plan, weights, d["indices"], d["offsets"], p0.B, d["psw"], out=out, dev_status=status,
                                path=path, stream=cur)
                cur.wait_stream(side)
                tbe.tbe_backward_reduce(plan, d["grad"], obufs, per_sample_weights=d["psw"], dev_status=status,
                                        stream=cur)
            out_graphs.append(g)
        return out_graphs

    overlap_graphs = capture_overlap()
    # exact row-wise Adagrad step on the backward's outputs (timed on its own,
    # after the backward of the same batch, outside the headline step);
    # captured before the traced graphs, which must be the last traced capture
    total_rows = int(p0.table_row_base[-1])
    momentum = torch.zeros(total_rows, dtype=torch.float32, device=dev)
    upd_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(upd_graph):
        tbe.tbe_exact_update(plan, weights, bufs, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, OPT_LR, OPT_EPS,
                             momentum=momentum, dev_status=status)
    # the same Adagrad step fused into the backward (tbe_backward_update), for
    # layouts whose rows have at most 128 columns
    fused_graphs = []
    if int(p0.D.max()) <= 128:
        fbufs = tbe.BackwardBuffers(plan, p0.B, nmax, device=dev, row_grads_capacity=0)
        for k in range(N_BATCHES):
            d = dev_in[k]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                tbe.tbe_backward_update(plan, weights, tbe.TBE_OPT_EXACT_ROWWISE_ADAGRAD, OPT_LR, d["grad"],
                                        d["indices"], d["offsets"], p0.B, d["psw"], eps=OPT_EPS, momentum=momentum,
                                        bufs=fbufs, dev_status=status, want_run_starts=False,
                                        want_sorted_positions=False)
            fused_graphs.append(g)
    graphs = capture(False)
    traced_graphs = capture(True)
    for k in range(args.warmup):
        flush(k)
        step_graphs[k % N_BATCHES].replay()
        graphs[k % N_BATCHES][0].replay()
        graphs[k % N_BATCHES][1].replay()
        traced_graphs[k % N_BATCHES][1].replay()
        upd_graph.replay()
        if fused_graphs:
            fused_graphs[k % N_BATCHES].replay()
    torch.cuda.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    fwd_ms, bwd_ms, step_ms, stage = [], [], [], {}
    t_wall0 = time.perf_counter()
    for k in range(args.steps):  # headline: the whole step as one graph
        flush(k)
        e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        e0.record(stream)
        step_graphs[k % N_BATCHES].replay()
        e1.record(stream)
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    for k in range(args.steps):  # forward / backward split (separate graphs: each carries one graph launch)
        flush(k)
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        gf, gb = graphs[k % N_BATCHES]
        e0.record(stream)
        gf.replay()
        e1.record(stream)
        gb.replay()
        e2.record(stream)
        e2.synchronize()
        fwd_ms.append(e0.elapsed_time(e1))
        bwd_ms.append(e1.elapsed_time(e2))
    torch.cuda.synchronize()
    bwd_kernels = []  # the backward's kernel launches per step, from its trace
    for k in range(args.steps):  # per-kernel stage times (an event after every kernel)
        flush(k)
        traced_graphs[k % N_BATCHES][1].replay()
        trace = tbe.trace_read()
        for name, ms in trace:
            stage.setdefault(name, []).append(ms)
        bwd_kernels.append(sum(1 for name, _ in trace if name.startswith("bwd_")
                               and name not in ("bwd_memset", "bwd_empty")))
    torch.cuda.synchronize()
    upd_ms = []
    for k in range(args.steps):  # optimizer step after the backward of the same batch
        flush(k)
        graphs[k % N_BATCHES][1].replay()
        e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        e0.record(stream)
        upd_graph.replay()
        e1.record(stream)
        e1.synchronize()
        upd_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    fused_ms = []
    for k in range(args.steps if fused_graphs else 0):  # backward + Adagrad step as one call
        flush(k)
        e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        e0.record(stream)
        fused_graphs[k % N_BATCHES].replay()
        e1.record(stream)
        e1.synchronize()
        fused_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    overlap_ms = []
    for k in range(args.warmup):
        flush(k)
        overlap_graphs[k % N_BATCHES].replay()
    torch.cuda.synchronize()
    for k in range(args.steps):  # the step with the index stages beside the forward
        flush(k)
        e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        e0.record(stream)
        overlap_graphs[k % N_BATCHES].replay()
        e1.record(stream)
        e1.synchronize()
        overlap_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    warm_ms = []
    for k in range(args.steps):  # the same step graphs with the L2 left warm by the previous replay
        e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        e0.record(stream)
        step_graphs[k % N_BATCHES].replay()
        e1.record(stream)
        e1.synchronize()
        warm_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    control = None
    if args.workload == WORKLOAD:
        control = run_uniform_control(args, tbe, torch, plan, weights, out, bufs, status, dev, flush, stream)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    tbe.trace_enable(False)
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    eff = [effective_bytes(probs[k % N_BATCHES], uniq[k % N_BATCHES]) for k in range(args.steps)]
    fwd_bytes = sum(f for f, _ in eff)
    bwd_bytes = sum(b for _, b in eff)
    comp = [compulsory_bytes(probs[k % N_BATCHES], uniq[k % N_BATCHES]) for k in range(args.steps)]
    fwd_comp = sum(f for f, _ in comp)
    bwd_comp = sum(b for _, b in comp)
    lookups = sum(probs[k % N_BATCHES].N for k in range(args.steps))
    tot_s = sum(step_ms) / 1e3

    # dominant kernel: the forward gather against each backward kernel (the
    # trace holds one event per launch; the radix passes share one name)
    per_kernel = {"fwd_gather": float(np.mean(fwd_ms))}
    for name, v in stage.items():
        if name.startswith("bwd_") and name != "bwd_memset":
            per_kernel[name] = float(np.mean(v))
    U_mean = float(np.mean([u.sum() for u in uniq]))
    kb = kernel_bytes(p0, U_mean)
    kb["fwd_gather"] = float(np.mean([f for f, _ in eff]))
    dom = max(per_kernel, key=lambda n: per_kernel[n])
    peak, peak_kind = load_peaks()
    achieved = kb[dom] / (per_kernel[dom] * 1e-3) / 1e9

    upd_bytes = float(np.mean([optimizer_bytes(probs[k % N_BATCHES], uniq[k % N_BATCHES])
                               for k in range(args.steps)]))
    upd_mean = float(np.mean(upd_ms))
    optimizer = dict(kind="exact_rowwise_adagrad", lr=OPT_LR, eps=OPT_EPS, ms=upd_mean,
                     GBps=upd_bytes / (upd_mean * 1e-3) / 1e9, bytes_per_launch=upd_bytes,
                     frac=upd_bytes / (upd_mean * 1e-3) / 1e9 / peak, peak=peak, peak_kind=f"{peak_kind} (copy)",
                     traffic=traffic_from_profiles("exact_update"),
                     placement="timed alone right after the backward of the same batch (row gradients still in L2, "
                               "tables and momentum flushed with the step's L2 flush)")
    if fused_ms:
        optimizer["fused"] = dict(
            ms=float(np.mean(fused_ms)), separate_ms=float(np.mean(bwd_ms)) + upd_mean,
            note="tbe_backward_update: the same step applied where each row gradient is finished inside the "
                 "backward (no row gradients written); separate_ms = backward graph + update graph, each after "
                 "its own L2 flush")

    # e2e through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, tbe, torch, plan, probs, weights, out, bufs, status, dev, flush, uniq)

    res = dict(
        metric=METRIC,
        value=(fwd_bytes + bwd_bytes) / tot_s / 1e9,
        unit="GB/s",
        lookups_per_s_M=lookups / tot_s / 1e6,
        fwd=dict(GBps=fwd_bytes / (sum(fwd_ms) / 1e3) / 1e9, ms=float(np.mean(fwd_ms)),
                 Mlookups_per_s=lookups / (sum(fwd_ms) / 1e3) / 1e6,
                 pct_of_8TBs=100 * fwd_bytes / (sum(fwd_ms) / 1e3) / 1e9 / NOMINAL_HBM_GBS),
        bwd=dict(GBps=bwd_bytes / (sum(bwd_ms) / 1e3) / 1e9, ms=float(np.mean(bwd_ms)),
                 Mlookups_per_s=lookups / (sum(bwd_ms) / 1e3) / 1e6,
                 pct_of_8TBs=100 * bwd_bytes / (sum(bwd_ms) / 1e3) / 1e9 / NOMINAL_HBM_GBS),
        pct_of_8TBs=100 * (fwd_bytes + bwd_bytes) / tot_s / 1e9 / NOMINAL_HBM_GBS,
        pct_of_measured_peak=100 * (fwd_bytes + bwd_bytes) / tot_s / 1e9 / peak,
        compulsory=dict(GBps=(fwd_comp + bwd_comp) / tot_s / 1e9,
                        fwd_GBps=fwd_comp / (sum(fwd_ms) / 1e3) / 1e9,
                        bwd_GBps=bwd_comp / (sum(bwd_ms) / 1e3) / 1e9,
                        note="each distinct row and each output-gradient row once, plus ids, weights, "
                             "offsets and outputs (compulsory_bytes)"),
        stages_ms={k: float(np.mean(v)) for k, v in stage.items()},
        n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=float(np.mean(step_ms)),
        spread=dict(step=spread(step_ms), fwd=spread(fwd_ms), bwd=spread(bwd_ms)),
        overlap=dict(step=spread(overlap_ms), GBps=(fwd_bytes + bwd_bytes) / (sum(overlap_ms) / 1e3) / 1e9,
                     note="the same step with the backward's index stages (tbe_backward_index) on a second stream "
                          "beside the forward and the reduction (tbe_backward_reduce) after both; the headline "
                          "value keeps the forward and the whole backward in sequence"),
        warm_l2=dict(step=spread(warm_ms), GBps=(fwd_bytes + bwd_bytes) / (sum(warm_ms) / 1e3) / 1e9,
                     note="the step graphs replayed back to back with no L2 flush"),
        wall_s=t_wall,
        higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="f32", data="synthetic",
        config=dict(workload=WORKLOAD_DESC if args.workload == WORKLOAD else f"{args.workload}: {p0.recipe}",
                    global_batch=p0.B * world, tables=p0.T,
                    lookups_per_step=int(np.mean([p.N for p in probs])), index_batches=N_BATCHES,
                    l2="flushed before every step (256 MB write + 256 MB read of another buffer, outside the step events)",
                    table_dtype="/".join(sorted({DT_NAMES[int(d)] for d in p0.weights_dtype})), accumulate="f32",
                    out_dtype=DT_NAMES[int(p0.out_dtype)], index_bits=8 * INDEX_BYTES,
                    parallelism=f"replicas x{world}"),
        roofline=roofline_entry(dom, kb[dom], per_kernel[dom], achieved, peak, peak_kind),
        optimizer=optimizer,
        clocks=clocks,
        gpu_launches=args.steps + sum(bwd_kernels),
        launch="one CUDA graph per step (forward then backward); backward kernels chained with programmatic dependent launch",
        tuning=tuning,
    )
    if e2e is not None:
        res["e2e"] = e2e
    if control is not None:
        res["control_uniform"] = control
    return res, (fwd_bytes + bwd_bytes), tot_s, lookups


# what the ncu captures of the dominant kernels show limits them (mid-size
# skewed workload), for the roofline entry
LIMITERS = {
    "fwd_gather": "issue and dependent-load latency (DRAM bytes equal the compulsory bytes; DRAM and L2 "
                  "throughput far below peak)",
    "bwd_reduce": "L2 latency of the bag -> grad_out chain (grad_out and the row gradients stay in L2; DRAM "
                  "traffic is a few per cent of the algorithmic bytes)",
}


def roofline_entry(kernel, nbytes, launch_ms, achieved, peak, peak_kind):
    """Roofline of the dominant kernel.  `achieved` is the effective rate
    (algorithmic bytes per launch / launch time); `dram_frac` is the HBM
    side: the ncu-measured DRAM bytes of a launch (when the committed record
    matches the current source) over the same time, against the same peak."""
    traffic = traffic_from_profiles(kernel)
    dram = None if traffic is None else traffic / (launch_ms * 1e-3) / 1e9
    return dict(bound="hbm", kernel=kernel, achieved=achieved, achieved_kind="effective (algorithmic bytes)",
                peak=peak, unit="GB/s", frac=achieved / peak, peak_kind=f"{peak_kind} (copy)",
                bytes_per_launch=nbytes, launch_ms=launch_ms, traffic=traffic,
                dram_GBps=dram, dram_frac=None if dram is None else dram / peak,
                limiter=LIMITERS.get(kernel))


def run_uniform_control(args, tbe, torch, plan, weights, out, bufs, status, dev, flush, stream):
    """The mid-size workload's tables, bag lengths and empty bags with
    uniform ids (no skew): forward and backward graphs timed like the
    headline's split."""
    from tbe_inputs import make_config

    probs = [make_config("mid_uniform", batch=k) for k in range(2)]
    outs = []
    for p in probs:
        d = dict(indices=torch.from_numpy(p.indices).to(dev), offsets=torch.from_numpy(p.offsets).to(dev),
                 grad=torch.from_numpy(p.grad_out).to(dev))
        if p.N > bufs.N:
            return None
        gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        tbe.tbe_forward(plan, weights, d["indices"], d["offsets"], p.B, out=out, dev_status=status)
        tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, bufs=bufs, dev_status=status,
                         want_run_starts=False, want_sorted_positions=False)
        torch.cuda.synchronize()
        U = np.diff(bufs.unique_count.cpu().numpy())
        with torch.cuda.graph(gf):
            tbe.tbe_forward(plan, weights, d["indices"], d["offsets"], p.B, out=out, dev_status=status)
        with torch.cuda.graph(gb):
            tbe.tbe_backward(plan, d["grad"], d["indices"], d["offsets"], p.B, bufs=bufs, dev_status=status,
                             want_run_starts=False, want_sorted_positions=False)
        outs.append((p, d, gf, gb, U))
    fwd_ms, bwd_ms, fb, bb = [], [], 0, 0
    for k in range(args.warmup + args.steps):
        p, d, gf, gb, U = outs[k % len(outs)]
        flush(k)
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        gf.replay()
        e1.record(stream)
        gb.replay()
        e2.record(stream)
        e2.synchronize()
        if k >= args.warmup:
            fwd_ms.append(e0.elapsed_time(e1))
            bwd_ms.append(e1.elapsed_time(e2))
            f, b = effective_bytes(p, U)
            fb += f
            bb += b
    return dict(workload="mid_uniform: the mid-size tables, bag lengths and empty bags with uniform ids",
                lookups=int(np.mean([o[0].N for o in outs])), unique_rows=int(np.mean([o[4].sum() for o in outs])),
                fwd=dict(spread(fwd_ms), GBps=fb / (sum(fwd_ms) / 1e3) / 1e9),
                bwd=dict(spread(bwd_ms), GBps=bb / (sum(bwd_ms) / 1e3) / 1e9))


def run_e2e(args, tbe, torch, plan, probs, weights, out, bufs, status, dev, flush, uniq):
    """Same metric through the public API with pinned host buffers: the
    timed step copies the batch in, runs forward + backward, and reads the
    results back (pooled output, unique rows and their row gradients)."""
    host = []
    for p in probs:
        host.append(dict(indices=torch.from_numpy(p.indices.astype(IDX_NP[INDEX_BYTES])).pin_memory(),
                         offsets=torch.from_numpy(p.offsets.astype(IDX_NP[INDEX_BYTES])).pin_memory(),
                         grad=torch.from_numpy(p.grad_out).pin_memory()))
    nmax = max(p.N for p in probs)
    idt = torch.int32 if INDEX_BYTES == 4 else torch.int64
    d_ind = torch.empty(nmax, dtype=idt, device=dev)
    d_off = torch.empty(probs[0].offsets.shape[0], dtype=idt, device=dev)
    d_grad = torch.empty(probs[0].grad_out.shape, dtype=torch.float32, device=dev)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_rows = torch.empty(nmax, dtype=torch.int64).pin_memory()
    h_rg = torch.empty(bufs.row_grads.numel(), dtype=torch.float32).pin_memory()
    h_uc = torch.empty(plan.T + 1, dtype=torch.int64).pin_memory()
    D = int(probs[0].D[0])
    times, bin_, bout, nbytes = [], 0, 0, 0
    for k in range(args.warmup + args.steps):
        p = probs[k % N_BATCHES]
        h = host[k % N_BATCHES]
        flush(k)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        n = p.N
        d_ind[:n].copy_(h["indices"], non_blocking=True)
        d_off.copy_(h["offsets"], non_blocking=True)
        d_grad.copy_(h["grad"], non_blocking=True)
        tbe.tbe_forward(plan, weights, d_ind[:n], d_off, p.B, None, out=out, dev_status=status)
        tbe.tbe_backward(plan, d_grad, d_ind[:n], d_off, p.B, None, bufs=bufs, dev_status=status,
                         want_run_starts=False, want_sorted_positions=False)
        h_out.copy_(out, non_blocking=True)
        h_uc.copy_(bufs.unique_count, non_blocking=True)
        torch.cuda.synchronize()
        U = int(h_uc[-1])
        h_rows[:U].copy_(bufs.unique_rows[:U], non_blocking=True)
        h_rg[:U * D].copy_(bufs.row_grads[:U * D], non_blocking=True)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        if k >= args.warmup:
            times.append(t1 - t0)
            bi = (n + p.offsets.shape[0]) * INDEX_BYTES + p.grad_out.nbytes
            bo = out.numel() * out.element_size() + h_uc.numel() * 8 + U * 8 + U * D * 4
            bin_ += bi
            bout += bo
            f, b = effective_bytes(p, uniq[k % N_BATCHES])
            nbytes += f + b
    steps = len(times)
    return dict(value=nbytes / sum(times) / 1e9, unit="GB/s", h2d_bytes_per_step=bin_ // steps,
                d2h_bytes_per_step=bout // steps, ms_per_step=1e3 * float(np.mean(times)))


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and CPU baseline)
# ---------------------------------------------------------------------------

def oracle_steps(workload, seconds=None, steps=None, nthreads=0):
    """Time the oracle's forward + backward on full batches of the workload.
    Returns (effective bytes, seconds, lookups, steps, threads)."""
    import oracle
    from tbe_inputs import make_config, materialize_weights

    nthreads = nthreads or (os.cpu_count() or 1)
    probs = [make_config(workload, batch=k) for k in range(N_BATCHES)]
    w = materialize_weights(probs[0]).numpy()
    lay = probs[0].layout_arrays()
    done, tot_s, tot_b, tot_n = 0, 0.0, 0, 0
    while True:
        p = probs[done % N_BATCHES]
        t0 = time.perf_counter()
        st, _, _ = oracle.forward(lay, w, p.indices, p.offsets, p.B, p.per_sample_weights, nthreads=nthreads)
        idx = oracle.backward_indexing(lay, p.indices, p.offsets, p.B)
        st2, _, _, _ = oracle.backward_values(lay, p.offsets, p.B, p.grad_out, idx, p.per_sample_weights,
                                              nthreads=nthreads)
        dt = time.perf_counter() - t0
        assert st == 0 and st2 == 0
        f, b = effective_bytes(p, np.diff(idx["unique_count"]))
        tot_s += dt
        tot_b += f + b
        tot_n += p.N
        done += 1
        if steps is not None and done >= steps:
            break
        if steps is None and tot_s >= seconds:
            break
    return tot_b, tot_s, tot_n, done, nthreads


def batch_size(workload):
    from tbe_inputs import make_config

    return int(make_config(workload, with_grad=False).B)


def cpu_baseline(workload, seconds, single_steps=2):
    """The oracle on the host cores: full forward+backward batches for about
    `seconds` on every core, then `single_steps` batches on one thread."""
    b, s, n, steps, cores = oracle_steps(workload, seconds=seconds)
    b1, s1, _, steps1, _ = oracle_steps(workload, steps=single_steps, nthreads=1)
    return dict(value=b / s / 1e9, unit="GB/s", cores=cores, kind="oracle",
                sample=f"{steps} full forward+backward batches of the workload ({s:.1f} s of CPU work, fp64 oracle)",
                single_thread=dict(value=b1 / s1 / 1e9, unit="GB/s", cores=1,
                                   sample=f"{steps1} batches on one thread ({s1:.1f} s)"))


def run_reference(args):
    import oracle

    oracle.load()
    oracle_steps(args.workload, steps=max(args.warmup, 0) or 1)  # warm-up (page-in, build)
    b, s, n, steps, cores = oracle_steps(args.workload, steps=args.steps)
    v = b / s / 1e9
    return dict(
        impl="reference", metric=METRIC, value=v, unit="GB/s", lookups_per_s_M=n / s / 1e6,
        n_gpus=args.gpus, steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * s / steps,
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
        config=dict(workload=WORKLOAD_DESC if args.workload == WORKLOAD else args.workload,
                    global_batch=batch_size(args.workload), parallelism="cpu"),
        cpu_baseline=dict(value=v, unit="GB/s", cores=cores, kind="oracle",
                          sample=f"{steps} full forward+backward batches of the workload (oracle, fp64)"),
        e2e=dict(value=v, unit="GB/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0),
    )


def combine_ranks(tot_s, nbytes, lookups, steps, device):
    """Whole-job figures of a multi-rank run (an initialised process group):
    the bytes and lookups of every rank over the slowest rank's timed
    seconds.  Every rank gets the same result."""
    import torch
    import torch.distributed as dist

    slowest = torch.tensor([tot_s], dtype=torch.float64, device=device)
    units = torch.tensor([nbytes, lookups], dtype=torch.float64, device=device)
    dist.all_reduce(slowest, op=dist.ReduceOp.MAX)
    dist.all_reduce(units, op=dist.ReduceOp.SUM)
    t = float(slowest[0])
    return dict(value=float(units[0]) / t / 1e9, lookups_per_s_M=float(units[1]) / t / 1e6,
                ms_per_step=1e3 * t / steps)


def main():
    global INDEX_BYTES
    args = parse_args()
    INDEX_BYTES = args.index_bits // 8
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    import torch

    if args.profile:
        print(json.dumps(run_profile(args)), flush=True)
        return
    if args.sweep:
        run_sweep(args)
        return
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res, nbytes, tot_s, lookups = run_ours(args, world, rank, local)
    if world > 1:
        res.update(combine_ranks(tot_s, nbytes, lookups, args.steps, device="cuda"))
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
