"""Throughput of the hot path on one GB300 (or N independent replicas).

A step is one pass of the whole path over the 200 000-clip workload: core
distances (exact k-NN of every clip against all clips, min_samples = 10) and
the mutual-reachability minimum spanning tree (Boruvka with the exact
shortcuts).  ``value`` is clips per second with the clips already resident in
device memory; ``e2e`` is the same metric through the public Python API with
host buffers (host->device copy of the clips and device->host copy of the
core distances and the tree inside the timed region).  A secondary line item
times exact k-NN on the 200 000 x 192 workload against its 20 000-point
subset (rows per second).

The K timed steps run without instrumentation; the same K steps then run
again with a CUDA event pair around every kernel launch, which gives the
per-kernel breakdown and the roofline of the distance tile
(``profiled_ms_per_step`` is that second pass's step time).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

``--impl reference`` times the float64 CPU oracle instead (a bounded sample of
the same workload on the host cores).  Under torchrun (N > 1) every rank runs
the full workload on its own GPU (replicas: the path needs no exchange);
rank 0 prints the line.
"""

from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MR-MST clips/s & exact k-NN rows/s; distance-tile FLOP/s vs GB300 peak"
WORKLOAD = "hdbscan_200k_d61"
KNN_WORKLOAD = "knn_200k_d192"
WORKLOAD_TEXT = ("200,000 clips x 61 fp32 features, 50 Gaussian clusters (sigma ~ U(0.5,2)), "
                 "10% uniform outliers, 1% exact duplicates, min_samples=10; core distances + "
                 "mutual-reachability MST by Boruvka with exact shortcuts")
KNN_TEXT = "200,000 points x 192 fp32 features, 100 clusters, k=10 against every 10th point (20,000)"
L2_FLUSH_BYTES = 256 << 20
# the page's "Results" quote min_cluster_size = 20
MIN_CLUSTER_SIZE = 20
# the split-product covariance: windows of 60 000 samples of a recording of
# 384 (and 64) channels, starting at an odd column
MOMENT_CHANNELS = (384, 64)
MOMENT_SAMPLES = 60000
MOMENT_OFFSET = 1001


def moment_recording(channels: int) -> np.ndarray:
    """A synthetic channel-major recording: per channel a DC level, a scale and
    white noise, seeded; 1 001 + 60 000 + 999 samples."""
    rng = np.random.default_rng(7 + channels)
    T = MOMENT_OFFSET + MOMENT_SAMPLES + 999
    scale = rng.uniform(5.0, 50.0, (channels, 1))
    level = rng.uniform(-200.0, 200.0, (channels, 1))
    return (rng.standard_normal((channels, T)) * scale + level).astype(np.float32)


# the k-NN graph consumer: 200 initial clusters (the seed count of page
# "Kilosort4 clustering and matching"), resolution 1, on the k-NN lists above
ASSIGN_CLUSTERS = 200
ASSIGN_TEXT = ("bipartite modularity assignment over the k-NN graph of the 200,000 x 192 "
               "workload (k=10 into the 20,000-point subset), 200 seeded initial clusters, "
               "gamma=1, rounds until no spike moves")
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
# FP32 FFMA: 128 lanes per SM, 2 flops per lane per clock
FP32_LANES_PER_SM = 128
# nominal dense tensor rates: TF32 1.1 PFLOP/s, BF16 2.25 PFLOP/s
TF32_PER_BF16 = 1.1 / 2.25
# DRAM bytes per step of each distance tile (all its launches in one step,
# like the roofline's achieved rate) from one one-pass ncu capture of the full
# workload (dram__bytes_read.sum + dram__bytes_write.sum), valid only while
# the kernel's sources are those the capture ran (their sha256 below);
# otherwise the line reports null.
TRAFFIC = {
    ("knn_tile", "hdbscan_200k_d61"): {
        # per step: the home pass (52.20 MB read, 3.79 MB written) and the
        # pruned second pass (83.95 MB read - the home lists it starts from
        # included - and 9.26 MB written)
        "bytes": 52.20e6 + 3.79e6 + 83.95e6 + 9.26e6,
        "sources": ("hdbscan_mst_gb300/csrc/tc_knn.cu", "hdbscan_mst_gb300/csrc/tc_pipe.cuh",
                    "hdbscan_mst_gb300/csrc/tc.cuh"),
        "sha256": "5aa1b00de8a6d67783d45effb35cf8d64ea1cf55ff642e7ac4b8bd2004b8defa",
    },
    ("boruvka_scan", "hdbscan_200k_d61"): {
        # per step: the one-sided scans of rounds 1 and 2 (55.01 + 53.26 MB
        # read) and the symmetric scans of rounds 3 and 4, home pass and
        # pruned pass each (49.22 + 51.48 + 48.69 + 49.69 MB read); under
        # 0.01 MB written in all
        "bytes": (55.01 + 53.26 + 49.22 + 51.48 + 48.69 + 49.69 + 0.006) * 1e6,
        "sources": ("hdbscan_mst_gb300/csrc/tc_scan.cu", "hdbscan_mst_gb300/csrc/tc_sym.cu",
                    "hdbscan_mst_gb300/csrc/tc_pipe.cuh", "hdbscan_mst_gb300/csrc/tc.cuh"),
        "sha256": "c6010b05c9ae77cec18fa7607374edf66545da9f3fb8398cf3876a9047ab17fe",
    },
}
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={SMI_FIELDS}", "--format=csv",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
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
            return None
        rows = [ln.strip() for ln in open(self.path) if ln.strip()]
        os.unlink(self.path)
        if len(rows) < 2:
            return None
        sms, mx, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows[1:]:
            f = [x.strip() for x in r.split(",")]
            try:
                sms.append(float(f[1].split()[0]))
                mx = float(f[2].split()[0])
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names[1:], f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------ GPU arm

def flush_l2(buf):
    buf.add_(1)


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(ws, "nccl")
    import hdbscan_mst_gb300 as H
    H.set_scan_form(args.scan_form)

    X, task = workloads.workload(args.workload)
    ms = task["min_samples"]
    d, n = X.shape
    Xd = torch.from_numpy(X).to(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        core, idx, dist_ = H.core_distances(Xd, ms)
        edges, w = H.mr_mst(Xd, core, idx, dist_)
        return core, edges, w

    # the clock sampler starts before the warm-up: nvidia-smi's start-up
    # (NVML initialisation) must not fall inside the timed steps
    clk = ClockSampler(local).__enter__()
    time.sleep(0.5)
    for _ in range(args.warmup):
        flush_l2(flush)
        step()
    torch.cuda.synchronize(device)

    def timed(fn):
        """K steps with CUDA events on the launching stream around each; L2
        flushed before each step, outside the events.  Python's garbage
        collector is paused meanwhile: a collection inside a step would leave
        the GPU waiting for the host's next launch."""
        out = []
        gc_on = gc.isenabled()
        gc.disable()
        try:
            for _ in range(args.steps):
                flush_l2(flush)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                out.append(e0.elapsed_time(e1))
        finally:
            if gc_on:
                gc.enable()
        return out

    # ---- timed region: data resident, no instrumentation
    launches0 = H.launch_count()
    barrier(dist, device)
    torch.cuda.synchronize(device)
    try:
        times = timed(step)
        torch.cuda.synchronize(device)
    finally:
        clk.__exit__(None, None, None)
    barrier(dist, device)
    launches = H.launch_count() - launches0
    rounds = H.last_mst_rounds()
    core_exact_rows = H.last_knn_exact_rows()
    core_pairs = H.last_knn_tile_pairs()
    scan_pairs = H.last_mst_scan_pairs()

    # ---- the same K steps again with an event pair around every kernel
    # launch: per-kernel times for the breakdown and the roofline
    H.profile_enable(True)
    H.profile_read()
    prof_times = timed(step)
    prof = H.profile_read()
    H.profile_enable(False)
    clocks = clk.summary()
    total_ms = max_over_ranks(dist, sum(times), device)
    ms_per_step = total_ms / args.steps
    value = ws * n * args.steps / (total_ms / 1e3)

    # ---- end to end through the public API with host buffers
    Xh = torch.from_numpy(X).pin_memory()
    e2e_times = []
    gc_on = gc.isenabled()
    gc.disable()
    for i in range(0 if args.skip_e2e else args.warmup + args.steps):
        flush_l2(flush)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        core, edges, w = H.hdbscan_mst(Xh, ms)  # host in, host out
        t1 = time.perf_counter()
        if i >= args.warmup:
            e2e_times.append((t1 - t0) * 1e3)
    if gc_on:
        gc.enable()
    e2e_total = max_over_ranks(dist, sum(e2e_times), device)

    # ---- the back half on the host (labels from the tree of the last call):
    # the whole method, as the page times it, is the e2e call plus this
    label_times, labels = [], None
    for i in range(0 if args.skip_e2e else 3):
        t0 = time.perf_counter()
        labels = H.hdbscan_labels(edges, w, MIN_CLUSTER_SIZE)
        label_times.append((time.perf_counter() - t0) * 1e3)
    h2d = X.nbytes
    d2h = n * 4 + (n - 1) * 12  # core distances, (lo, hi) pairs, weights

    # ---- secondary: exact k-NN rows/s on the 200k x 192 workload
    Xk, tk = workloads.workload(KNN_WORKLOAD if not args.skip_knn else "knn_1416_d102")
    Yk = workloads.subset_columns(Xk, tk["y_stride"])
    Xkd, Ykd = torch.from_numpy(Xk).to(device), torch.from_numpy(Yk).to(device)
    for _ in range(args.warmup):
        flush_l2(flush)
        H.knn(Xkd, Ykd, tk["k"])
    torch.cuda.synchronize(device)
    kt = timed(lambda: H.knn(Xkd, Ykd, tk["k"]))
    knn_exact_rows = H.last_knn_exact_rows()
    knn_pairs = H.last_knn_tile_pairs()
    H.profile_enable(True)
    H.profile_read()
    timed(lambda: H.knn(Xkd, Ykd, tk["k"]))
    kprof = H.profile_read()
    H.profile_enable(False)
    k_total = max_over_ranks(dist, sum(kt), device)

    # ---- the k-NN graph consumer on the GPU's own lists: bipartite
    # modularity assignment of the spikes and the subset, 200 initial clusters
    a_item = None
    if not args.skip_knn:
        gi_k, _ = H.knn(Xkd, Ykd, tk["k"])
        mk = Yk.shape[1]
        r0 = torch.from_numpy(np.random.default_rng(12).integers(0, ASSIGN_CLUSTERS, mk)
                              .astype(np.int32)).to(device)
        res = {}

        def assign_call():
            res["out"] = H.bipartite_assign(gi_k, mk, r0, ASSIGN_CLUSTERS, 1.0)

        for _ in range(args.warmup):
            flush_l2(flush)
            assign_call()
        torch.cuda.synchronize(device)
        at = timed(assign_call)
        a_rounds, a_moved = res["out"][2], res["out"][3]
        H.profile_enable(True)
        H.profile_read()
        timed(assign_call)
        aprof = H.profile_read()
        H.profile_enable(False)
        a_total = max_over_ranks(dist, sum(at), device)
        a_item = {"metric": "bipartite assignment spikes/s (all rounds of one call)",
                  "workload": ASSIGN_TEXT,
                  "value": round(ws * Xk.shape[1] * args.steps / (a_total / 1e3), 1),
                  "unit": "spikes/s", "ms_per_call": round(a_total / args.steps, 3),
                  "rounds": a_rounds, "moved": a_moved,
                  "kernel_ms_per_call": {
                      k_: {"ms": round(v[0] / args.steps, 4), "launches": v[1] / args.steps}
                      for k_, v in sorted(aprof.items(), key=lambda kv: -kv[1][0])}}

    # ---- the split-product covariance of a 384-channel window of 60 000
    # samples (the configuration the covariance page reports), 64 channels too
    m_items = None
    if not args.skip_knn:
        m_items = {}
        for mc in MOMENT_CHANNELS:
            Xm = torch.from_numpy(moment_recording(mc)).to(device)
            t0m = MOMENT_OFFSET
            res_m = {}

            def moment_call():
                res_m["out"] = H.second_moment(Xm, t0m, MOMENT_SAMPLES, centred=True,
                                               out=res_m.get("out"))

            for _ in range(args.warmup):
                flush_l2(flush)
                moment_call()
            torch.cuda.synchronize(device)
            mt = timed(moment_call)
            H.profile_enable(True)
            H.profile_read()
            timed(moment_call)
            mprof = H.profile_read()
            H.profile_enable(False)
            m_total = max_over_ranks(dist, sum(mt), device)
            ms_call = m_total / args.steps
            splits = -(-MOMENT_SAMPLES // 4096)
            cpad = -(-mc // 128) * 128
            blocks = cpad // 128
            pairs = blocks * (blocks + 1) // 2
            # algorithmic work: the upper triangle's products, 2 flop per
            # (channel pair, sample); issued: 3 products over whole 128 x 128
            # tiles and 4096-sample splits
            alg_flop = 2.0 * mc * (mc + 1) / 2 * MOMENT_SAMPLES
            issued = 3 * 2.0 * pairs * 128 * 128 * 4096 * splits
            prod_ms = mprof.get("moment_product", (float("nan"), 1))[0] / args.steps
            m_items[f"{mc}ch"] = {
                "metric": "covariance windows/s", "channels": mc, "samples": MOMENT_SAMPLES,
                "value": round(ws * args.steps / (m_total / 1e3), 1), "unit": "windows/s",
                "ms_per_call": round(ms_call, 4),
                "input_gb_per_s": round(4.0 * mc * MOMENT_SAMPLES / (ms_call / 1e3) / 1e9, 1),
                "kernel_ms_per_call": {
                    k_: {"ms": round(v[0] / args.steps, 4), "launches": v[1] / args.steps}
                    for k_, v in sorted(mprof.items(), key=lambda kv: -kv[1][0])},
                "product_tflops_algorithmic": round(alg_flop / (prod_ms / 1e3) / 1e12, 1),
                "product_tflops_issued": round(issued / (prod_ms / 1e3) / 1e12, 1)}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    max_mhz = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * max_mhz * 1e6 / 1e12  # TFLOP/s
    bf16 = peaks.get("bf16_tflops")
    tf32_peak = bf16 * TF32_PER_BF16 if bf16 else FALLBACK_BF16_TFLOPS * TF32_PER_BF16
    tf32_basis = ("measured bf16 burst x nominal tf32/bf16 (1.1/2.25)" if bf16 else
                  "fallback bf16 x nominal tf32/bf16 (1.1/2.25)")

    def engine_of(d_, knn=False):
        """The tensor-core operand form the default engine uses for d features
        (padded to whole 32-feature slabs): two-part FP16 at 64, and for the
        k-NN tile also at 128 and 192; else three-pass TF32."""
        if d_ > 192:
            return "fp32"
        dk = (d_ + 31) // 32 * 32
        return "f16" if dk == 64 or (knn and dk in (128, 192)) else "tf32"

    def roofline(prof_, name, d_, pairs, dense_pairs, engine, workload=None):
        """A distance tile: algorithmic flops 2 d per (row, column) pair the
        tile evaluated (blocks the bounds prune are not evaluated), over the
        tile's time per step (all its launches: the same ratio as a launch's
        average); traffic, the measured DRAM bytes per launch (the step's
        bytes over its launches), with the step's total beside it."""
        if name not in prof_:
            return None
        tot_ms, nl = prof_[name]
        step_s = tot_ms / args.steps / 1e3
        flops = 2.0 * d_ * pairs
        ach = flops / step_s / 1e12
        common = {"avg_launch_ms": round(tot_ms / nl, 3), "launches_per_step": nl / args.steps,
                  "ms_per_step": round(step_s * 1e3, 3), "flops_per_step": flops,
                  "pairs_evaluated": int(pairs), "pairs_dense": int(dense_pairs),
                  "evaluated_frac": round(pairs / dense_pairs, 4) if dense_pairs else None,
                  "dense_equivalent_tflops": round(2.0 * d_ * dense_pairs / step_s / 1e12, 1)}
        if engine in ("f16", "tf32"):
            if engine == "f16":
                dk = (d_ + 31) // 32 * 32  # padded halves per part
                peak = bf16 if bf16 else FALLBACK_BF16_TFLOPS
                basis = ("measured bf16 burst (dense fp16 runs at the bf16 rate)" if bf16 else
                         "fallback bf16 (dense fp16 runs at the bf16 rate)")
                eng = "tcgen05 kind::f16, two-part fp16 operands (3 products)"
            else:
                dk = (d_ + 31) // 32 * 32  # padded features: whole 32-feature slabs
                peak, basis = tf32_peak, tf32_basis
                eng = "tcgen05 kind::tf32 (3 products)"
            issued = 3 * 2.0 * dk * pairs / step_s / 1e12
            # DRAM bytes per launch, like achieved: the step's measured bytes
            # over its launches of the tile
            tstep = traffic_for(name, workload)
            tlaunch = round(tstep / (nl / args.steps)) if tstep is not None else None
            return {"kernel": name, "engine": eng, "bound": "tensor",
                    "achieved": round(ach, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                    "frac": round(ach / peak, 4), "traffic": tlaunch,
                    "traffic_per_step": tstep,
                    "peak_basis": basis, "issued_tflops": round(issued, 1),
                    "issued_frac": round(issued / peak, 4),
                    "fp32_alu_equiv_frac": round(ach / fp32_peak, 4), **common}
        return {"kernel": name, "engine": "FP32 FFMA", "bound": "alu", "achieved": round(ach, 2),
                "peak": round(fp32_peak, 2), "unit": "TFLOP/s", "frac": round(ach / fp32_peak, 4),
                "traffic": None,
                "peak_basis": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x {max_mhz:.0f} MHz",
                **common}

    # core distances: every clip against every clip, pruned by the pivot bounds;
    # the Boruvka scan: every active clip against the clips of other components
    knn_tile_roof = roofline(prof, "knn_tile", d, core_pairs, float(n) * n, engine_of(d, knn=True),
                             args.workload)
    scan_dense = float(sum(a for a, _, _ in rounds)) * n
    scan_roof = roofline(prof, "boruvka_scan", d, scan_pairs, scan_dense, engine_of(d),
                         args.workload)
    # the line's roofline is the dominant kernel's (the larger share of the step)
    cands = [r for r in (scan_roof, knn_tile_roof) if r is not None]
    main_roof = max(cands, key=lambda r: r["ms_per_step"]) if cands else None
    knn_roof = roofline(kprof, "knn_tile", Xk.shape[0], knn_pairs,
                        float(Xk.shape[1]) * Yk.shape[1], engine_of(Xk.shape[0], knn=True),
                        KNN_WORKLOAD if not args.skip_knn else None)
    breakdown = {k: {"ms_per_step": round(v[0] / args.steps, 3), "launches_per_step": v[1] / args.steps}
                 for k, v in sorted(prof.items(), key=lambda kv: -kv[1][0])}
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "clips/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT if args.workload == WORKLOAD else args.workload,
                   "n": n, "d": d, "min_samples": ms,
                   "l2": "flushed between timed steps (256 MiB write outside the events)",
                   "scan_form": args.scan_form,
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": main_roof,
        "rooflines": {"boruvka_scan": scan_roof, "knn_tile": knn_tile_roof},
        "kernel_ms_per_step": breakdown,
        "profiled_ms_per_step": round(sum(prof_times) / args.steps, 3),
        "step_ms": {"min": round(min(times), 3), "median": round(statistics.median(times), 3),
                    "max": round(max(times), 3)},
        "core_exact_rows": core_exact_rows,
        "boruvka_rounds": [{"scanned": a, "scanned_frac": round(a / n, 4), "edges": e,
                            "exact_rows": x} for a, e, x in rounds],
        "gpu_launches": launches,
        "e2e": None if args.skip_e2e else {
            "value": round(ws * n * args.steps / (e2e_total / 1e3), 1), "unit": "clips/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "clocks": clocks,
        "hdbscan": None if args.skip_e2e else {
            "metric": "HDBSCAN clips/s (core distances + MR-MST on the GPU through the host API, "
                      "labels on the host)",
            "value": round(n / ((e2e_total / max(len(e2e_times), 1) + min(label_times)) / 1e3), 1),
            "unit": "clips/s", "labels_ms": round(min(label_times), 3),
            "min_cluster_size": MIN_CLUSTER_SIZE,
            "clusters": int(len(set(labels.tolist()) - {-1})),
            "noise_frac": round(float((labels < 0).mean()), 4)},
        "knn": None if args.skip_knn else {"metric": "exact k-NN rows/s", "workload": KNN_TEXT,
                "value": round(ws * Xk.shape[1] * args.steps / (k_total / 1e3), 1),
                "unit": "rows/s", "ms_per_step": round(k_total / args.steps, 3),
                "exact_rows": knn_exact_rows,
                "roofline": knn_roof},
        "assign": a_item,
        "covariance": m_items,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return line


def sources_sha256(paths) -> str:
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(kernel: str, workload: str):
    """Measured DRAM bytes per step, or None when not measured for this
    kernel and workload or the kernel changed since the capture."""
    rec = TRAFFIC.get((kernel, workload))
    if rec is None:
        return None
    try:
        if sources_sha256(rec["sources"]) != rec["sha256"]:
            return None
    except OSError:
        return None
    return rec["bytes"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p))
        except ValueError:
            pass
    return {}


# ------------------------------------------------------------------ oracle (CPU) arm

def oracle_sample_rate(n_sample: int):
    """Time the oracle (core distances + dense Prim) on the first ``n_sample``
    clips of the workload; return (seconds, clips/s at the full size by the
    oracle's O(n^2) cost, threads)."""
    import oracle
    X, task = workloads.workload(WORKLOAD)
    n = X.shape[1]
    Xs = np.ascontiguousarray(X[:, :n_sample])
    t0 = time.perf_counter()
    core = oracle.core_distances(Xs, task["min_samples"])
    oracle.prim_mst(Xs, core)
    dt = time.perf_counter() - t0
    full_seconds = dt * (n / n_sample) ** 2
    return dt, n / full_seconds, oracle.threads()


# One bounded sample of the workload for both CPU legs (the cpu_baseline key
# of the GPU line and the reference arm): the first 20 000 clips, about 1.6 s
# on 16 host cores (26 core-seconds), scaled to 200 000 by the oracle's
# O(n^2) cost.
ORACLE_SAMPLE = 20000


def cpu_baseline(args, n_sample: int = ORACLE_SAMPLE):
    dt, rate, thr = oracle_sample_rate(n_sample)
    return {"value": round(rate, 2), "unit": "clips/s", "cores": thr, "kind": "oracle",
            "sample": (f"oracle core distances + dense Prim on the first {n_sample} of the "
                       f"200,000 clips ({dt:.1f} s), scaled to 200,000 by the oracle's "
                       f"O(n^2) cost"),
            "extrapolated_from": n_sample, "extrapolation": "(200000 / n_sample)^2",
            "measured_sample_clips_per_s": round(n_sample / dt, 1)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    n_sample = ORACLE_SAMPLE
    for _ in range(args.warmup):
        oracle_sample_rate(n_sample)
    secs, thr = [], 0
    for _ in range(args.steps):
        dt, _, thr = oracle_sample_rate(n_sample)
        secs.append(dt)
    value = args.steps * 200000 / (sum(secs) * (200000 / n_sample) ** 2)
    sample = (f"oracle core distances + dense Prim on the first {n_sample} of the 200,000 clips "
              f"per step, scaled to 200,000 by the oracle's O(n^2) cost")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "clips/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(secs) / args.steps * (200000 / n_sample) ** 2, 1),
        "measured_ms_per_step": round(1e3 * sum(secs) / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT, "n": 200000, "d": 61, "min_samples": 10,
                   "sample_clips": n_sample},
        "cpu_baseline": {"value": round(value, 2), "unit": "clips/s", "cores": thr,
                         "kind": "oracle", "sample": sample, "extrapolated_from": n_sample,
                         "extrapolation": "(200000 / n_sample)^2"},
        "e2e": {"value": round(value, 2), "unit": "clips/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the oracle on the host (the line omits cpu_baseline)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(
        k for k, v in workloads.WORKLOADS.items() if v["task"] == "mst"),
        help="HDBSCAN workload of the main step (profiling runs use smaller ones)")
    ap.add_argument("--skip-e2e", action="store_true", help="omit the host-buffer leg")
    ap.add_argument("--skip-knn", action="store_true", help="omit the k-NN line item")
    ap.add_argument("--scan-form", default="auto", choices=["auto", "one_sided", "symmetric"],
                    help="form of the Boruvka scan (the tree is the same; profiling of the "
                         "one-sided form)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least three untimed steps
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    main()
