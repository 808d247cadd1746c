"""Benchmark of the exact epsilon self-join on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C | --all-configs]
                    [--impl hiss|reference]

One step is the whole hot path on one synthetic workload: hiss_build (variance
order), hiss_count (grid index + count pass) and hiss_join (batched
refinement + compaction to CSR, results left on the device).  The default
workload is the largest: 5,000,000 points, 16 dimensions, i.i.d.
exponential(1) coordinates, eps set for a mean of 1,000 neighbours per point
(about 5e9 result pairs), joined in batches of at most 64 GiB of device
memory.  ``--all-configs`` prints one line per workload (1 to 5).

``value`` is result pairs per second (self pairs included) with the points
already resident in device memory; ``e2e`` is the same metric through the
host-buffer entry points (points copied in, every batch of results copied out
to pinned host memory, both inside the timed region).  The L2 cache is
flushed (a 512 MB write) before every timed step, outside the timed region.

``roofline`` is the refinement kernel's: its algorithmic FP32 work (3 flop
per pair and dimension over the dimensions each candidate pair needs with
per-pair early exit, counted exactly by hiss_work_profile outside the timed
region) per second of its CUDA-event time, against the FP32 peak (SMs from the
device properties x 128 FP32 lanes x the measured maximum SM clock x 2 flop
per fused multiply-add).  It also carries the kernel's algorithmic bytes
(query rows, candidate rows once per query tile, mask bits) at the measured
HBM bandwidth, so that the roofline time max(F/P, B/BW) is reported beside
the FP32 fraction.  ``join_roofline`` does the same for the whole step.

``--impl reference`` times the fp64 CPU oracle (plain brute force) on a
bounded sample of query rows of the same workload and reports the same
metric.  Under torchrun each rank runs an independent replica of the
workload (the join does not need a collective); ``value`` sums all ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import datagen  # noqa: E402

METRIC = "eps-self-join result pairs/s (and candidate distance evaluations/s) at 1 GB300"
UNIT = "pairs/s"
DEFAULT_CONFIG = 5
DEFAULT_BATCH_BYTES = 64 << 30         # a batch's mask, arrays and CSR stay within this
FP32_LANES_PER_SM = 128                # sm_100-family SM: 4 sub-partitions x 32 FP32 lanes
CPU_SAMPLE_COORD_OPS = 2.5e11          # cpu_baseline sample: rows x n x d (about 18 s on 16 host cores)
REF_STEP_COORD_OPS = 6e10              # --impl reference: rows x n x d per step (about 4 s)


def load_eps(cfg):
    with open(os.path.join(ROOT, "tests", "golden", "eps_configs.json")) as f:
        return json.load(f)[str(cfg)]["eps"]


def code_sha(path):
    """sha256 prefix of a source file's code: comments (from // to the end of
    a line) and blank lines left out, so that comment edits keep it."""
    import hashlib
    import re
    lines = []
    for line in open(path, encoding="utf-8"):
        line = re.sub(r"//.*$", "", line).rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def refine_traffic_per_unit(cfg):
    """DRAM bytes per refinement unit of workload cfg from the committed ncu
    figures (profiles/k_refine_traffic.json), or None when the code of
    refine.cu has changed since those counters were taken."""
    src = os.path.join(ROOT, "exact_dimensional_distance_gb300", "csrc", "refine.cu")
    path = os.path.join(ROOT, "profiles", "k_refine_traffic.json")
    try:
        sha = code_sha(src)
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("refine_cu_code_sha256_16") != sha:
        return None
    ent = rec.get("workloads", {}).get(str(cfg))
    return None if ent is None else float(ent["dram_bytes_per_unit"])


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


def fp32_peak_tflops(sm_count, sm_mhz):
    """FP32 peak: SMs x 128 FP32 lanes x clock x 2 flop (one fused
    multiply-add per lane per cycle)."""
    return sm_count * FP32_LANES_PER_SM * sm_mhz * 1e6 * 2.0 / 1e12


def index_geometry(j, st):
    """Cell sizes, stencil bounds and query tiles of the current index."""
    ix = j.index()
    cs = ix["cell_start"].cpu().numpy().astype(np.int64)
    size = np.diff(cs)
    bound = ix["cell_bound"].cpu().numpy().astype(np.int64)
    d4 = int(st["d_pad"])
    tq = 128 if d4 <= 64 else 64
    tiles = (size + tq - 1) // tq
    return size, bound, tiles, d4


def refine_algorithmic_bytes(j, st, n):
    """Algorithmic bytes of the refinement: the query rows (4 N d4), each
    cell's stencil candidate rows once per query tile of the cell (4 d4 bytes
    each), and one mask bit per candidate pair written."""
    size, bound, tiles, d4 = index_geometry(j, st)
    return float(4 * n * d4 + 4 * d4 * int((tiles * bound).sum()) + st["candidates"] / 8)


def join_algorithmic_bytes(j, st, n, d):
    """Algorithmic bytes of one whole join (build, index, count, refinement,
    compaction), from the index's cell sizes and stencils:
      index   4 N d (statistics) + 24 N per sort digit pass (key and value
              read and written) + 8 N d4 (variance-ordered copy and gather)
              + 16 C + 4 P (cell ranges and stencil lists);
      points  4 N d4 (query rows) + sum over cells i of the candidate rows
              of i's stencil, 4 d4 bytes each, once per query tile of i;
      results K_c / 8 written and read (one mask bit per candidate pair)
              + 4 |R| + 8 N (CSR columns and row offsets)."""
    size, bound, tiles, d4 = index_geometry(j, st)
    passes = (int(st["key_bits"]) + 7) // 8
    C, P, K, R = st["cells"], st["cell_pairs"], st["candidates"], st["pairs"]
    index = 4 * n * d + 24 * n * passes + 8 * n * d4 + 16 * C + 4 * P
    points = 4 * n * d4 + 4 * d4 * int((tiles * bound).sum())
    results = K / 8 + K / 8 + 4 * R + 8 * n
    return {"index": float(index), "points": float(points), "results": float(results)}


class Clocks:
    """nvidia-smi samples during the timed region."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.path or not os.path.exists(self.path):
            return out
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [v.strip() for v in line.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for name, v in zip(names, p[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if sm:
            out.update(sm_mhz=statistics.median(sm), sm_max_mhz=max(mx), reasons=sorted(reasons),
                       samples=len(sm))
        return out


def aggregate(t_local, units_local, dist=None, device=None):
    """Whole-job timing across ranks: the slowest rank's time and the units
    (result pairs) all ranks processed.  Works on any torch.distributed
    backend (nccl on the GPUs, gloo in the CPU tests)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(t_local), int(units_local)
    import torch
    t = torch.tensor([float(t_local)], dtype=torch.float64, device=device)
    u = torch.tensor([int(units_local)], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), int(u.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _oracle_threads():
    cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    os.environ.setdefault("OMP_PROC_BIND", "close")
    return cores


def sample_rows(n, d, coord_ops):
    """Query rows of a bounded oracle sample: about coord_ops = rows x n x d."""
    return int(max(64, min(n, coord_ops // (n * d))))


def run_reference(args, world, rank):
    """fp64 CPU oracle on a bounded sample of query rows per step."""
    if rank != 0:
        return
    import oracle
    cfg = args.config
    name, n, d, k = datagen.CONFIGS[cfg]
    x = datagen.generate(cfg)
    eps = load_eps(cfg)
    rows_per_step = args.ref_step_rows or sample_rows(n, d, REF_STEP_COORD_OPS)
    cores = _oracle_threads()
    rng = np.random.default_rng(12345)
    times, pairs = [], []
    for step in range(args.warmup + args.steps):
        q = rng.choice(n, size=rows_per_step, replace=False)
        t0 = time.perf_counter()
        row_ptr, _, _, _ = oracle.rows(x, eps, q, band=0.0)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            pairs.append(int(row_ptr[-1]))
    t = sum(times)
    value = sum(pairs) / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args, cfg, eps),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "omp_proc_bind": os.environ.get("OMP_PROC_BIND"),
                             "sample": "%d random query rows x all %d points per step (fp64 brute force)"
                                       % (rows_per_step, n)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "candidate_evals_per_s": rows_per_step * n * args.steps / t}
    print(json.dumps(line), flush=True)


def workload_config(args, cfg, eps):
    name, n, d, k = datagen.CONFIGS[cfg]
    if getattr(args, "n", None):
        name, n = name + " (reduced instance for profiling)", args.n
    return {"workload": "%s N=%d d=%d mean_neighbours=%d" % (name, n, d, k), "config": cfg, "n": n, "d": d,
            "eps": eps, "eps_hex": float(eps).hex(), "batch_bytes": args.batch_bytes,
            "l2": "flushed between steps",
            "parallelism": "one join sharded over the GPUs" if getattr(args, "shard", False) else "replica per GPU",
            "refine": "tensor cores (TF32 Gram prefilter + exact recheck)" if getattr(args, "refine", "cuda") == "tensor"
            else "CUDA cores"}


def cpu_baseline(x, eps, rows_req):
    """The oracle as it stands on a bounded sample (rank 0, N = 1 only), with
    the full join's time extrapolated (brute-force cost is the same for every
    query row)."""
    import oracle
    n, d = x.shape
    cores = _oracle_threads()
    rows = rows_req or sample_rows(n, d, CPU_SAMPLE_COORD_OPS)
    full = rows >= n
    q = np.arange(n) if full else np.random.default_rng(777).choice(n, size=rows, replace=False)
    t0 = time.perf_counter()
    row_ptr, _, _, _ = oracle.rows(x, eps, q, band=0.0)
    dt = time.perf_counter() - t0
    return {"value": int(row_ptr[-1]) / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "omp_proc_bind": os.environ.get("OMP_PROC_BIND"),
            "sample": ("the full join (%d query rows)" if full else "%d random query rows") % q.size
                      + " x all %d points, fp64 brute force, %.1f s" % (n, dt),
            "candidate_evals_per_s": q.size * n / dt,
            "full_join_s": dt * n / q.size, "full_join_s_kind": "measured" if full else "extrapolated"}


def run_config(args, cfg, world, rank, local, dist):
    import torch
    import exact_dimensional_distance_gb300 as edd

    x = datagen.generate(cfg, n=args.n)
    eps = load_eps(cfg)
    n, d = x.shape
    stream = torch.cuda.Stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        xd = torch.from_numpy(x).cuda()
        j = edd.Join(stream)
        j.set_refine(args.refine == "tensor")
    torch.cuda.synchronize()

    def step():
        j.build(xd)
        j.count(eps, out=False)
        st_count = j.stats()
        if args.shard:
            st_join = j.join_shard(eps, rank, world, args.batch_bytes)
        else:
            st_join = j.join(eps, args.batch_bytes)
        st_join["ms_index"] = st_count["ms_index"]
        st_join["ms_build"] = st_count["ms_build"]
        return st_join

    for _ in range(args.warmup):
        st = step()
    total_units = None
    if args.shard:
        total_units = j.join(eps, args.batch_bytes)["refine_units"]  # the whole join, untimed
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    stats = []
    launches0 = j.launches()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            ev[i][0].record(stream)
            stats.append(step())
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    launches = j.launches() - launches0
    ms = [a.elapsed_time(b) for a, b in ev]
    t_local = sum(ms) / 1e3
    pairs = stats[-1]["pairs"]
    cand = stats[-1]["candidates"]
    t, units = aggregate(t_local, pairs * args.steps, dist, torch.device("cuda", local))
    value = units / t
    clocks = clk.summary()

    # roofline of the refinement kernel (its launches are timed by the
    # library's CUDA events on the context's stream)
    st = stats[-1]
    refine_ms = statistics.median(s["ms_refine"] for s in stats)
    refine_launches = st["batches"]
    dims_alg, dims_exec = j.work_profile(eps)
    if args.shard and world > 1:
        # the profile covers the whole join; this rank refined its share of the units
        share = st["refine_units"] / float(total_units or 1)
        dims_alg, dims_exec = dims_alg * share, dims_exec * share
    flops = 3.0 * dims_alg
    pk, pk_kind = peaks()
    sm_count = torch.cuda.get_device_properties(local).multi_processor_count
    sm_mhz = float(pk.get("sm_max_mhz", 2070.0))
    peak = fp32_peak_tflops(sm_count, sm_mhz)
    hbm = float(pk.get("hbm_gbs", 6800.0))
    t_ref = refine_ms / 1e3
    achieved = flops / t_ref / 1e12
    rbytes = refine_algorithmic_bytes(j, st, n)
    t_flop = flops / (peak * 1e12) * 1e3
    t_bytes = rbytes / (hbm * 1e9) * 1e3
    tpu = refine_traffic_per_unit(cfg) if args.n is None and args.refine == "cuda" else None
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None if tpu is None else tpu * st["refine_units"] / refine_launches,
                "traffic_unit": "bytes per launch (ncu DRAM read+write per unit x units per launch)",
                "kernel": "k_refine",
                "work": "3 flop x sum over candidate pairs of the dimensions needed with per-pair exit every 4",
                "work_per_step_flop": flops, "launches_per_step": refine_launches,
                "ms_per_launch": refine_ms / refine_launches, "refine_units": st["refine_units"],
                "peak_kind": "%d SMs (device properties) x %d FP32 lanes x %s sm_max_mhz %.0f x 2 flop (FMA)"
                             % (sm_count, FP32_LANES_PER_SM, pk_kind, sm_mhz),
                # a pair-dimension is a subtract and a fused multiply-add: 3 flop
                # in 2 lane-instructions, so the instruction mix caps it at 0.75
                "issue_frac": achieved / (0.75 * peak),
                "executed_issue_frac": 3.0 * dims_exec / t_ref / 1e12 / (0.75 * peak),
                "mean_dims_alg": dims_alg / cand, "mean_dims_executed": dims_exec / cand,
                "full_dims_frac": 3.0 * cand * d / t_ref / 1e12 / peak,
                "bytes": rbytes, "hbm_gbs": hbm, "t_flop_ms": t_flop, "t_bytes_ms": t_bytes,
                "t_kernel_ms": refine_ms, "t_roof_ms": max(t_flop, t_bytes),
                "roof_bound": "fp32" if t_flop >= t_bytes else "hbm",
                "time_frac": max(t_flop, t_bytes) / refine_ms}

    # whole-join roofline: the slower of the refinement's algorithmic flops at
    # the FP32 peak and the join's algorithmic bytes at the HBM peak, against
    # the measured step time
    jb = join_algorithmic_bytes(j, st, n, d)
    jbytes = sum(jb.values())
    tj_flop = flops / (peak * 1e12) * 1e3
    tj_bytes = jbytes / (hbm * 1e9) * 1e3
    t_join = 1e3 * t_local / args.steps
    join_roofline = {"bound": "fp32" if tj_flop >= tj_bytes else "hbm", "flop": flops, "bytes": jbytes,
                     "bytes_split": jb, "t_flop_ms": tj_flop, "t_bytes_ms": tj_bytes,
                     "t_roof_ms": max(tj_flop, tj_bytes), "t_join_ms": t_join,
                     "frac": max(tj_flop, tj_bytes) / t_join, "fp32_peak_tflops": peak, "hbm_gbs": hbm,
                     "peak_kind": pk_kind}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
            "scaling": "strong" if args.shard else "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(args, cfg, eps), "gpu_launches": int(launches),
            "candidate_evals_per_s": world * cand * args.steps / t,
            "replicas": world,
            "pairs_per_step": pairs, "candidates_per_step": cand,
            "pruning": 1.0 - cand / float(n) ** 2,
            # candidate pairs left after the refinement's group-box stage
            # skip (the rest are proved farther than eps before streaming)
            "candidates_refined_per_step": st.get("candidates_refined"),
            "pruning_refined": (1.0 - st["candidates_refined"] / float(n) ** 2
                                if st.get("candidates_refined", -1) >= 0 else None),
            "phase_ms": {k: st[k] for k in ("ms_build", "ms_index", "ms_count", "ms_refine", "ms_compact",
                                            "ms_deliver")},
            "batches": st["batches"], "deliveries": st["deliveries"], "cells": st["cells"], "clocks": clocks,
            "roofline": roofline, "join_roofline": join_roofline}

    if not args.no_e2e:
        # end to end through the host-buffer entry points
        bb = args.e2e_batch_bytes or args.batch_bytes
        hx_t = torch.from_numpy(x).pin_memory()
        hx = hx_t.numpy()
        d2h = [0]

        def on_batch(b):
            d2h[0] += 8 * b.nq + 8 * (b.nq + 1) + 4 * b.nq + 4 * b.nnz

        def e2e_step():
            j.build(hx)
            j.count(eps, out=False)
            if args.shard:
                j.join_shard(eps, rank, world, bb, edd.HISS_OUT_CSR, True, on_batch)
            else:
                j.join(eps, bb, edd.HISS_OUT_CSR, True, on_batch)

        e2e_step()
        torch.cuda.synchronize()
        d2h[0] = 0
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize()
        te, e2e_units = aggregate(time.perf_counter() - t0, pairs * args.steps, dist, torch.device("cuda", local))
        line["e2e"] = {"value": e2e_units / te, "unit": UNIT,
                       "h2d_bytes_per_step": int(x.nbytes), "d2h_bytes_per_step": int(d2h[0] // args.steps),
                       "ms_per_step": 1e3 * te / args.steps, "batch_bytes": bb,
                       "batches": j.stats()["batches"], "deliveries": j.stats()["deliveries"]}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, eps, args.ref_rows)
    j.close()
    del xd, flush
    torch.cuda.empty_cache()
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--all-configs", action="store_true", help="one line per workload, 1 to 5")
    ap.add_argument("--impl", default="hiss", choices=["hiss", "reference"])
    ap.add_argument("--shard", action="store_true",
                    help="under torchrun: each rank runs its shard of one join (strong scaling) instead of a replica")
    ap.add_argument("--refine", default="cuda", choices=["cuda", "tensor"],
                    help="refinement: CUDA cores (default) or the tensor-core prefilter with exact recheck")
    ap.add_argument("--batch-bytes", type=int, default=DEFAULT_BATCH_BYTES)
    ap.add_argument("--ref-rows", type=int, default=None,
                    help="query rows of the cpu_baseline sample (default: about 2.5e11 / (n d), ~18 s on 16 cores)")
    ap.add_argument("--ref-step-rows", type=int, default=None,
                    help="query rows per step of --impl reference (default: about 6e10 / (n d), ~4 s per step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-batch-bytes", type=int, default=None,
                    help="batch bytes of the end-to-end leg (default: --batch-bytes); with several batches one "
                         "batch's copies to host overlap the next batch's refinement")
    ap.add_argument("--n", type=int, default=None,
                    help="draw a smaller instance of the workload (profiling only; not the benchmark workload)")
    args = ap.parse_args()
    world, rank, local = dist_env()

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    for cfg in (sorted(datagen.CONFIGS) if args.all_configs else [args.config]):
        line = run_config(args, cfg, world, rank, local, dist)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
