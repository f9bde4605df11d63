"""Benchmark of the dual-epsilon sandwich tail (and decode latency) on GB300.

Default workload (one "step" = one call of the fused tail over one batch):
  sandwich tail, rows=4096, n=6656, f32, eps_post=1e-8, eps_pre=1e-5; each
  block_out row has mean square log-uniform over 1e-4..1e2 (seeded synthetic).
Reported: achieved HBM GB/s of that call (algorithmic bytes: block_out and
residual read once, out_stream and normed written once, both gammas once =
(4*rows*n + 2*n)*4 bytes), rows/s, the fraction of the measured copy bandwidth,
and the decode latency of the same kernel at rows=1 (us/call, plain stream
launches and inside a CUDA graph).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mrn|reference]
For N > 1 launch under torchrun; every rank runs its own batch (rows are
independent, no data exchange) and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and rows/s at n=6656; decode µs/call"
UNIT = "GB/s"
KERNEL_SOURCES = ["dual_epsilon_sandwich_gb300/csrc/mrn_kernels.cuh",
                  "dual_epsilon_sandwich_gb300/csrc/mrn_ops_sandwich.cu",
                  "dual_epsilon_sandwich_gb300/csrc/mrn_api.cpp"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ncu_sandwich_f32_rows4096_n6656.md")
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=("mrn", "reference"), default="mrn")
    p.add_argument("--rows", type=int, default=4096)
    p.add_argument("--n", type=int, default=6656)
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--decode-calls", type=int, default=2000)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--reference-seconds", type=float, default=120.0,
                   help="--impl reference: wall time budget of the whole run")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the bf16 16384x4096 and f32 4x6656 secondary measurements")
    p.add_argument("--shard", action="store_true",
                   help="N > 1: split one global batch of --rows rows into contiguous row "
                        "blocks, one per rank (strong scaling; gammas replicated, no "
                        "collective on the data path); default: every rank runs its own "
                        "--rows batch (weak scaling)")
    p.add_argument("--profile-launches", type=int, default=0,
                   help="only run --warmup + this many launches of the timed call (for ncu)")
    p.add_argument("--profile-op", choices=("sandwich", "seam_f16", "q8_1", "wide_f32",
                                            "decode", "qk_norm", "add_rmsnorm", "widest_f32",
                                            "sandwich_n6655", "plain_f32"),
                   default="sandwich",
                   help="with --profile-launches: the call to launch -- the timed sandwich, the "
                        "fused f16 seam at the same shape, RMSNorm + Q8_1 at 16384 x 4096 bf16, "
                        "plain f32 RMSNorm at 1024 x 65536, the decode sandwich (1 x 6656 f32), "
                        "QK-norm (163840 x 128 bf16), residual add + norm (4096 x 6656 f32), or "
                        "plain f32 RMSNorm at 256 x 262144 (the looped kernel), the sandwich "
                        "at 4096 x 6655 f32 (rows not 16-byte aligned: the edge-staged kernel), "
                        "or plain f32 RMSNorm at 4096 x 6656 (eight slots, three CTAs per SM)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# helpers shared by both arms
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_rows(total_rows: int, world: int, rank: int):
    """Contiguous row block of `rank` when `total_rows` are split over `world`."""
    base, extra = divmod(total_rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_plan(total_rows: int, n: int, elem_bytes: int, world: int, rank: int) -> dict:
    """What one rank runs in the row-sharded mode: rows [row0, row0 + rows) of
    one global row-major [total_rows x n] batch, held in its own device copy.
    byte_offset is where that block starts in the global tensor (row0 * n *
    elem_bytes); the rank calls the library on its copy with `rows` rows, the
    gammas replicated, and nothing crosses between ranks on the data path."""
    lo, hi = shard_rows(total_rows, world, rank)
    return {"row0": lo, "rows": hi - lo, "byte_offset": lo * n * elem_bytes,
            "bytes": (hi - lo) * n * elem_bytes}


def local_block(arrays: dict, plan: dict, row_keys=("block_out", "residual")) -> dict:
    """This rank's inputs in the row-sharded mode: its row block of every row
    operand (views of the global host arrays) and every other array (the
    gammas) whole."""
    lo, hi = plan["row0"], plan["row0"] + plan["rows"]
    return {k: (v[lo:hi] if k in row_keys else v) for k, v in arrays.items()}


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (one scalar all-reduce; identity
    without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sandwich_bytes(rows: int, n: int, elem: int = 4) -> int:
    """Algorithmic bytes of one sandwich call: 2 row reads + 2 row writes + 2 gammas."""
    return (4 * rows * n + 2 * n) * elem


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    """Hash of the code (comments and whitespace removed) of the files that
    define the timed kernel and its launch."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel sources as they are now; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"kernel_source_digest:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_source_digest():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, rows split over host threads
# ---------------------------------------------------------------------------
class OracleRunner:
    """The oracle's sandwich tail over row blocks, one block per host thread
    (ctypes releases the GIL, so the blocks run in parallel)."""

    def __init__(self, arrays64, n, threads=None):
        import numpy as np

        import oracle
        self.np = np
        self.orc = oracle.default()
        self.arrays64 = arrays64
        self.b, self.r, self.gp, self.gq = arrays64
        self.n = n
        self.threads = threads or os.cpu_count() or 1
        self.pool = ThreadPoolExecutor(max_workers=self.threads)
        self.eps_post = float(np.float32(1e-8))
        self.eps_pre = float(np.float32(1e-5))

    def one_pass(self, rows: int) -> float:
        """Process the first `rows` rows once; returns the wall time in seconds."""
        bounds = self.np.linspace(0, rows, self.threads + 1).astype(int)

        def work(i):
            lo, hi = int(bounds[i]), int(bounds[i + 1])
            if hi > lo:
                self.orc.norm_residual_norm(self.b[lo:hi], self.r[lo:hi], self.gp, self.gq,
                                            self.eps_post, self.eps_pre)

        t0 = time.perf_counter()
        list(self.pool.map(work, range(self.threads)))
        return time.perf_counter() - t0

    def rate(self, rows: int, target_seconds: float):
        """Repeat passes over `rows` rows for about target_seconds; GB/s, rows/s, passes, s."""
        passes, elapsed = 0, 0.0
        while passes == 0 or (elapsed < target_seconds and passes < 1000):
            elapsed += self.one_pass(rows)
            passes += 1
        return (sandwich_bytes(rows, self.n) * passes / elapsed / 1e9, rows * passes / elapsed,
                passes, elapsed)


def oracle_configs(threads: int, seconds_each: float = 1.0):
    """The oracle, as it stands, on the other workloads' inputs (bounded
    samples, each timed for about `seconds_each`): single-threaded, and with
    rows split over `threads` host threads where a workload has enough rows.
    Units follow the GPU lines they sit beside (us per call for the decode
    workloads, GB/s of algorithmic bytes for the batched ones)."""
    import numpy as np

    import oracle
    from dual_epsilon_sandwich_gb300 import workloads as wl
    orc = oracle.default()
    pool = ThreadPoolExecutor(max_workers=threads)

    def timed(fn):
        fn()                                      # untimed first call (first touch)
        calls, elapsed = 0, 0.0
        while calls == 0 or elapsed < seconds_each:
            t0 = time.perf_counter()
            fn()
            elapsed += time.perf_counter() - t0
            calls += 1
        return elapsed / calls

    def split(fn, rows):
        bounds = np.linspace(0, rows, threads + 1).astype(int)
        return lambda: list(pool.map(lambda i: fn(int(bounds[i]), int(bounds[i + 1])),
                                     range(threads)))

    out = {}
    w = wl.plain_decode_rows()
    x, g = w.arrays["x"].astype(np.float64), w.arrays["gamma"].astype(np.float64)
    e = float(np.float32(w.eps))
    out[w.name] = {"us_per_call_1_thread": 1e6 * timed(lambda: orc.rmsnorm(x, g, e))}
    w = wl.sandwich_decode()
    b, r, gp, gq = (w.arrays[k].astype(np.float64) for k in
                    ("block_out", "residual", "gamma_post", "gamma_pre"))
    e1, e2 = float(np.float32(1e-8)), float(np.float32(1e-5))
    out[w.name] = {"us_per_call_1_thread": 1e6 * timed(
        lambda: orc.norm_residual_norm(b, r, gp, gq, e1, e2))}
    rows = 1024                                   # a sample drawn as the 16384 rows are
    w = wl.llama_bf16(rows=rows)
    x = orc.double_from_bf16(w.arrays["x"])
    res = orc.double_from_bf16(w.arrays["residual"])
    g = orc.double_from_bf16(w.arrays["gamma"])
    e = float(np.float32(w.eps))
    n = w.n
    for name, nbytes, one in (
            ("rmsnorm_bf16_rows16384_n4096", (2 * rows * n + n) * 2,
             lambda lo, hi: orc.rmsnorm(x[lo:hi], g, e)),
            ("then_add_bf16_rows16384_n4096", (3 * rows * n + n) * 2,
             lambda lo, hi: orc.rmsnorm_then_add(x[lo:hi], g, res[lo:hi], e))):
        t1 = timed(lambda: one(0, rows))
        tn = timed(split(one, rows))
        out[name] = {"GB_per_s_1_thread": nbytes / t1 / 1e9,
                     f"GB_per_s_{threads}_threads": nbytes / tn / 1e9,
                     "sample": f"{rows} rows drawn as the workload's 16384 are"}
    pool.shutdown()
    return out


def run_reference(args):
    """The oracle, timed on the host cores, on the same workload's rows: each
    step processes a bounded sample of rows, sized so that the whole
    --warmup + --steps run takes about two minutes."""
    import numpy as np

    from dual_epsilon_sandwich_gb300 import workloads as wl
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = wl.sandwich_prefill(rows=args.rows, n=args.n)
    a = w.arrays
    runner = OracleRunner([a[k].astype(np.float64) for k in ("block_out", "residual",
                                                             "gamma_post", "gamma_pre")], args.n)
    calib_rows = min(args.rows, 256)
    runner.one_pass(calib_rows)
    rows_per_s = calib_rows / runner.one_pass(calib_rows)
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    sample_rows = int(min(args.rows, max(8, rows_per_s * per_step)))
    for _ in range(args.warmup):
        runner.one_pass(sample_rows)
    times = [runner.one_pass(sample_rows) for _ in range(args.steps)]
    total = sum(times)
    value = sandwich_bytes(sample_rows, args.n) * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "rows": args.rows, "n": args.n, "eps_post": 1e-8,
                   "eps_pre": 1e-5, "sample_rows_per_step": sample_rows},
        "rows_per_s": sample_rows * args.steps / total,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": runner.threads, "kind": "oracle",
                         "sample": f"first {sample_rows} of the {args.rows} rows per step, "
                                   f"split over {runner.threads} host threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------
def run_mrn(args):
    import numpy as np
    import torch

    from dual_epsilon_sandwich_gb300 import _build, mrn
    from dual_epsilon_sandwich_gb300 import workloads as wl

    rank, world, local = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        _build.build()
    if pg is not None:
        pg.barrier()
    mrn.lib()

    if args.profile_launches and args.profile_op != "sandwich":
        return profile_other(args, dev)

    global_rows, n = args.rows, args.n
    w = wl.sandwich_prefill(rows=global_rows, n=n)
    a = w.arrays
    plan = None
    if args.shard:
        # row-sharded: this rank's contiguous block of the one global batch
        plan = shard_plan(global_rows, n, 4, world, rank)
        a = local_block(a, plan)
    rows = plan["rows"] if plan else global_rows
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    # two resident buffer sets, used alternately: 2 x 436 MB > L2 between reuse
    sets = []
    for _ in range(2):
        b = torch.from_numpy(a["block_out"]).to(dev)
        r = torch.from_numpy(a["residual"]).to(dev)
        gp = torch.from_numpy(a["gamma_post"]).to(dev)
        gq = torch.from_numpy(a["gamma_pre"]).to(dev)
        sets.append((b, r, gp, gq, torch.empty_like(b), torch.empty_like(b)))

    def call(sset, nrows=rows):
        b, r, gp, gq, s, o = sset
        st = mrn.mrn_norm_residual_norm(b.data_ptr(), r.data_ptr(), gp.data_ptr(),
                                        gq.data_ptr(), s.data_ptr(), o.data_ptr(), nrows, n,
                                        1e-8, 1e-5, mrn.MRN_F32, sh)
        if st != 0:
            raise mrn.MrnError(st, "mrn_norm_residual_norm")

    geometry = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, rows, n, mrn.MRN_F32, True)

    for i in range(args.warmup):
        call(sets[i % 2])
    torch.cuda.synchronize()
    if args.profile_launches:
        for i in range(args.profile_launches):
            call(sets[i % 2])
        torch.cuda.synchronize()
        print(json.dumps({"profile_launches": args.profile_launches, "geometry": geometry}))
        return 0

    # -- device-resident timed region -------------------------------------
    # One launch per step, back to back on one stream, bracketed by a barrier
    # and a synchronize on both sides; the average launch duration is the
    # region's time over K (the region holds nothing but these launches).
    K = args.steps
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if world == 1 else local)
    sampler.start()
    time.sleep(0.3)
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    launches0 = mrn.mrn_launch_count()
    t_begin.record(stream)
    for i in range(K):
        call(sets[i % 2])
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg is not None:
        pg.barrier()
    clocks = sampler.stop()
    launches = mrn.mrn_launch_count() - launches0
    local_ms = t_begin.elapsed_time(t_end)
    total_ms = max_over_ranks(local_ms, pg, dev)
    avg_kernel_ms = local_ms / max(1, launches)
    step_bytes = sandwich_bytes(rows, n)
    # whole-job bytes per step: every rank's batch (weak) or the one global batch (sharded)
    job_bytes = (4 * global_rows * n + 2 * n * world) * 4 if plan else world * step_bytes
    job_rows = global_rows if plan else world * rows
    value = job_bytes * K / (total_ms * 1e-3) / 1e9
    achieved = step_bytes / (avg_kernel_ms * 1e-3) / 1e9

    # -- end to end through the C ABI with host buffers --------------------
    # Each step copies its inputs host -> device, runs the call and copies both
    # outputs device -> host, all from pinned memory.  Steps alternate between
    # two streams and two device buffer sets, as a user streaming batches
    # would: one step's device -> host copy overlaps the next step's host ->
    # device copy (separate copy engines) and kernel.
    pin = {k: torch.from_numpy(a[k]).pin_memory() for k in ("block_out", "residual",
                                                             "gamma_post", "gamma_pre")}
    host_out = [(torch.empty((rows, n), dtype=torch.float32).pin_memory(),
                 torch.empty((rows, n), dtype=torch.float32).pin_memory()) for _ in range(2)]
    e2e_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    h2d = sum(t.numel() * 4 for t in pin.values())
    d2h = 2 * rows * n * 4

    def e2e_step(i, call=True):
        st = e2e_streams[i % 2]
        b, r, gp, gq, s, o = sets[i % 2]
        host_s, host_o = host_out[i % 2]
        with torch.cuda.stream(st):
            b.copy_(pin["block_out"], non_blocking=True)
            r.copy_(pin["residual"], non_blocking=True)
            gp.copy_(pin["gamma_post"], non_blocking=True)
            gq.copy_(pin["gamma_pre"], non_blocking=True)
            if call:
                stc = mrn.mrn_norm_residual_norm(b.data_ptr(), r.data_ptr(), gp.data_ptr(),
                                                 gq.data_ptr(), s.data_ptr(), o.data_ptr(), rows,
                                                 n, 1e-8, 1e-5, mrn.MRN_F32, st.cuda_stream)
                if stc != 0:
                    raise mrn.MrnError(stc, "mrn_norm_residual_norm")
            host_s.copy_(s, non_blocking=True)
            host_o.copy_(o, non_blocking=True)

    def e2e_drain():
        for st in e2e_streams:
            st.synchronize()

    torch.cuda.synchronize()
    # Warm up the host-link path (the first copies from fresh pinned buffers run
    # up to ~1.6x slower for a few tens of ms): at least 10 steps and 100 ms.
    t_warm = time.perf_counter()
    for i in range(10000):
        e2e_step(i)
        e2e_drain()
        if i >= 9 and time.perf_counter() - t_warm > 0.1:
            break
    if pg is not None:
        pg.barrier()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i)
    e2e_drain()
    e2e_s = (time.perf_counter() - t0) / args.e2e_steps
    e2e_s = max_over_ranks(e2e_s, pg, dev)
    e2e_value = job_bytes / e2e_s / 1e9
    # The same steps without the call: the host link's own ceiling for this
    # traffic on this machine, in the same unit.
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i, call=False)
    e2e_drain()
    link_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, pg, dev)
    link_value = job_bytes / link_s / 1e9

    # -- decode latency: rows=1, n=6656 ---------------------------------------
    decode = decode_latency(args, dev, stream)
    secondary = {} if args.no_secondary else secondary_workloads(dev, stream)

    peak, peak_kind = measured_peaks()
    traffic = profiled_traffic()
    parallelism = (f"one global batch of {global_rows} rows in contiguous row blocks over "
                   f"{world} ranks ({rows} here, from row {plan['row0']}); gammas replicated, "
                   f"no exchange" if plan else f"rows x{world}, no exchange")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "strong" if plan else "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "rows": rows, "n": n, "eps_post": 1e-8, "eps_pre": 1e-5,
                   "global_batch": job_rows, "parallelism": parallelism,
                   "l2": "inputs larger than L2: two resident buffer sets of 436 MB used "
                         "alternately", "geometry": geometry,
                   "launch": "programmatic dependent launch (the library's default; "
                             "mrn_set_launch_options(0) turns it off)"
                   if mrn.mrn_launch_options() & mrn.MRN_LAUNCH_PDL else "stream-ordered"},
        "rows_per_s": job_rows * K / (total_ms * 1e-3),
        "pct_of_peak": 100.0 * value / (world * peak),
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": step_bytes,
                     "avg_launch_ms": avg_kernel_ms},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies_only": link_value,
                "note": "pinned host buffers; every step copies its inputs H2D, runs the call "
                        "and copies both outputs D2H; steps alternate over two streams and "
                        "two device buffer sets; copies_only = the same steps without the "
                        "call (the host link's ceiling)"},
        "decode": decode,
        "secondary": secondary,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        runner = OracleRunner([a[k].astype(np.float64) for k in ("block_out", "residual",
                                                                 "gamma_post", "gamma_pre")], n)
        gbs, rps, passes, elapsed = runner.rate(rows, args.cpu_seconds)
        single = OracleRunner(runner.arrays64, n, threads=1)
        sample = min(rows, 256)
        gbs1, _, passes1, elapsed1 = single.rate(sample, max(0.5, args.cpu_seconds / 5))
        line["cpu_baseline"] = {"value": gbs, "unit": UNIT, "cores": runner.threads,
                                "kind": "oracle",
                                "sample": f"all {rows} rows x {passes} passes ({elapsed:.1f} s), "
                                          f"rows split over {runner.threads} host threads",
                                "rows_per_s": rps,
                                "single_thread": {"value": gbs1, "unit": UNIT,
                                                  "sample": f"the first {sample} rows x "
                                                            f"{passes1} passes ({elapsed1:.1f} s)"},
                                "configs": oracle_configs(runner.threads,
                                                          max(0.2, args.cpu_seconds / 10))}
    # Last in the line, short: every workload's headline figure, so that a
    # reader who keeps only the end of the line still sees all of them.
    line["workloads"] = workload_summary(line, peak)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def workload_summary(line: dict, peak: float) -> dict:
    """One compact entry per workload (rounded; the detailed figures are in
    `decode`, `secondary` and the top-level keys of the same line)."""
    def r(v, nd=1):
        return None if v is None else round(float(v), nd)

    dec = line.get("decode") or {}
    sec = line.get("secondary") or {}
    out = {
        "1_rmsnorm_f32_rows4_n6656_us_per_call_graph":
            r(sec.get("rmsnorm_f32_rows4_n6656", {}).get("us_per_call_graph"), 3),
        "2_decode_sandwich_f32_rows1_n6656_us_per_call":
            {"graph": r(dec.get("us_per_call_graph"), 3),
             "graph_l2_hot": r(dec.get("us_per_call_graph_l2_hot"), 3),
             "stream": r(dec.get("us_per_call_stream"), 3)} if dec else None,
        "3_sandwich_f32_rows4096_n6656":
            {"GB_per_s": r(line["value"]), "pct_of_copy": r(100 * line["value"] /
                                                             (line["n_gpus"] * peak), 2),
             "us_per_call": r(1e3 * line["ms_per_step"], 2)},
    }
    for key, name in (("4_rmsnorm_bf16_rows16384_n4096_GB_per_s", "rmsnorm_bf16_rows16384_n4096"),
                      ("4_then_add_bf16_rows16384_n4096_GB_per_s",
                       "then_add_bf16_rows16384_n4096")):
        out[key] = r(sec.get(name, {}).get("GB_per_s"))
    sweep = sec.get("sweep_large_f32") or {}
    out["5_sweep_f32_GB_per_s_rmsnorm_then_add"] = {
        shape: [r(e.get("rmsnorm", {}).get("GB_per_s"), 0), r(e.get("then_add", {}).get("GB_per_s"), 0)]
        for shape, e in sweep.items()} or None
    small = sec.get("sweep_small_f32_us_per_call_graph") or {}
    out["5_sweep_small_f32_us_per_call_graph_rmsnorm_then_add"] = {
        shape: [r(e.get("rmsnorm"), 2), r(e.get("then_add"), 2)]
        for shape, e in small.items()} or None
    nxt = {}
    for name in ("add_rmsnorm_f32_rows4096_n6656", "then_add_scale_bf16_rows16384_n4096",
                 "rmsnorm_q8_1_bf16_rows16384_n4096", "qk_norm_bf16_rows163840_n128",
                 "seam_f16_from_f32_rows4096_n6656", "seam_bf16_from_bf16_rows16384_n4096",
                 "sandwich_f32_rows4096_n6655", "rmsnorm_f32_rows4096_n6655",
                 "rmsnorm_f32_rows256_n262144"):
        if name in sec:
            nxt[name] = r(sec[name].get("GB_per_s"))
    out["next_GB_per_s"] = nxt or None
    return out


def decode_latency(args, dev, stream):
    """us per call of the sandwich tail at rows=1, n=6656: back-to-back stream
    launches and a CUDA graph, each over 1024 rotating buffer sets (160 MB > L2)."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    from dual_epsilon_sandwich_gb300 import workloads as wl
    w = wl.sandwich_decode()
    a = w.arrays
    nsets = 1024
    n = w.n
    big = {k: torch.from_numpy(a[k]).to(dev).repeat(nsets, 1).contiguous()
           for k in ("block_out", "residual")}
    gp = torch.from_numpy(a["gamma_post"]).to(dev)
    gq = torch.from_numpy(a["gamma_pre"]).to(dev)
    s = torch.empty((nsets, n), device=dev)
    o = torch.empty((nsets, n), device=dev)
    sh = stream.cuda_stream
    ptrs = [(big["block_out"][i].data_ptr(), big["residual"][i].data_ptr(), s[i].data_ptr(),
             o[i].data_ptr()) for i in range(nsets)]

    def call(i, handle):
        b, r, ss, oo = ptrs[i % nsets]
        st = mrn.mrn_norm_residual_norm(b, r, gp.data_ptr(), gq.data_ptr(), ss, oo, 1, n,
                                        1e-8, 1e-5, mrn.MRN_F32, handle)
        if st != 0:
            raise mrn.MrnError(st, "decode")

    calls = args.decode_calls
    for i in range(64):
        call(i, sh)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(calls):
        call(i, sh)
    e1.record(stream)
    torch.cuda.synchronize()
    stream_us = e0.elapsed_time(e1) * 1e3 / calls

    # graph of `per_graph` calls on rotating sets, replayed
    per_graph = nsets
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(per_graph):
                call(i, side.cuda_stream)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, calls // per_graph)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    graph_us = e0.elapsed_time(e1) * 1e3 / (reps * per_graph)
    # the same call on one buffer set (L2-resident, as right after the producer)
    g_hot = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_hot, stream=side):
            for _ in range(per_graph):
                call(0, side.cuda_stream)
    stream.wait_stream(side)
    g_hot.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g_hot.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    hot_us = e0.elapsed_time(e1) * 1e3 / (reps * per_graph)
    # the rotating graph again without programmatic dependent launch (the
    # library launches with it by default)
    mrn.mrn_set_launch_options(0)
    g_pdl = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_pdl, stream=side):
            for i in range(per_graph):
                call(i, side.cuda_stream)
    mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL)
    stream.wait_stream(side)
    g_pdl.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g_pdl.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    pdl_us = e0.elapsed_time(e1) * 1e3 / (reps * per_graph)
    geometry = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, 1, n, mrn.MRN_F32, True)
    return {"workload": w.name, "us_per_call_stream": stream_us,
            "us_per_call_graph": graph_us, "us_per_call_graph_l2_hot": hot_us,
            "us_per_call_graph_no_pdl": pdl_us,
            "bytes_per_call": sandwich_bytes(1, n), "rotating_sets": nsets,
            "geometry": geometry}


def secondary_workloads(dev, stream):
    """The other measured workloads: Llama-style bf16 plain RMSNorm and
    then-add at 16384 x 4096 (GB/s, two rotating buffer sets of >= 268 MB),
    plain f32 RMSNorm at 4 x 6656 (us/call in a CUDA graph over 512 rotating
    buffer sets, 122 MB > L2), the sweep's shapes (GB/s from rows x n >= 2^26,
    us/call in a CUDA graph below), and the operations beyond the base three."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    from dual_epsilon_sandwich_gb300 import workloads as wl
    out = {}
    sh = stream.cuda_stream
    w = wl.llama_bf16()
    a = w.arrays

    def bf16(arr):
        return torch.from_numpy(arr.view("int16")).to(dev).view(torch.bfloat16)

    sets = [(bf16(a["x"]), bf16(a["gamma"]), bf16(a["residual"])) for _ in range(2)]
    outs = [torch.empty_like(sets[0][0]) for _ in range(2)]
    rows, n = w.rows, w.n
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, op, nbytes in (("rmsnorm_bf16_rows16384_n4096", 0, (2 * rows * n + n) * 2),
                             ("then_add_bf16_rows16384_n4096", 1, (3 * rows * n + n) * 2)):
        def call(i):
            x, g, r = sets[i % 2]
            y = outs[i % 2]
            if op == 0:
                st = mrn.mrn_rmsnorm(x.data_ptr(), g.data_ptr(), y.data_ptr(), rows, n, w.eps,
                                     mrn.MRN_BF16, sh)
            else:
                st = mrn.mrn_rmsnorm_then_add(x.data_ptr(), g.data_ptr(), r.data_ptr(),
                                              y.data_ptr(), rows, n, w.eps, mrn.MRN_BF16, sh)
            if st != 0:
                raise mrn.MrnError(st, name)
        for i in range(20):
            call(i)
        torch.cuda.synchronize()
        iters = 500
        e0.record(stream)
        for i in range(iters):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / iters
        out[name] = {"GB_per_s": nbytes / (us * 1e-6) / 1e9, "us_per_call": us,
                     "rows_per_s": rows / (us * 1e-6), "bytes_per_call": nbytes,
                     "geometry": mrn.mrn_query_geometry(op, rows, n, mrn.MRN_BF16, True)}
    del sets, outs
    torch.cuda.empty_cache()
    out.update(more_ops(dev, stream))
    out.update(seam_ops(dev, stream))
    out["sweep_large_f32"] = sweep_large(dev, stream)
    out["sweep_small_f32_us_per_call_graph"] = sweep_small(dev, stream)

    w = wl.plain_decode_rows()
    nsets = 512
    x = torch.from_numpy(w.arrays["x"]).to(dev).repeat(nsets, 1).view(nsets, w.rows, w.n)
    g = torch.from_numpy(w.arrays["gamma"]).to(dev)
    y = torch.empty_like(x)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for i in range(nsets):
            mrn.mrn_rmsnorm(x[i].data_ptr(), g.data_ptr(), y[i].data_ptr(), w.rows, w.n, w.eps,
                            mrn.MRN_F32, side.cuda_stream)
        with torch.cuda.graph(graph, stream=side):
            for i in range(nsets):
                st = mrn.mrn_rmsnorm(x[i].data_ptr(), g.data_ptr(), y[i].data_ptr(), w.rows, w.n,
                                     w.eps, mrn.MRN_F32, side.cuda_stream)
                if st != 0:
                    raise mrn.MrnError(st, w.name)
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    reps = 4
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * nsets)
    out[w.name] = {"us_per_call_graph": us, "bytes_per_call": (2 * w.rows * w.n + w.n) * 4,
                   "geometry": mrn.mrn_query_geometry(0, w.rows, w.n, mrn.MRN_F32, True)}
    return out


def more_ops(dev, stream):
    """The operations beyond plain RMSNorm, then-add and the sandwich, timed the same way
    (GB/s of algorithmic bytes, two rotating buffer sets larger than L2,
    seeded torch inputs): residual add + norm at the benchmark's width, the
    sandwich and plain RMSNorm at one element less (rows not 16-byte aligned),
    then-add-scale and RMSNorm + Q8_1 at 16384 x 4096 bf16, and the per-head
    QK-norm shape (163840 rows of 128, bf16)."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    sh = stream.cuda_stream
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261202)
    out = {}

    def run(name, op, dtype, rows, n, nbytes, launch):
        tdt = torch.float32 if dtype == mrn.MRN_F32 else torch.bfloat16
        sets = []
        for _ in range(2):
            x = torch.randn(rows, n, device=dev, generator=gen).to(tdt)
            r = torch.randn(rows, n, device=dev, generator=gen).to(tdt)
            g = (1 + 0.1 * torch.randn(n, device=dev, generator=gen)).to(tdt)
            y = torch.empty_like(x)
            y2 = torch.empty((rows * (n // 32) * 36 + 16,), dtype=torch.uint8, device=dev) \
                if op == mrn.MRN_OP_RMSNORM_Q8_1 else torch.empty_like(x)
            sc = torch.full((1,), 0.5, device=dev).to(tdt)
            sets.append((x, r, g, y, y2, sc))
        for i in range(20):
            launch(sets[i % 2])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        iters = 400
        e0.record(stream)
        for i in range(iters):
            launch(sets[i % 2])
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / iters
        out[name] = {"GB_per_s": nbytes / (us * 1e-6) / 1e9, "us_per_call": us,
                     "rows_per_s": rows / (us * 1e-6), "bytes_per_call": nbytes,
                     "geometry": mrn.mrn_query_geometry(op, rows, n, dtype, True)}
        del sets
        torch.cuda.empty_cache()

    def check(st, what):
        if st != 0:
            raise mrn.MrnError(st, what)

    F, B = mrn.MRN_F32, mrn.MRN_BF16
    rows, n = 4096, 6656
    run("add_rmsnorm_f32_rows4096_n6656", mrn.MRN_OP_ADD_RMSNORM, F, rows, n,
        (4 * rows * n + n) * 4,
        lambda t: check(mrn.mrn_add_rmsnorm(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(),
                                            t[3].data_ptr(), t[4].data_ptr(), rows, n, 1e-5, F,
                                            sh), "add_rmsnorm"))
    # the benchmark's width minus one: a row pitch of 26,620 bytes (not a multiple
    # of 16), every row staged as the 16-byte granules that cover it
    rows, n = 4096, 6655
    run("sandwich_f32_rows4096_n6655", mrn.MRN_OP_SANDWICH, F, rows, n, (4 * rows * n + 2 * n) * 4,
        lambda t: check(mrn.mrn_norm_residual_norm(t[0].data_ptr(), t[1].data_ptr(),
                                                   t[2].data_ptr(), t[2].data_ptr(),
                                                   t[3].data_ptr(), t[4].data_ptr(), rows, n,
                                                   1e-8, 1e-5, F, sh), "sandwich n=6655"))
    run("rmsnorm_f32_rows4096_n6655", mrn.MRN_OP_RMSNORM, F, rows, n, (2 * rows * n + n) * 4,
        lambda t: check(mrn.mrn_rmsnorm(t[0].data_ptr(), t[2].data_ptr(), t[3].data_ptr(), rows,
                                        n, 1e-5, F, sh), "rmsnorm n=6655"))
    rows, n = 16384, 4096
    run("then_add_scale_bf16_rows16384_n4096", mrn.MRN_OP_THEN_ADD_SCALE, B, rows, n,
        (3 * rows * n + n + 1) * 2,
        lambda t: check(mrn.mrn_rmsnorm_then_add_scale(t[0].data_ptr(), t[2].data_ptr(),
                                                       t[1].data_ptr(), t[5].data_ptr(),
                                                       t[3].data_ptr(), rows, n, 1e-6, B, sh),
                        "then_add_scale"))
    run("rmsnorm_q8_1_bf16_rows16384_n4096", mrn.MRN_OP_RMSNORM_Q8_1, B, rows, n,
        (rows * n + n) * 2 + rows * (n // 32) * 36,
        lambda t: check(mrn.mrn_rmsnorm_q8_1(t[0].data_ptr(), t[2].data_ptr(), t[4].data_ptr(),
                                             rows, n, 1e-6, B, sh), "q8_1"))
    rows, n = 163840, 128
    run("qk_norm_bf16_rows163840_n128", mrn.MRN_OP_RMSNORM, B, rows, n, (2 * rows * n + n) * 2,
        lambda t: check(mrn.mrn_rmsnorm(t[0].data_ptr(), t[2].data_ptr(), t[3].data_ptr(), rows,
                                        n, 1e-6, B, sh), "qk_norm"))
    return out


def profile_other(args, dev):
    """--profile-launches for a secondary call: --warmup + --profile-launches
    launches of it on seeded random inputs (two buffer sets), nothing else."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    sh = torch.cuda.current_stream().cuda_stream
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261204)
    if args.profile_op == "seam_f16":
        rows, n = args.rows, args.n
        sets = [(torch.randn(rows, n, device=dev, generator=gen),
                 (1 + 0.1 * torch.randn(n, device=dev, generator=gen)).half(),
                 torch.empty(rows, n, dtype=torch.float16, device=dev)) for _ in range(2)]

        def call(t):
            return mrn.mrn_rmsnorm_seam(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), rows,
                                        n, 1e-5, mrn.MRN_F32, mrn.MRN_F16, sh)
        geometry = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_SEAM, rows, n, mrn.MRN_F32, True)
    elif args.profile_op in ("decode", "add_rmsnorm", "sandwich_n6655"):
        # the decode sandwich tail (1 x 6656 f32, a cluster of 8 CTAs), the
        # residual add + norm at the prefill shape (the register batch kernel), or
        # the sandwich one element narrower (4096 x 6655, the edge-staged kernel)
        rows, n = {"decode": (1, 6656), "add_rmsnorm": (4096, 6656),
                   "sandwich_n6655": (4096, 6655)}[args.profile_op]
        sets = [tuple(torch.randn(rows, n, device=dev, generator=gen) for _ in range(2)) +
                tuple(1 + 0.1 * torch.randn(n, device=dev, generator=gen) for _ in range(2)) +
                tuple(torch.empty(rows, n, device=dev) for _ in range(2)) for _ in range(2)]
        if args.profile_op in ("decode", "sandwich_n6655"):
            def call(t):
                return mrn.mrn_norm_residual_norm(t[0].data_ptr(), t[1].data_ptr(),
                                                  t[2].data_ptr(), t[3].data_ptr(),
                                                  t[4].data_ptr(), t[5].data_ptr(), rows, n,
                                                  1e-8, 1e-5, mrn.MRN_F32, sh)
            geometry = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, rows, n, mrn.MRN_F32, True)
        else:
            def call(t):
                return mrn.mrn_add_rmsnorm(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(),
                                           t[4].data_ptr(), t[5].data_ptr(), rows, n, 1e-5,
                                           mrn.MRN_F32, sh)
            geometry = mrn.mrn_query_geometry(mrn.MRN_OP_ADD_RMSNORM, rows, n, mrn.MRN_F32,
                                              True)
    elif args.profile_op == "qk_norm":
        # per-head QK-norm: 163840 rows of 128 bf16 (the rows-per-warp kernel)
        rows, n = 163840, 128
        sets = [(torch.randn(rows, n, device=dev, generator=gen).bfloat16(),
                 (1 + 0.1 * torch.randn(n, device=dev, generator=gen)).bfloat16(),
                 torch.empty(rows, n, dtype=torch.bfloat16, device=dev)) for _ in range(2)]

        def call(t):
            return mrn.mrn_rmsnorm(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), rows, n,
                                   1e-6, mrn.MRN_BF16, sh)
        geometry = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, rows, n, mrn.MRN_BF16, True)
    elif args.profile_op == "widest_f32":
        # rows past the cluster kernels' reach (1 MB each): the looped kernel
        rows, n = 256, 262144
        sets = [(torch.randn(rows, n, device=dev, generator=gen),
                 1 + 0.1 * torch.randn(n, device=dev, generator=gen),
                 torch.empty(rows, n, device=dev)) for _ in range(2)]

        def call(t):
            return mrn.mrn_rmsnorm(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), rows, n,
                                   1e-5, mrn.MRN_F32, sh)
        geometry = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, rows, n, mrn.MRN_F32, True)
    elif args.profile_op in ("wide_f32", "plain_f32"):
        # plain f32 RMSNorm of 256 KB rows (the cluster-staged kernel, 8 CTAs a row),
        # or at the benchmark's shape (the register kernel at eight slots per thread)
        rows, n = (1024, 65536) if args.profile_op == "wide_f32" else (4096, 6656)
        sets = [(torch.randn(rows, n, device=dev, generator=gen),
                 1 + 0.1 * torch.randn(n, device=dev, generator=gen),
                 torch.empty(rows, n, device=dev)) for _ in range(2)]

        def call(t):
            return mrn.mrn_rmsnorm(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), rows, n,
                                   1e-5, mrn.MRN_F32, sh)
        geometry = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, rows, n, mrn.MRN_F32, True)
    else:
        rows, n = 16384, 4096
        sets = [(torch.randn(rows, n, device=dev, generator=gen).bfloat16(),
                 (1 + 0.1 * torch.randn(n, device=dev, generator=gen)).bfloat16(),
                 torch.empty(rows * (n // 32) * mrn.Q8_1_BLOCK_BYTES, dtype=torch.uint8,
                             device=dev)) for _ in range(2)]

        def call(t):
            return mrn.mrn_rmsnorm_q8_1(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), rows,
                                        n, 1e-6, mrn.MRN_BF16, sh)
        geometry = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_Q8_1, rows, n, mrn.MRN_BF16, True)
    for i in range(args.warmup + args.profile_launches):
        st = call(sets[i % 2])
        if st != 0:
            raise mrn.MrnError(st, args.profile_op)
    torch.cuda.synchronize()
    print(json.dumps({"profile_op": args.profile_op, "rows": rows, "n": n,
                      "profile_launches": args.profile_launches, "geometry": geometry}))
    return 0


def sweep_large(dev, stream):
    """The sweep workload's shapes with rows x n >= 2^26 (f32, plain and
    then-add, eps 1e-5): GB/s of algorithmic bytes, one buffer set (every
    operand exceeds L2), seeded device-side random inputs."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    sh = stream.cuda_stream
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261205)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {}
    for rows, n in ((65536, 2048), (65536, 5120), (65536, 6656), (65536, 8192),
                    (65536, 16384), (4096, 16384), (4096, 65536)):
        x = torch.randn(rows, n, device=dev, generator=gen)
        r = torch.randn(rows, n, device=dev, generator=gen)
        g = 1 + 0.1 * torch.randn(n, device=dev, generator=gen)
        y = torch.empty_like(x)
        entry = {}
        for op, nbytes in (("rmsnorm", (2 * rows * n + n) * 4),
                           ("then_add", (3 * rows * n + n) * 4)):
            def call():
                if op == "rmsnorm":
                    st = mrn.mrn_rmsnorm(x.data_ptr(), g.data_ptr(), y.data_ptr(), rows, n, 1e-5,
                                         mrn.MRN_F32, sh)
                else:
                    st = mrn.mrn_rmsnorm_then_add(x.data_ptr(), g.data_ptr(), r.data_ptr(),
                                                  y.data_ptr(), rows, n, 1e-5, mrn.MRN_F32, sh)
                if st != 0:
                    raise mrn.MrnError(st, f"sweep {rows}x{n} {op}")
            iters = max(20, min(200, int(2e10 // nbytes)))
            for _ in range(3):
                call()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(iters):
                call()
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / iters
            entry[op] = {"GB_per_s": nbytes / (us * 1e-6) / 1e9, "us_per_call": us}
        entry["geometry"] = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, rows, n, mrn.MRN_F32,
                                                   True)
        out[f"rows{rows}_n{n}"] = entry
        del x, r, y
        torch.cuda.empty_cache()
    return out


def sweep_small(dev, stream):
    """The sweep workload's shapes with rows x n < 2^26 (f32, plain and
    then-add, eps 1e-5): us per call in a CUDA graph over rotating buffer sets
    (at least 300 MB in all where at most 512 sets reach it; the smallest
    shapes stay L2-resident), seeded device-side random inputs."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    from dual_epsilon_sandwich_gb300 import workloads as wl
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261206)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    side = torch.cuda.Stream()
    out = {}
    for n, rows in wl.sweep_shapes():
        if rows * n >= 2 ** 26:
            continue
        per_set = 3 * rows * n * 4
        sets = max(2, min(512, -(-300 * 2 ** 20 // per_set)))
        calls = max(sets, 64)
        x = torch.randn(sets, rows, n, device=dev, generator=gen)
        r = torch.randn(sets, rows, n, device=dev, generator=gen)
        g = 1 + 0.1 * torch.randn(n, device=dev, generator=gen)
        y = torch.empty_like(x)
        entry = {}
        for op in ("rmsnorm", "then_add"):
            def call(i, handle):
                j = i % sets
                if op == "rmsnorm":
                    st = mrn.mrn_rmsnorm(x[j].data_ptr(), g.data_ptr(), y[j].data_ptr(), rows, n,
                                         1e-5, mrn.MRN_F32, handle)
                else:
                    st = mrn.mrn_rmsnorm_then_add(x[j].data_ptr(), g.data_ptr(), r[j].data_ptr(),
                                                  y[j].data_ptr(), rows, n, 1e-5, mrn.MRN_F32,
                                                  handle)
                if st != 0:
                    raise mrn.MrnError(st, f"sweep {rows}x{n} {op}")
            side.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                for i in range(4):
                    call(i, side.cuda_stream)
                with torch.cuda.graph(graph, stream=side):
                    for i in range(calls):
                        call(i, side.cuda_stream)
            stream.wait_stream(side)
            graph.replay()
            torch.cuda.synchronize()
            reps = 3
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            entry[op] = e0.elapsed_time(e1) * 1e3 / (reps * calls)
        entry["sets"] = sets
        out[f"{rows}x{n}"] = entry
        del x, r, y, graph
        torch.cuda.empty_cache()
    return out


def seam_ops(dev, stream):
    """The split-norm seam (the weightless norm published in f16 or bf16, the
    weight applied as a second operation in that format): the fused kernel
    against the split route (two kernels, the intermediate through HBM), at
    the benchmark's width with f32 input and at 16384 x 4096 bf16.  Same
    timing as the other secondary lines; GB/s of each form's own algorithmic
    bytes."""
    import torch

    from dual_epsilon_sandwich_gb300 import mrn
    sh = stream.cuda_stream
    gen = torch.Generator(device=dev)
    gen.manual_seed(20261203)
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(launch, sets, iters=300):
        for i in range(20):
            launch(sets[i % 2])
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(iters):
            launch(sets[i % 2])
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / iters

    def check(st, what):
        if st != 0:
            raise mrn.MrnError(st, what)

    for name, dtype, seam, rows, n in (
            ("seam_f16_from_f32_rows4096_n6656", mrn.MRN_F32, mrn.MRN_F16, 4096, 6656),
            ("seam_bf16_from_bf16_rows16384_n4096", mrn.MRN_BF16, mrn.MRN_BF16, 16384, 4096)):
        tdt = torch.float32 if dtype == mrn.MRN_F32 else torch.bfloat16
        sdt = torch.float16 if seam == mrn.MRN_F16 else torch.bfloat16
        e = 4 if dtype == mrn.MRN_F32 else 2
        sets = []
        for _ in range(2):
            x = torch.randn(rows, n, device=dev, generator=gen).to(tdt)
            g = (1 + 0.1 * torch.randn(n, device=dev, generator=gen)).to(sdt)
            u = torch.empty(rows, n, dtype=sdt, device=dev)
            y = torch.empty(rows, n, dtype=sdt, device=dev)
            sets.append((x, g, u, y))

        def fused(t):
            check(mrn.mrn_rmsnorm_seam(t[0].data_ptr(), t[1].data_ptr(), t[3].data_ptr(), rows, n,
                                       1e-5, dtype, seam, sh), name)

        def split(t):
            check(mrn.mrn_rmsnorm_unweighted(t[0].data_ptr(), t[2].data_ptr(), rows, n, 1e-5,
                                             dtype, seam, sh), name)
            check(mrn.mrn_seam_scale(t[2].data_ptr(), t[1].data_ptr(), t[3].data_ptr(), rows, n,
                                     seam, sh), name)

        us_f = timed(fused, sets)
        us_s = timed(split, sets)
        b_f = (e + 2) * rows * n + 2 * n
        b_s = (e + 2) * rows * n + 4 * rows * n + 2 * n
        out[name] = {"GB_per_s": b_f / (us_f * 1e-6) / 1e9, "us_per_call": us_f,
                     "rows_per_s": rows / (us_f * 1e-6), "bytes_per_call": b_f,
                     "split_route": {"GB_per_s": b_s / (us_s * 1e-6) / 1e9, "us_per_call": us_s,
                                     "bytes_per_call": b_s, "launches": 2},
                     "fused_speedup": us_s / us_f,
                     "geometry": mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_SEAM, rows, n, dtype,
                                                        True)}
        del sets
        torch.cuda.empty_cache()
    return out


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_mrn(args)


if __name__ == "__main__":
    sys.exit(main())
