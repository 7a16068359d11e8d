"""Benchmark of the row-normalisation hot path on GB300.

One step = one forward and one backward (trainable: dW / dB computed) of
RMSNorm, LayerNorm and FusedAddRMSNorm on bf16 activations of M x N
(default 8192 x 8192), i.e. every row kernel of the path plus the dW / dB
column reductions, each operation on its own seeded synthetic tensors.
The operations run in the order rms_fwd, ln_fwd, fadd_fwd, rms_bwd, ln_bwd,
fadd_bwd so that no two consecutive operations touch the same tensor, and
L2 is flushed (a write larger than twice the L2) before every step.

Reported (one JSON line on rank 0):
  value        algorithmic HBM bytes of the step / device time of the step
               (CUDA events on the launching stream, L2 flush excluded), GB/s,
               summed over ranks (each rank runs its own replica);
  roofline     the dominant operation (largest share of the step): its
               algorithmic bytes per call / its mean event-timed duration,
               against the measured HBM copy bandwidth;
  per_op       the same for every operation, trainable and frozen;
  e2e          the same metric with host buffers: pinned host -> device copies
               of every input and device -> host copies of every output inside
               the timed region, through the same C-ABI calls (uploads,
               kernels and downloads on three streams ordered by events), with
               the step's own copy roof measured in the same run;
  shapes       per-call times (one call at a time, clean L2) on the pages'
               shape grid, Gemma and FusedAdd shapes: the median over
               shuffled rounds, with an A/A pair as the noise floor;
  cpu_baseline the FP64 CPU oracle on a bounded row sample of the same
               workload, on this host's cores (a reported baseline).

--dtype runs the step on fp16, fp32 or bf16-activations-with-fp32-weights
tensors instead of bf16 (the headline); --impl reference times that oracle
alone (the pages give no runnable reference implementation), on the same
metric and workload.
--grid runs every operation of the shape grid twice, untimed, for an ncu
kernel-duration capture, and prints the call order.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = ("HBM GB/s (% of GB300 peak) & µs/call, bf16 RMSNorm/LayerNorm fwd+bwd at 8192×8192")
OPS = ["rms_fwd", "ln_fwd", "fadd_fwd", "rms_bwd", "ln_bwd", "fadd_bwd"]
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # the vendor HBM3e figure: a secondary denominator only


# ---------------------------------------------------------------------------
# algorithmic bytes (reads of x, dy, residual, dh_out, w, b, rstd, mean plus
# writes of y, h, dx, rstd, mean, dW, dB)
# ---------------------------------------------------------------------------
# activation / weight dtypes of a run (--dtype): synthetic_inputs names and
# element sizes; bf16 is the default and the headline workload
DTYPES = {"bf16": ("bfloat16", "bfloat16", 2, 2), "fp16": ("float16", "float16", 2, 2),
          "fp32": ("float32", "float32", 4, 4), "bf16w32": ("bfloat16", "float32", 2, 4)}
ELEM = [2, 2]   # element sizes of the current run (set by main)


def op_bytes(op, M, N, s=None, sw=None, trainable=True):
    s = ELEM[0] if s is None else s
    sw = ELEM[1] if sw is None else sw
    MN = M * N
    if op == "rms_fwd":
        return 2 * MN * s + N * sw + 4 * M
    if op == "rms_bwd":
        return 3 * MN * s + N * sw + 4 * M + (N * sw if trainable else 0)
    if op == "ln_fwd":
        return 2 * MN * s + 2 * N * sw + 8 * M
    if op == "ln_bwd":
        return 3 * MN * s + N * sw + 8 * M + (2 * N * sw if trainable else 0)
    if op == "fadd_fwd":
        return 4 * MN * s + N * sw + 4 * M
    if op == "fadd_bwd":
        return 4 * MN * s + N * sw + 4 * M + (N * sw if trainable else 0)
    raise ValueError(op)


def launches_per_op(op, trainable=True, world=1):
    """Kernels of ours one call launches: the row kernel; a trainable
    backward adds the column reduce and, sharded over ranks, one rank-order
    sum per gradient (dW, and dB for LayerNorm)."""
    if not (op.endswith("_bwd") and trainable):
        return 1
    return 2 + ((2 if op == "ln_bwd" else 1) if world > 1 else 0)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        v = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
        if isinstance(v, dict):
            v = v.get("value")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def host_inputs(M, N, seed=0, dtype="bf16"):
    """CPU tensors of every operation (distinct seeds per operation)."""
    act, wt = DTYPES[dtype][:2]
    rms = si.norm_case(M, N, seed=seed, dtype=act, w_dtype=wt, with_bias=False)
    ln = si.norm_case(M, N, seed=seed + 1, dtype=act, w_dtype=wt)
    fa = si.norm_case(M, N, seed=seed + 2, dtype=act, w_dtype=wt, with_bias=False, fused_add=True)
    return {"rms": rms, "ln": ln, "fadd": fa}


class Workload:
    """Device tensors of one step; `run(op)` issues one operation.

    With world > 1 the rows are this rank's shard of one M-sharded problem:
    a trainable backward then reduces this rank's dW / dB in FP32 and sums
    them over the ranks in rank order (dist.sharded_backward), inside the
    call."""

    def __init__(self, g, host, M, N, dev="cuda", world=1):
        self.g, self.M, self.N, self.world = g, M, N, world
        bf = host["rms"]["x"].dtype     # activation dtype
        wdt = host["rms"]["w"].dtype    # weight (and dW / dB) dtype
        e = lambda: torch.empty(M, N, dtype=bf, device=dev)  # noqa: E731
        f32 = lambda n: torch.empty(n, dtype=torch.float32, device=dev)  # noqa: E731
        self.t = {}
        for k, case in host.items():
            for name, v in case.items():
                self.t[f"{k}.{name}"] = v.to(dev)
        for k in ("rms", "ln", "fadd"):
            self.t[f"{k}.y"] = e()
            self.t[f"{k}.dx"] = e()
            self.t[f"{k}.rstd"] = f32(M)
            self.t[f"{k}.dw"] = torch.empty(N, dtype=wdt, device=dev)
        self.t["ln.mean"] = f32(M)
        self.t["ln.db"] = torch.empty(N, dtype=wdt, device=dev)
        self.t["fadd.h"] = e()
        nb = max(g.norm_bwd_workspace_bytes(M, N, True, True), 16)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        if world > 1:
            from row_normalization_rmsnorm_gb300 import dist as gdist
            self.gdist = gdist
            self.partials = {k: (f32(N), f32(N)) for k in ("rms", "ln", "fadd")}

    def run(self, op, trainable=True, stream=None):
        g, t = self.g, self.t
        ws = self.ws if trainable else None
        if self.world > 1 and trainable and op.endswith("_bwd"):
            # one M-sharded problem: dW / dB combined over the ranks
            k = op[:-4]
            stats = {"rms": t["rms.rstd"], "ln": (t["ln.mean"], t["ln.rstd"]), "fadd": t["fadd.rstd"]}[k]
            x = t["fadd.h"] if k == "fadd" else t[f"{k}.x"]
            self.gdist.sharded_backward(k, t[f"{k}.dy"], x, t[f"{k}.w"], stats, t[f"{k}.dx"], t[f"{k}.dw"],
                                        t["ln.db"] if k == "ln" else None,
                                        t["fadd.dh_out"] if k == "fadd" else None, 0.0, 1e-6, ws,
                                        self.partials[k])
            return
        if op == "rms_fwd":
            g.norm_rms_fwd(t["rms.x"], t["rms.w"], t["rms.y"], t["rms.rstd"], 0.0, 1e-6, stream)
        elif op == "ln_fwd":
            g.norm_ln_fwd(t["ln.x"], t["ln.w"], t["ln.b"], t["ln.y"], t["ln.mean"], t["ln.rstd"], 0.0, 1e-6,
                          stream)
        elif op == "fadd_fwd":
            g.norm_fused_add_rms_fwd(t["fadd.x"], t["fadd.residual"], t["fadd.w"], t["fadd.y"], t["fadd.h"],
                                     t["fadd.rstd"], 0.0, 1e-6, stream)
        elif op == "rms_bwd":
            g.norm_rms_bwd(t["rms.dy"], t["rms.x"], t["rms.w"], t["rms.rstd"], t["rms.dx"],
                           t["rms.dw"] if trainable else None, ws, 0.0, 1e-6, stream)
        elif op == "ln_bwd":
            g.norm_ln_bwd(t["ln.dy"], t["ln.x"], t["ln.w"], t["ln.mean"], t["ln.rstd"], t["ln.dx"],
                          t["ln.dw"] if trainable else None, t["ln.db"] if trainable else None, ws, 0.0, 1e-6,
                          stream)
        elif op == "fadd_bwd":
            g.norm_fused_add_rms_bwd(t["fadd.dy"], t["fadd.dh_out"], t["fadd.h"], t["fadd.w"], t["fadd.rstd"],
                                     t["fadd.dx"], t["fadd.dw"] if trainable else None, ws, 0.0, 1e-6, stream)
        else:
            raise ValueError(op)

    # tensors a host-buffer user supplies / reads back, per operation
    IN = {"rms_fwd": ["rms.x", "rms.w"], "ln_fwd": ["ln.x", "ln.w", "ln.b"],
          "fadd_fwd": ["fadd.x", "fadd.residual", "fadd.w"],
          "rms_bwd": ["rms.dy"], "ln_bwd": ["ln.dy"], "fadd_bwd": ["fadd.dy", "fadd.dh_out"]}
    OUT = {"rms_fwd": ["rms.y"], "ln_fwd": ["ln.y"], "fadd_fwd": ["fadd.y", "fadd.h"],
           "rms_bwd": ["rms.dx", "rms.dw"], "ln_bwd": ["ln.dx", "ln.dw", "ln.db"],
           "fadd_bwd": ["fadd.dx", "fadd.dw"]}
    # every operation that reads a host-supplied tensor (a forward's input is
    # read again by its backward)
    READERS = {"rms.x": ["rms_fwd", "rms_bwd"], "rms.w": ["rms_fwd", "rms_bwd"], "rms.dy": ["rms_bwd"],
               "ln.x": ["ln_fwd", "ln_bwd"], "ln.w": ["ln_fwd", "ln_bwd"], "ln.b": ["ln_fwd"],
               "ln.dy": ["ln_bwd"], "fadd.x": ["fadd_fwd"], "fadd.residual": ["fadd_fwd"],
               "fadd.w": ["fadd_fwd", "fadd_bwd"], "fadd.dy": ["fadd_bwd"], "fadd.dh_out": ["fadd_bwd"]}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples go to a temporary file; the JSON line carries their summary
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix=f"norm_bench_clocks_rank{index}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.err = open(self.path + ".err", "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=self.err)
            t0 = time.time()   # start timing only once the sampler is producing lines
            while time.time() - t0 < 5 and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.05)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()
            self.err.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------
def host_cores():
    """Threads this process may run on (its CPU affinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_blocks(host, rows, nblocks):
    """FP64 copies of the first `rows` rows of every operation's inputs, cut
    into `nblocks` contiguous row blocks (prepared outside any timed region)."""
    f = lambda t: np.ascontiguousarray(t[:rows].double().numpy())  # noqa: E731
    w = {k: host[k]["w"].double().numpy() for k in host}
    rms, ln, fa = host["rms"], host["ln"], host["fadd"]
    full = dict(rx=f(rms["x"]), rdy=f(rms["dy"]), lx=f(ln["x"]), ldy=f(ln["dy"]),
                fx=f(fa["x"]), fr=f(fa["residual"]), fdy=f(fa["dy"]), fdh=f(fa["dh_out"]))
    cuts = np.linspace(0, rows, nblocks + 1).astype(int)
    blocks = [{k: np.ascontiguousarray(v[lo:hi]) for k, v in full.items()}
              for lo, hi in zip(cuts[:-1], cuts[1:]) if hi > lo]
    return blocks, w, ln["b"].double().numpy()


def oracle_block(a, w, lb):
    """The six operations of one step on one row block; returns the block's
    dW / dB partial sums (the column reduction over its rows)."""
    import oracle
    oracle.rms_fwd(a["rx"], w["rms"], 0.0, 1e-6)
    oracle.ln_fwd(a["lx"], w["ln"], lb, 0.0, 1e-6)
    _, h, _ = oracle.fused_add_rms_fwd(a["fx"], a["fr"], w["fadd"], 0.0, 1e-6)
    _, dw_r, _ = oracle.rms_bwd(a["rx"], a["rdy"], w["rms"], 0.0, 1e-6)
    _, dw_l, db_l, _ = oracle.ln_bwd(a["lx"], a["ldy"], w["ln"], 0.0, 1e-6)
    _, dw_f, _ = oracle.fused_add_rms_bwd(h, a["fdy"], w["fadd"], a["fdh"], 0.0, 1e-6)
    return dw_r, dw_l, db_l, dw_f


def oracle_step(host, rows, threads=1, prepared=None):
    """Run the oracle on the first `rows` rows of every operation's inputs,
    split into `threads` row blocks run concurrently (the oracle's C calls
    release the interpreter lock); the blocks' dW / dB partial sums are added
    in block order.  Returns (seconds, algorithmic bytes of that sample)."""
    from concurrent.futures import ThreadPoolExecutor
    blocks, w, lb = prepared or oracle_blocks(host, rows, threads)
    N = blocks[0]["rx"].shape[1]
    t0 = time.perf_counter()
    if len(blocks) == 1:
        parts = [oracle_block(blocks[0], w, lb)]
    else:
        with ThreadPoolExecutor(len(blocks)) as ex:
            parts = list(ex.map(lambda a: oracle_block(a, w, lb), blocks))
    total = [p.copy() for p in parts[0]]
    for p in parts[1:]:
        for t, q in zip(total, p):
            t += q
    dt = time.perf_counter() - t0
    return dt, sum(op_bytes(op, rows, N) for op in OPS)


def timed_oracle(host, threads, target_s):
    """GB/s of the oracle on `threads` threads: a row sample sized to about
    target_s seconds, repeated until target_s has passed."""
    import oracle
    oracle.build()
    M = host["rms"]["x"].shape[0]
    rows = min(M, 16 * threads)
    dt, _ = oracle_step(host, rows, threads)
    rows = int(min(M, max(16 * threads, rows * (target_s / 2) / max(dt, 1e-3))))
    prepared = oracle_blocks(host, rows, threads)
    total, nbytes, reps = 0.0, 0, 0
    while total < target_s or reps == 0:
        dt, b = oracle_step(host, rows, threads, prepared)
        total += dt
        nbytes += b
        reps += 1
    return nbytes / total / 1e9, rows, reps, total


def cpu_baseline(host, target_s=10.0):
    """The FP64 oracle on a row sample of the same workload, on every core of
    this host (one thread per core, each on its own row block), with the
    single-thread figure beside it."""
    cores = host_cores()
    v, rows, reps, total = timed_oracle(host, cores, target_s)
    v1, rows1, _, total1 = timed_oracle(host, 1, target_s / 3)
    N = host["rms"]["x"].shape[1]
    return {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_thread_value": v1,
            "sample": f"{rows} rows of each of the 6 operations at N={N} in {cores} row blocks on {cores} threads, "
                      f"{reps} repetition(s), {total:.1f} s (FP64 C oracle; dW/dB block partials added in block "
                      f"order); single thread: {rows1} rows, {total1:.1f} s"}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    M, N = args.M, args.N
    ELEM[:] = DTYPES[args.dtype][2:]
    host = host_inputs(M, N, seed=0, dtype=args.dtype)
    import oracle
    oracle.build()
    cores = host_cores()
    rows = max(args.ref_rows, 16 * cores)
    prepared = oracle_blocks(host, rows, cores)
    for _ in range(args.warmup):
        oracle_step(host, rows, cores, prepared)
    times, nbytes = [], 0
    for _ in range(args.steps):
        dt, nbytes = oracle_step(host, rows, cores, prepared)
        times.append(dt)
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.dtype} {M}x{N} RMSNorm+LayerNorm+FusedAddRMSNorm fwd+bwd (trainable)",
                   "M": M, "N": N, "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} rows of each of the 6 operations per step, in {cores} row blocks "
                                   f"on {cores} threads"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--dtype", default="bf16", choices=sorted(DTYPES),
                    help="activation / weight dtypes of the step (bf16/bf16 by default; bf16w32 = bf16 "
                         "activations with fp32 weights and gradients)")
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--ref-rows", type=int, default=1024,
                    help="rows of each operation per reference-arm step (the FP64 oracle on every host core)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ops", default=",".join(OPS),
                    help="comma-separated subset of the step's operations (profiling)")
    ap.add_argument("--no-shapes", action="store_true", help="skip the per-shape table")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the frozen timings, the e2e run and the CPU baseline (profiling)")
    ap.add_argument("--grid", action="store_true",
                    help="run every operation of the shape grid twice, untimed, and print the call order "
                         "(for an ncu kernel-duration capture)")
    ap.add_argument("--traffic", action="store_true",
                    help="run each operation once after an L2 flush and before a read-only L2 scrub, untimed, "
                         "for an ncu DRAM-bytes capture that includes the operation's deferred write-backs")
    ap.add_argument("--traffic-from", metavar="CSV",
                    help="summarise an ncu CSV of a --traffic run into profiles/ncu_traffic_<M>x<N>.json")
    ap.add_argument("--traffic-table", action="store_true",
                    help="collect every profiles/ncu_traffic_<M>x<N>.json into profiles/ncu_traffic_shapes.csv")
    ap.add_argument("--grid-from", nargs=2, metavar=("CSV", "ORDER_LOG"),
                    help="print a markdown table of an ncu kernel-duration CSV of a --grid run, given the "
                         "grid run's own output (its call order)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.grid:
        return run_grid()
    if args.traffic:
        return run_traffic(args.M, args.N)
    if args.traffic_from:
        return summarise_traffic(args.traffic_from, args.M, args.N)
    if args.traffic_table:
        return traffic_table()
    if args.grid_from:
        return summarise_grid(*args.grid_from)

    import row_normalization_rmsnorm_gb300 as g
    from row_normalization_rmsnorm_gb300 import dist as gdist
    ws, rank, local = gdist.rank_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    M, N = args.M, args.N
    ops = [o for o in args.ops.split(",") if o]
    assert all(o in OPS for o in ops), ops
    ELEM[:] = DTYPES[args.dtype][2:]
    host = host_inputs(M, N, seed=rank, dtype=args.dtype)
    wl = Workload(g, host, M, N, world=ws)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")
    scrub = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device="cuda").fill_(1.0)

    def flush_l2():
        # write a buffer larger than L2, then read another one: no line of
        # the step's tensors survives, and the dirty lines of the write are
        # evicted before (not during) the timed step
        flush.zero_()
        scrub.sum()

    def step(events=None):
        flush_l2()
        if events is not None:
            events[0].record(stream)
        for i, op in enumerate(ops):
            wl.run(op, True, stream)
            if events is not None:
                events[i + 1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    g.norm_debug_launches(reset=True)
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for k in range(args.steps):
            step(evs[k])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    launched = g.norm_debug_launches()   # this library's kernels in the timed region (this rank)
    op_ms = {op: [evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps)] for i, op in enumerate(ops)}
    step_ms = [evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps)]
    ms_step = sum(step_ms) / len(step_ms)
    ms_step = gdist.max_over_ranks(ms_step, device="cuda")
    step_bytes = sum(op_bytes(op, M, N) for op in ops)
    value = step_bytes * ws / (ms_step * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # per-operation figures, trainable (inside the timed steps) and frozen
    per_op = {}
    for op in ops:
        us = 1e3 * statistics.mean(op_ms[op])
        b = op_bytes(op, M, N)
        per_op[op] = {"us": us, "GBps": b / us / 1e3, "frac": b / us / 1e3 / peak, "bytes": b}
    for op in ([] if args.no_extras else [o for o in ("rms_bwd", "ln_bwd", "fadd_bwd") if o in ops]):
        # the first call of the frozen instantiation loads its code: untimed
        wl.run(op, False, stream)
        torch.cuda.synchronize()
        ts = []
        for _ in range(max(5, min(50, args.steps // 2))):
            flush_l2()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            wl.run(op, False, stream)
            b_.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b_))
        us = 1e3 * statistics.mean(ts)
        b = op_bytes(op, M, N, trainable=False)
        per_op[op + "_frozen"] = {"us": us, "GBps": b / us / 1e3, "frac": b / us / 1e3 / peak, "bytes": b}

    dom = max(ops, key=lambda op: per_op[op]["us"])
    prof = load_profile_traffic(dom, M, N) if args.dtype == "bf16" else None   # captured for bf16
    roofline = {"bound": "hbm", "kernel": f"{dom} (row kernel"
                + (" + dW/dB column reduce)" if dom.endswith("_bwd") else ")"),
                "achieved": per_op[dom]["GBps"], "peak": peak, "unit": "GB/s",
                "frac": per_op[dom]["GBps"] / peak, "traffic": prof, "peak_kind": peak_kind,
                "algorithmic_bytes_per_call": per_op[dom]["bytes"],
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": per_op[dom]["GBps"] / NOMINAL_HBM_GBS,
                "step_frac": value / ws / peak, "step_frac_of_nominal": value / ws / NOMINAL_HBM_GBS}

    # end to end: host buffers, copies inside the timed region
    e2e = None if args.no_extras else run_e2e(wl, stream, args.e2e_steps, M, N, ops)

    cpu = None
    if rank == 0 and ws == 1 and not (args.no_cpu_baseline or args.no_extras):
        cpu = cpu_baseline(host)
    shapes = None if (args.no_extras or args.no_shapes) else shape_table(g, flush_l2)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
            "config": {"workload": f"{args.dtype} {M}x{N} RMSNorm+LayerNorm+FusedAddRMSNorm fwd+bwd (trainable)",
                       "M": M, "N": N, "ops": ops,
                       "l2": "flushed before every step (zero-fill of 2x L2, then a read of another 2x L2 "
                             "so the flush's dirty lines are written back before timing); every tensor > L2",
                       "timing": "CUDA events on the launching stream; flush excluded",
                       "wall_s_timed_region": wall,
                       "parallelism": ("1 GPU" if ws == 1 else
                                       f"M-sharded x{ws}: each rank normalises {M} rows of one {M * ws}x{N} "
                                       "problem; the backward's dW/dB are summed over ranks in rank order "
                                       "(NCCL all_gather) inside the step")},
            "roofline": roofline,
            "per_op": per_op,
            "shapes": shapes,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launched * ws,   # counted by the library; every rank runs the same step
            "gpu_launches_expected": args.steps * ws * sum(launches_per_op(op, world=ws) for op in ops),
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


# Shapes the pages report on ("perf(norm): ...", Benchmark Results: the
# frozen-parameter backward grid; "fix(cutedsl): ...", Benchmark results:
# Gemma RMSNorm and FusedAddRMSNorm), timed one call at a time with a clean
# L2, as context for the pages' numbers (other GPUs).
GRID_SHAPES = [(2048, 4096), (4096, 4096), (4096, 8192), (8192, 4096), (8192, 8192)]
GEMMA_SHAPES = [(1, 4096), (128, 4096), (2048, 4096), (8192, 4096), (128, 8192), (2048, 8192), (128, 18432)]
FADD_SHAPES = [(128, 4096), (2048, 4096), (2048, 8192)]


def grid_families():
    """(M, N) -> operation families of the shape grid: RMSNorm and LayerNorm on
    the bf16 grid, FusedAdd on its shapes and at 8192x8192, RMSNorm on the
    Gemma shapes."""
    fams = {}
    for sh in GRID_SHAPES:
        fams.setdefault(sh, []).extend(["rms", "ln"])
    for sh in FADD_SHAPES + [(8192, 8192)]:
        fams.setdefault(sh, []).append("fadd")
    for sh in GEMMA_SHAPES:
        if "rms" not in fams.setdefault(sh, []):
            fams[sh].append("rms")
    return fams


def run_grid():
    """Each (shape, operation) of grid_families() twice -- forward, trainable
    backward, frozen backward -- with nothing timed, so that an ncu launch
    list (gpu__time_duration) gives every kernel's duration; the JSON line
    lists the calls in launch order (a trainable backward launches its row
    kernel and then the column reduce)."""
    import row_normalization_rmsnorm_gb300 as g
    st = torch.cuda.current_stream()
    order = []
    for (M, N), fams in grid_families().items():
        wl = Workload(g, host_inputs(M, N, 0), M, N)
        for fam in fams:
            for op, tr in [(fam + "_fwd", True), (fam + "_bwd", True), (fam + "_bwd", False)]:
                for rep in range(2):
                    wl.run(op, tr, st)
                    order.append([M, N, op, tr, rep])
        torch.cuda.synchronize()
        del wl
        torch.cuda.empty_cache()
    print(json.dumps({"grid_order": order}), flush=True)
    return 0


def shape_items(g, gen):
    """The calls of the shape table, keyed (family, M, N, call): the RMSNorm
    and LayerNorm forward, trainable and frozen backward on the bf16 grid,
    the Gemma RMSNorm forward and forward + backward, the FusedAdd forward
    and forward + backward.  Tensors are made once per shape and shared by
    every call on it (the forward runs first so the saved statistics are
    valid)."""
    tens = {}

    def tensors(M, N):
        if (M, N) in tens:
            return tens[(M, N)]
        bf = dict(dtype=torch.bfloat16, device="cuda")
        r = lambda: torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16)  # noqa: E731
        t = {"x": r(), "dy": r(), "res": r(), "dh": r(), "y": torch.empty(M, N, **bf),
             "dx": torch.empty(M, N, **bf), "h": torch.empty(M, N, **bf),
             "w": (1 + 0.1 * torch.randn(N, device="cuda", generator=gen)).to(torch.bfloat16),
             "wg": (0.01 * torch.randn(N, device="cuda", generator=gen)).to(torch.bfloat16),
             "b": (0.1 * torch.randn(N, device="cuda", generator=gen)).to(torch.bfloat16),
             "rstd": torch.empty(M, device="cuda"), "mean": torch.empty(M, device="cuda"),
             "dw": torch.empty(N, **bf), "db": torch.empty(N, **bf)}
        t["ws"] = torch.empty(max(16, g.norm_bwd_workspace_bytes(M, N, True, True)), dtype=torch.uint8,
                              device="cuda")
        tens[(M, N)] = t
        return t

    items = {}
    for M, N in GRID_SHAPES:
        t = tensors(M, N)
        items[("rms", M, N, "fwd_us")] = lambda t=t: g.norm_rms_fwd(t["x"], t["w"], t["y"], t["rstd"])
        items[("rms", M, N, "bwd_us")] = lambda t=t: g.norm_rms_bwd(t["dy"], t["x"], t["w"], t["rstd"], t["dx"],
                                                                    t["dw"], t["ws"])
        items[("rms", M, N, "bwd_frozen_us")] = lambda t=t: g.norm_rms_bwd(t["dy"], t["x"], t["w"], t["rstd"],
                                                                           t["dx"])
        items[("ln", M, N, "fwd_us")] = lambda t=t: g.norm_ln_fwd(t["x"], t["w"], t["b"], t["y"], t["mean"],
                                                                  t["rstd"])
        items[("ln", M, N, "bwd_us")] = lambda t=t: g.norm_ln_bwd(t["dy"], t["x"], t["w"], t["mean"], t["rstd"],
                                                                  t["dx"], t["dw"], t["db"], t["ws"])
        items[("ln", M, N, "bwd_frozen_us")] = lambda t=t: g.norm_ln_bwd(t["dy"], t["x"], t["w"], t["mean"],
                                                                         t["rstd"], t["dx"])
    for M, N in GEMMA_SHAPES:
        t = tensors(M, N)
        fwd = lambda t=t: g.norm_rms_fwd(t["x"], t["wg"], t["y"], t["rstd"], 1.0)  # noqa: E731
        items[("gemma_rms", M, N, "fwd_us")] = fwd
        items[("gemma_rms", M, N, "fwd_bwd_us")] = lambda t=t, fwd=fwd: (
            fwd(), g.norm_rms_bwd(t["dy"], t["x"], t["wg"], t["rstd"], t["dx"], t["dw"], t["ws"], 1.0))
    for M, N in FADD_SHAPES:
        t = tensors(M, N)
        fwd = lambda t=t: g.norm_fused_add_rms_fwd(t["x"], t["res"], t["w"], t["y"], t["h"], t["rstd"], 1.0)  # noqa
        items[("fadd_rms", M, N, "fwd_us")] = fwd
        items[("fadd_rms", M, N, "fwd_bwd_us")] = lambda t=t, fwd=fwd: (
            fwd(), g.norm_fused_add_rms_bwd(t["dy"], t["dh"], t["h"], t["w"], t["rstd"], t["dx"], t["dw"],
                                            t["ws"], 1.0))
    # forwards first, so that every backward reads valid statistics
    for k, fn in items.items():
        if k[3] == "fwd_us":
            fn()
    return items


AA_ITEM = ("rms", 8192, 8192, "fwd_us")


def shape_table(g, flush_l2, rounds=11, calls=4, warm_ms=5.0, seed=0):
    """Per-call times on the pages' shapes, one call at a time with a clean L2.

    Every item of shape_items() is timed in `rounds` rounds.  A round visits
    all items in a fresh shuffle (seeded) and times `calls` calls of each,
    flushing L2 before every call and bracketing the call alone with CUDA
    events.  An item's figure is the median over rounds of its per-round
    mean: the event clock here ticks in ~2 us steps, so one call's time is
    coarse and the mean over a few calls dithers it.  One item (the RMSNorm
    forward at 8192x8192) is timed twice as two independent items, an A/A
    pair whose gap is the table's noise floor.  Every item runs untimed for
    at least `warm_ms` before the first round."""
    import random
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    items = shape_items(g, gen)
    keys = list(items) + [AA_ITEM + ("aa",)]
    fn_of = lambda k: items[k[:4]]  # noqa: E731

    t0 = time.perf_counter()
    while True:
        for k in keys:
            fn_of(k)()
        torch.cuda.synchronize()
        if (time.perf_counter() - t0) * 1e3 >= warm_ms:
            break

    rng = random.Random(seed)
    per_round = {k: [] for k in keys}
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    for _ in range(rounds):
        order = keys[:]
        rng.shuffle(order)
        for k in order:
            fn = fn_of(k)
            for a, b in ev:
                flush_l2()
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            per_round[k].append(statistics.mean(a.elapsed_time(b) * 1e3 for a, b in ev))

    med = {k: statistics.median(v) for k, v in per_round.items()}
    rows = {}
    for k in items:
        fam, M, N, call = k
        r = rows.setdefault((fam, M, N), {"op": fam, "M": M, "N": N})
        r[call] = round(med[k], 2)
        q = statistics.quantiles(per_round[k], n=10)   # the spread over rounds
        r[call[:-3] + "_p10_p90_us"] = [round(q[0], 2), round(q[-1], 2)]
    for (fam, M, N), r in rows.items():
        if "bwd_frozen_us" in r:
            r["bwd_frozen_GBps"] = round(op_bytes(fam + "_bwd", M, N, trainable=False) / r["bwd_frozen_us"] / 1e3)
    a, b = med[AA_ITEM], med[AA_ITEM + ("aa",)]
    return {"method": f"median over {rounds} rounds (shuffled order, seed {seed}) of the mean of {calls} "
                      f"event-timed calls, L2 flushed before each call; >= {warm_ms:g} ms warm-up; "
                      f"*_p10_p90_us: 10th and 90th percentiles over the rounds",
            "aa_pair": {"item": "rms_fwd 8192x8192", "a_us": round(a, 2), "b_us": round(b, 2),
                        "rel_gap": round(abs(a - b) / min(a, b), 4)},
            "rows": list(rows.values())}


def kernel_source_hash():
    """Hash of the code that decides what the GPU runs and how it is launched
    -- the kernels, their helpers, the launch-shape rules and the per-op
    instantiations -- with comments and blank space removed, so that only a
    change to that code invalidates committed counters.  The entry points'
    argument checks (api.cu) and the no-allocation wrapper are not part of it."""
    import glob
    import hashlib
    import re
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "row_normalization_rmsnorm_gb300", "csrc", "*"))):
        if not f.endswith((".cu", ".cuh", ".h")) or os.path.basename(f) in ("api.cu", "noalloc.cu"):
            continue
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(os.path.basename(f).encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


TRAFFIC_ORDER = OPS   # the operations of a --traffic run, in launch order


def run_traffic(M, N):
    """One round of warm-up, then for each operation of the step: an L2 flush
    (a write, then a read, of 2x L2), the operation (trainable), and a
    read-only scrub of 2x L2.  The scrub only reads, so the DRAM bytes it
    writes are the operation's dirty lines evicted from L2: an ncu capture of
    dram__bytes_read/write over every launch, with ncu's own cache flushing
    off (--cache-control none), gives each operation's whole DRAM traffic,
    its deferred write-backs included (--traffic-from)."""
    import row_normalization_rmsnorm_gb300 as g
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream()
    wl = Workload(g, host_inputs(M, N, 0), M, N)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")
    scrub = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device="cuda").fill_(1.0)
    for op in TRAFFIC_ORDER:   # warm-up: code loaded, launch shapes cached
        wl.run(op, True, st)
    torch.cuda.synchronize()
    for op in TRAFFIC_ORDER:
        flush.zero_()
        scrub.sum()
        wl.run(op, True, st)
        scrub.sum()
    torch.cuda.synchronize()
    print(json.dumps({"traffic_order": TRAFFIC_ORDER, "M": M, "N": N}), flush=True)
    return 0


def summarise_traffic(csv_path, M, N):
    """Per-call DRAM bytes of every operation from an ncu CSV of a --traffic
    run (metrics dram__bytes_read.sum, dram__bytes_write.sum per launch):
    the last len(OPS) groups of [flush write, flush read, op kernels, scrub]
    are attributed in launch order; an operation's traffic is its kernels'
    reads and writes plus the writes of the scrub after it."""
    import csv
    rows = {}
    with open(csv_path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        key = (int(r["ID"]), r["Kernel Name"])
        v = float(r["Metric Value"].replace(",", ""))
        unit = r.get("Metric Unit", "byte")
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1024, "MB": 1 << 20, "GB": 1 << 30,
                 "ns": 1e-3, "nsecond": 1e-3, "us": 1, "usecond": 1, "ms": 1e3, "msecond": 1e3}.get(unit, 1)
        rows.setdefault(key, {})[r["Metric Name"]] = v * scale   # bytes, or microseconds for durations
    launches = [(k[1], m) for k, m in sorted(rows.items())]
    ours = lambda name: any(t in name for t in ("staged_kernel", "loop_kernel", "colreduce"))  # noqa: E731
    # walk backwards: each operation is a run of our kernels followed by one scrub (a torch reduction)
    out, i = {}, len(launches) - 1
    for op in reversed(TRAFFIC_ORDER):
        scrub = launches[i]
        assert not ours(scrub[0]), scrub[0]
        j = i - 1
        kernels = []
        while j >= 0 and ours(launches[j][0]):
            kernels.append(launches[j])
            j -= 1
        kernels.reverse()
        rd = sum(m.get("dram__bytes_read.sum", 0.0) for _, m in kernels)
        wr = sum(m.get("dram__bytes_write.sum", 0.0) for _, m in kernels)
        wb = scrub[1].get("dram__bytes_write.sum", 0.0)
        us = sum(m.get("gpu__time_duration.sum", 0.0) for _, m in kernels)
        out[op] = {"kernels": [n for n, _ in kernels], "dram_read": rd, "dram_write": wr,
                   "deferred_write_back": wb, "per_call": rd + wr + wb,
                   "algorithmic": op_bytes(op, M, N), "ratio": (rd + wr + wb) / op_bytes(op, M, N),
                   "kernel_us": us, "dram_GBps_in_kernel": (rd + wr) / us / 1e3 if us else None}
        i = j - 2   # skip the flush's write and read kernels
    res = {"workload": f"bf16 {M}x{N}, one call per operation, trainable", "source_hash": kernel_source_hash(),
           "command": f"ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
                      f"--cache-control none --clock-control none --csv --log-file traffic.csv "
                      f"python bench.py --traffic --M {M} --N {N}",
           "note": "per_call = the operation's kernels' DRAM reads and writes plus the DRAM writes of the "
                   "read-only L2 scrub that follows it (its dirty lines written back late)",
           "traffic": out}
    path = os.path.join(ROOT, "profiles", f"ncu_traffic_{M}x{N}.json")
    with open(path, "w") as f:
        json.dump(res, f, indent=1)
    print(json.dumps({k: round(v["ratio"], 4) for k, v in out.items()}))
    return 0


def traffic_table():
    """One CSV of every committed per-shape traffic capture: per shape and
    operation, DRAM bytes read, written inside the kernels and written back
    later, their total per call against the algorithmic bytes, and whether
    the capture was taken from the current kernel sources."""
    import csv
    import glob
    import re
    cur = kernel_source_hash()
    rows = []
    for path in glob.glob(os.path.join(ROOT, "profiles", "ncu_traffic_*x*.json")):
        m = re.search(r"ncu_traffic_(\d+)x(\d+)\.json$", path)
        if not m:
            continue
        with open(path) as f:
            d = json.load(f)
        for op in OPS:
            t = d["traffic"].get(op)
            if t is None:
                continue
            rows.append({"M": int(m.group(1)), "N": int(m.group(2)), "op": op,
                         "dram_read_MB": round(t["dram_read"] / 1e6, 2),
                         "dram_write_in_kernel_MB": round(t["dram_write"] / 1e6, 2),
                         "deferred_write_back_MB": round(t["deferred_write_back"] / 1e6, 2),
                         "per_call_MB": round(t["per_call"] / 1e6, 2),
                         "algorithmic_MB": round(t["algorithmic"] / 1e6, 2),
                         "ratio": round(t["ratio"], 4),
                         "kernel_us": round(t["kernel_us"], 2) if t.get("kernel_us") else None,
                         "dram_GBps_in_kernel": round(t["dram_GBps_in_kernel"]) if t.get("dram_GBps_in_kernel") else None,
                         "algorithmic_GBps": (round(t["algorithmic"] / t["kernel_us"] / 1e3)
                                              if t.get("kernel_us") else None),
                         "current_sources": d.get("source_hash") == cur})
    rows.sort(key=lambda r: (r["M"] * r["N"], r["M"], OPS.index(r["op"])))
    out = os.path.join(ROOT, "profiles", "ncu_traffic_shapes.csv")
    with open(out, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=list(rows[0]) if rows else ["M"])
        w.writeheader()
        w.writerows(rows)
    print(f"{len(rows)} rows -> {out}")
    return 0


def summarise_grid(csv_path, order_log):
    """Markdown table of a --grid ncu capture (gpu__time_duration.sum of our
    kernels, in launch order): for each (shape, operation) the second of its
    two calls, row kernel plus column reduce, with GB/s of algorithmic bytes
    and the fraction of the measured HBM peak."""
    import csv
    order = None
    with open(order_log) as f:
        for ln in f:
            if ln.startswith("{") and "grid_order" in ln:
                order = json.loads(ln)["grid_order"]
    with open(csv_path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    launches = []
    for r in csv.DictReader(lines):
        if r["Metric Name"] == "gpu__time_duration.sum":
            unit = r.get("Metric Unit", "ns")
            v = float(r["Metric Value"].replace(",", "")) * {"ns": 1e-3, "us": 1.0, "usecond": 1.0,
                                                             "nsecond": 1e-3, "ms": 1e3, "msecond": 1e3}.get(unit, 1e-3)
            launches.append((int(r["ID"]), r["Kernel Name"], v))
    launches.sort()
    peak, kind = measured_peak()
    rows, i = [], 0
    for M, N, op, tr, rep in order:
        n = 2 if (op.endswith("_bwd") and tr) else 1
        ks = launches[i:i + n]
        i += n
        if rep != 1:
            continue
        row_us = ks[0][2]
        cr_us = ks[1][2] if n == 2 else 0.0
        b = op_bytes(op, M, N, trainable=tr)
        gbs = b / (row_us + cr_us) / 1e3
        name = ks[0][1].replace("gb300norm::", "").replace("__nv_bfloat16", "bf16").split("(")[0]
        rows.append(f"| {M}×{N} | {op}{'' if tr or not op.endswith('_bwd') else ' frozen'} | {row_us:.1f} | "
                    f"{cr_us:.1f} | {gbs:.0f} | {100 * gbs / peak:.0f} % | `{name}` |")
    assert i == len(launches), (i, len(launches))
    print(f"| shape | op | row kernel µs | + column reduce µs | GB/s (row + reduce) | % of {kind} {peak:.0f} GB/s "
          f"| kernel |")
    print("|---|---|---|---|---|---|---|")
    print("\n".join(rows))
    return 0


def load_profile_traffic(op, M, N):
    """DRAM bytes (read + write) per call of the operation's kernels, from the
    committed ncu capture of this exact workload -- or None when there is
    none, or when the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"ncu_traffic_{M}x{N}.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    t = d.get("traffic", {}).get(op)
    return None if t is None else t.get("per_call")


def run_e2e(wl, stream, steps, M, N, ops, windows=5):
    """Same metric through the same calls, from pinned host buffers."""
    host_in = {k: torch.empty_like(wl.t[k], device="cpu").pin_memory()
               for op in ops for k in Workload.IN[op]}
    for k, v in host_in.items():
        v.copy_(wl.t[k])
    host_out = {k: torch.empty_like(wl.t[k], device="cpu").pin_memory()
                for op in ops for k in Workload.OUT[op]}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    # Three streams: uploads (`up`), kernels (`stream`) and downloads (`side`),
    # ordered by events, so the copies of both directions run while kernels
    # do.  An operation's kernel waits for its uploads; its download waits for
    # its kernel; the next step's upload into a tensor waits until every
    # kernel that reads it has run, and an operation's next kernel until its
    # previous outputs are downloaded.  Inputs and outputs are disjoint
    # buffers.
    up = torch.cuda.Stream()
    side = torch.cuda.Stream()
    uploaded = {op: torch.cuda.Event() for op in ops}
    done = {op: torch.cuda.Event() for op in ops}
    out_free = {op: torch.cuda.Event() for op in ops}
    started = set()

    def one():
        for op in ops:
            for r in {r for k in Workload.IN[op] for r in Workload.READERS[k]}:
                if r in started:
                    up.wait_event(done[r])     # every earlier reader is done with these inputs
            with torch.cuda.stream(up):
                for k in Workload.IN[op]:
                    wl.t[k].copy_(host_in[k], non_blocking=True)
            uploaded[op].record(up)
            stream.wait_event(uploaded[op])
            if op in started:
                stream.wait_event(out_free[op])
            wl.run(op, True, stream)
            done[op].record(stream)
            side.wait_event(done[op])
            with torch.cuda.stream(side):
                for k in Workload.OUT[op]:
                    host_out[k].copy_(wl.t[k], non_blocking=True)
            out_free[op].record(side)
            started.add(op)

    one()
    torch.cuda.synchronize()
    # `windows` timed windows of `steps` steps each; the median window is
    # reported (one window can catch a stall of the shared host link)
    per_window = []
    for _ in range(windows):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_event(a)
        side.wait_event(a)
        for _ in range(steps):
            one()
        stream.wait_stream(side)   # the last downloads are inside the timed region
        stream.wait_stream(up)
        b.record(stream)
        torch.cuda.synchronize()
        per_window.append(a.elapsed_time(b) / steps)
    ms = statistics.median(per_window)
    step_bytes = sum(op_bytes(op, M, N) for op in ops)
    roof = copy_roof(wl, host_in, host_out, stream, side)
    roof["value_at_roof"] = step_bytes / (roof["both_ms"] * 1e-3) / 1e9
    roof["frac"] = roof["both_ms"] / ms
    return {"value": step_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "windows_ms_per_step": [round(x, 4) for x in per_window], "steps_per_window": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "copy_roof": roof}


def copy_roof(wl, host_in, host_out, stream, side, reps=3):
    """The e2e step's own roof, measured in the same run: the step's uploads
    alone, its downloads alone, and both at once on two streams (the two
    directions of the host link), each the best of `reps` event-timed
    rounds.  `both_ms` is the least time the e2e step could take if its
    kernels cost nothing."""
    def timed(up, down):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            side.wait_event(a)
            if up:
                for k, v in host_in.items():
                    wl.t[k].copy_(v, non_blocking=True)
            if down:
                with torch.cuda.stream(side):
                    for k, v in host_out.items():
                        v.copy_(wl.t[k], non_blocking=True)
            stream.wait_stream(side)
            b.record(stream)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best
    up_ms, down_ms, both_ms = timed(True, False), timed(False, True), timed(True, True)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    return {"h2d_GBps": h2d / (up_ms * 1e-3) / 1e9, "d2h_GBps": d2h / (down_ms * 1e-3) / 1e9,
            "both_ms": both_ms, "both_GBps": (h2d + d2h) / (both_ms * 1e-3) / 1e9,
            "how": "pinned host buffers of the step, cudaMemcpyAsync per tensor, best of 3 (CUDA events)"}


if __name__ == "__main__":
    sys.exit(main())
