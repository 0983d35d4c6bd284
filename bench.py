"""SparseGemv benchmark: achieved HBM GB/s and us/call at M = 1.

Workload (default): the 7B-style decoder layer set -- q, k, v, o 4096x4096,
gate, up 11008x4096, down 4096x11008 -- each matrix N:4 pruned and INT4
group-quantised with a seeded per-matrix (N, g), x one binary16 row.  One
step = the seven SparseGemv calls of one decode step.  Weights are
synthetic and seeded (the paper's model is not public).

Timing: W warm-up steps, then exactly K steps, as CUDA graphs replayed on
one stream, bracketed by a barrier + device synchronisation; CUDA events
on that stream give the duration; steps rotate over enough distinct copies
of the packed weights (> 4x the L2 size) that no weight byte is served
from L2.  value = algorithmic bytes of all steps on all ranks / max time.

Prints one JSON line on rank 0.  --impl reference times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SparseGemv achieved HBM GB/s and us/call (M=1) vs 8 TB/s roofline"
NOMINAL_HBM_GBS = 8000.0   # the metric's stated roofline; roofline.peak is the measured copy rate
WORKLOAD = ("7B decoder layer set, M=1: q,k,v,o 4096x4096; gate,up 11008x4096; "
            "down 4096x11008; seeded per-matrix (N:4, group)")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no collective on the data path)
# ---------------------------------------------------------------------------

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, world: int, device=None) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks: NVML polled from a thread during the timed region
# ---------------------------------------------------------------------------

_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting",
            0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sync_boost",
            0x40: "sw_thermal_slowdown", 0x80: "hw_thermal_slowdown",
            0x100: "hw_power_brake_slowdown", 0x200: "display_clock_setting"}


class ClockSampler:
    """Reads SM clock and clock-event reasons (read-only NVML queries)."""

    def __init__(self, index: int, period_s: float = 0.0002):
        self.samples = []
        self.period = period_s
        self.ok = False
        self._stop = threading.Event()
        self._thr = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return
            self._nv, self._h = nv, h
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _read(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(c))
        fn = getattr(self._nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nv.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self._h, ctypes.byref(r))
        return c.value, r.value

    def _loop(self):
        while not self._stop.is_set():
            self.samples.append(self._read())
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._thr = threading.Thread(target=self._loop, daemon=True)
            self._thr.start()

    def count(self) -> int:
        return len(self.samples)

    def stop(self):
        if self._thr:
            self._stop.set()
            self._thr.join()
            self.samples.append(self._read())

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "source": "unavailable"}
        mhz = [s[0] for s in self.samples]
        reasons = set()
        for _, bits in self.samples:
            for b, name in _REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz),
                "samples_timed": getattr(self, "timed", len(mhz)),
                "source": "nvml poll every ~0.2 ms during the timed region (topped up "
                          "to >= 10 samples by replaying the same steps untimed)"}


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------

# matrices of the layer that share one activation x
GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def workload(seed: int = 0):
    return synth.config3(seed)


def step_bytes(gvs, m=1):
    return sum(g.bytes(m) for g in gvs)


def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s"


def read_traffic(kernel_tag: str):
    """Per-launch DRAM bytes from a committed ncu summary, or None if the
    summary is missing or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel_tag)
    if not ent:
        return None
    from sparse_weight_only_gb300.build import _stamp
    files = ent.get("source_files")
    if not files or ent.get("source_stamp") != _stamp(files):
        return None
    return ent


TRAFFIC_FILES = ["sgemv_m1.cu", "sgemv_internal.cuh", "sgemv_api.cu"]


def record_traffic(csv_path: str, out_path: str, command: str) -> int:
    """Writes the per-step DRAM record from an ncu CSV log holding the k_m1
    launches of one grouped step (dram__bytes_read.sum, dram__bytes_write.sum
    and gpu__time_duration.sum per launch), stamped with the current source of
    those kernels -- the record is re-taken, never re-stamped."""
    import csv
    from sparse_weight_only_gb300.build import _stamp
    per = {}
    hdr = None
    with open(csv_path) as f:
        for row in csv.reader(f):
            if not row:
                continue
            if row[0] == "ID":
                hdr = row
                continue
            if hdr is None or len(row) != len(hdr):
                continue
            d = dict(zip(hdr, row))
            ent = per.setdefault(int(d["ID"]), {"kernel": d["Kernel Name"]})
            ent[d["Metric Name"]] = float(d["Metric Value"].replace(",", ""))
    launches = [per[k] for k in sorted(per)]
    if not launches or any("dram__bytes_read.sum" not in l for l in launches):
        print(f"no DRAM counters in {csv_path}", file=sys.stderr)
        return 1
    total = sum(l["dram__bytes_read.sum"] + l.get("dram__bytes_write.sum", 0.0) for l in launches)
    rec = {"sgemv_layerset_m1": {
        "bytes_per_step": int(total),
        "algorithmic_bytes_per_step": int(step_bytes(workload(0), 1)),
        "launches_per_step": len(launches),
        "per_launch": [{"kernel": l["kernel"].split("(")[0].split("::")[-1],
                        "dram_bytes": int(l["dram__bytes_read.sum"] + l.get("dram__bytes_write.sum", 0.0)),
                        "ncu_us": round(l.get("gpu__time_duration.sum", 0.0) / 1e3, 3)}
                       for l in launches],
        "source_files": TRAFFIC_FILES,
        "source_stamp": _stamp(TRAFFIC_FILES),
        "command": command,
        "note": "sum of dram__bytes_read.sum + dram__bytes_write.sum over the k_m1 launches "
                "of one grouped step (q+k+v in one launch, o, gate+up, down)",
    }}
    with open(out_path, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print(json.dumps(rec["sgemv_layerset_m1"]))
    return 0


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline key)
# ---------------------------------------------------------------------------

def oracle_time(packed, budget_s: float, min_rows: int = 1):
    """Times the oracle's matvec on whole row blocks of every matrix until
    `budget_s` has elapsed.  Returns (bytes, seconds, rows_done)."""
    import oracle
    total_b, total_t, rows_done = 0, 0.0, 0
    nmat = len(packed)
    i = 0
    while True:
        gv, p, x = packed[i % nmat]
        nr = max(min_rows, gv.rows // 64)
        start = (i // nmat * nr) % max(gv.rows - nr + 1, 1)
        rows = np.arange(start, start + nr, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.matvec(p, x, rows)
        total_t += time.perf_counter() - t0
        frac = nr / gv.rows
        total_b += frac * gv.packed_bytes() + 2 * gv.cols + 2 * nr
        rows_done += nr
        i += 1
        if total_t >= budget_s and i >= nmat:
            break
    return total_b, total_t, rows_done


def oracle_time_threads(packed, budget_s: float, threads: int):
    """The same row blocks as oracle_time, spread over `threads` host threads
    (the oracle's C matvec runs without the interpreter lock), in whole passes
    over the matrices until `budget_s` of wall time has elapsed.  Returns
    (bytes, seconds, rows_done)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    tasks = []
    for gv, p, x in packed:
        nr = max(1, gv.rows // 64)
        for start in range(0, gv.rows - nr + 1, nr):
            tasks.append((gv, p, x, start, nr))
    # interleave the matrices so that any prefix samples all of them
    tasks.sort(key=lambda t: (t[3] // t[4], t[0].name))
    t0 = time.perf_counter()

    def one(task):
        gv, p, x, start, nr = task
        if time.perf_counter() - t0 >= budget_s:
            return 0.0, 0
        oracle.matvec(p, x, np.arange(start, start + nr, dtype=np.int64))
        return nr / gv.rows * gv.packed_bytes() + 2 * gv.cols + 2 * nr, nr

    total_b, total_r = 0.0, 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while True:   # whole passes over the layer set until the budget is spent
            done = list(ex.map(one, tasks))
            total_b += sum(d[0] for d in done)
            total_r += sum(d[1] for d in done)
            if time.perf_counter() - t0 >= budget_s:
                break
    return total_b, time.perf_counter() - t0, total_r


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    gvs = workload(args.seed)
    packed = []
    for gv in gvs:
        W = gv.weight()
        packed.append((gv, oracle.pack(W, gv.n_keep, gv.group), gv.x(1)))
        del W
    # each step: one row block (1/64 of the rows) of one matrix, rotating;
    # the whole W + K run is bounded to about two minutes
    per_step = max(0.0005, min(1.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_time(packed, 0.0)
    b, t, rows = 0.0, 0.0, 0
    for _ in range(args.steps):
        bb, tt, rr = oracle_time(packed, per_step)
        b, t, rows = b + bb, t + tt, rows + rr
    gbs = b / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m": 1, "seed": args.seed},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} rows in row blocks of 1/64 of each matrix, "
                                   "single-threaded fp64 dequantise + naive matvec"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def run_batch_only(args, local):
    """--batch-only M: the verification-batch layer set (seven 2:4 g128
    matrices) at M rows, timed as in batch_m; for ncu captures of the batch
    kernels."""
    import torch
    import sparse_weight_only_gb300 as swo
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    swo.build()
    swo.load()
    stream = torch.cuda.Stream(device=dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 * 2 ** 20
    out = run_batch_sweep(args, swo, dev, stream, l2, None, (args.batch_only,))
    print(json.dumps({"batch_only": args.batch_only, "config4": out}), flush=True)
    return 0


def run_ours(args, rank, world, local):
    import torch
    import sparse_weight_only_gb300 as swo

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    swo.build()
    swo.load()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    m = 1

    gvs = workload(args.seed)
    t_pack = time.perf_counter()
    base = []
    for gv in gvs:
        W = gv.weight()
        h = swo.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, max_m=m,
                           device=local)
        h.pack(W)
        del W
        base.append(h)
    t_pack = time.perf_counter() - t_pack
    canon = [h.export_canonical() for h in base]

    sb = step_bytes(gvs, m)
    wbytes = sum(g.packed_bytes() for g in gvs)
    copies = max(2, math.ceil(4 * l2 / wbytes) + 1)
    sets = [base]
    for _ in range(copies - 1):
        cp = []
        for gv, c in zip(gvs, canon):
            h = swo.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, max_m=m,
                               device=local)
            h.import_canonical(*c)
            cp.append(h)
        sets.append(cp)

    # x is shared where a decoder layer shares it: q, k, v read one x and
    # gate, up read one x; o and down have their own
    pos = {g.name: i for i, g in enumerate(gvs)}
    groups = [[pos[n] for n in grp] for grp in GROUPS]
    xs = [None] * len(gvs)
    for grp in groups:
        x0 = torch.from_numpy(gvs[grp[0]].x(m)).to(dev)
        for i in grp:
            xs[i] = x0
    ys = [torch.empty((m, gv.rows), dtype=torch.float16, device=dev) for gv in gvs]
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    grouped = not args.ungrouped

    def launch_step(k, grouped=grouped):
        st = sets[k % copies]
        if grouped:
            for grp in groups:
                if len(grp) == 1:
                    st[grp[0]].run(xs[grp[0]], ys[grp[0]], sptr)
                else:
                    swo.run_group([st[i] for i in grp], xs[grp[0]],
                                  [ys[i] for i in grp], sptr)
        else:
            for h, x, y in zip(st, xs, ys):
                h.run(x, y, sptr)

    def capture(nsteps, first, grouped=grouped):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for k in range(nsteps):
                    launch_step(first + k, grouped)
        return g

    # graphs: a block of `copies` steps (each copy once) and a remainder
    block = copies
    with torch.cuda.stream(stream):
        for k in range(2):
            launch_step(k)            # eager warm-up before capture
            launch_step(k, not grouped)
    torch.cuda.synchronize()
    g_block = capture(block, 0)

    def replay(nsteps, rem_graphs, gb=None):
        q, r = divmod(nsteps, block)
        for _ in range(q):
            (gb or g_block).replay()
        if r:
            rem_graphs[r].replay()

    rem = {}
    for n in {args.steps % block, args.warmup % block} - {0}:
        rem[n] = capture(n, 0)

    with torch.cuda.stream(stream):
        replay(args.warmup, rem)
    torch.cuda.synchronize()

    # Timed region: exactly K steps, bracketed by barrier + synchronize,
    # replayed `repeats` times with fresh events; value and ms_per_step are
    # the median repetition (the max over ranks of each repetition first).
    clocks = ClockSampler(local)
    clocks.start()
    rep_t = []
    for _ in range(args.repeats):
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            replay(args.steps, rem)
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        rep_t.append(max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev))
    clocks.timed = clocks.count()
    t_top = time.perf_counter()
    while clocks.ok and clocks.count() < 10 and time.perf_counter() - t_top < 1.0:
        with torch.cuda.stream(stream):     # same steps, untimed: the clocks under load
            replay(args.steps, rem)
        torch.cuda.synchronize()
    clocks.stop()
    t_max = float(np.median(rep_t))
    t_local = t_max
    total_bytes = sum_over_ranks(sb * args.steps, world, dev)
    value = total_bytes / t_max / 1e9
    ms_step = 1e3 * t_max / args.steps
    repeat_info = {"repeats": args.repeats, "statistic": "median",
                   "ms_per_step_min": 1e3 * min(rep_t) / args.steps,
                   "ms_per_step_max": 1e3 * max(rep_t) / args.steps}
    if grouped:
        per_step = len(groups)      # one launch per group (both N in one launch)
    else:
        per_step = len(gvs)
    launches = per_step * args.steps

    if args.step_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "GB/s",
                              "ms_per_step": ms_step, "steps": args.steps,
                              "note": "--step-only: the headline region alone (profiling)"}),
                  flush=True)
        return 0

    # the per-call protocol as well: a graph of >= 200 back-to-back launches
    # (whole steps, rotating copies), median of 10 timed replays
    n200 = max(block, -(-200 // per_step))
    g200 = capture(n200, 0)
    with torch.cuda.stream(stream):
        g200.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(10)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            a.record(stream)
            g200.replay()
            b.record(stream)
    torch.cuda.synchronize()
    us200 = float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e3 / n200
    graph200 = {"launches_per_graph": n200 * per_step, "steps_per_graph": n200,
                "us_per_step": round(us200, 3), "gbs": round(sb / us200 / 1e3, 1),
                "statistic": "median of 10 replays"}
    del g200

    # the other launch mode, same steps, for comparison
    g_other = capture(block, 0, not grouped)
    rem_o = {}
    if args.steps % block:
        rem_o[args.steps % block] = capture(args.steps % block, 0, not grouped)
    with torch.cuda.stream(stream):
        g_other.replay()              # warm-up: one block of steps
    torch.cuda.synchronize()
    o0 = torch.cuda.Event(enable_timing=True)
    o1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        o0.record(stream)
        replay(args.steps, rem_o, g_other)
        o1.record(stream)
    torch.cuda.synchronize()
    t_other = o0.elapsed_time(o1) / 1e3
    other = {"mode": "per-matrix calls" if grouped else "grouped calls",
             "ms_per_step": 1e3 * t_other / args.steps,
             "gbs": sb * args.steps / t_other / 1e9}
    del g_other, rem_o

    # correctness of what was timed: all copies produce identical y
    y_check = [y.clone() for y in ys]
    with torch.cuda.stream(stream):
        launch_step(1)
    torch.cuda.synchronize()
    same = all(torch.equal(a, b) for a, b in zip(y_check, ys))

    # per-matrix times (same rotation, one matrix at a time, graphs)
    per = []
    for i, gv in enumerate(gvs):
        gi = torch.cuda.CUDAGraph()
        reps = 4 * copies
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gi, stream=stream):
                for k in range(reps):
                    sets[k % copies][i].run(xs[i], ys[i], sptr)
        gi.replay()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a0.record(stream)
            for _ in range(5):
                gi.replay()
            a1.record(stream)
        torch.cuda.synchronize()
        us = a0.elapsed_time(a1) * 1e3 / (5 * reps)
        per.append({"name": gv.name, "shape": [gv.rows, gv.cols],
                    "n_keep": gv.n_keep, "group": gv.group,
                    "bytes": gv.bytes(m), "us": round(us, 3),
                    "gbs": round(gv.bytes(m) / us / 1e3, 1)})
        del gi

    # dense fp16 GEMV baseline (cuBLAS via torch), same shapes and rotation
    dense_us = None
    try:
        dense_bytes = sum(2 * g.rows * g.cols for g in gvs)
        dcopies = max(2, math.ceil(4 * l2 / dense_bytes) + 1)
        dws = [[torch.randn(g.rows, g.cols, device=dev, dtype=torch.float16)
                for g in gvs] for _ in range(dcopies)]
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for k in range(2):
                for w, x in zip(dws[k % dcopies], xs):
                    torch.nn.functional.linear(x, w)
            with torch.cuda.graph(gd, stream=stream):
                for k in range(dcopies * 2):
                    for w, x, y in zip(dws[k % dcopies], xs, ys):
                        torch.matmul(x, w.t(), out=y)
        gd.replay()
        torch.cuda.synchronize()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            d0.record(stream)
            for _ in range(5):
                gd.replay()
            d1.record(stream)
        torch.cuda.synchronize()
        dense_us = d0.elapsed_time(d1) * 1e3 / (5 * dcopies * 2)
        del dws, gd
    except Exception as exc:  # pragma: no cover - reported, not fatal
        dense_us = f"failed: {exc}"

    # small-M verification batches (beam / prefix-tree nodes): the config-4
    # layer set, all 2:4 g = 128, x with M rows; bytes and kept-weight flops
    batch = None
    batch_mixed = None
    rowg = None
    sweep = None
    if not args.no_batch and not args.no_sweep:
        sweep = run_gemv_sweep(args, swo, dev, stream, l2, read_peak()[0])
    if not args.no_batch:
        batch = run_batch_sweep(args, swo, dev, stream, l2)
        # the same verification batches on the mixed (N, g) layer set
        batch_mixed = run_batch_sweep(args, swo, dev, stream, l2, gvs, (4, 16, 64))
        rowg = run_rowgroup_case(args, swo, dev, stream, l2)

    # End to end, x from and y to page-locked host memory every step, two
    # ways through the public API: (a) one copy of the step's activations
    # in, the grouped device-buffer calls (sgemv_run_group over q/k/v and
    # gate/up, sgemv_run for o and down: kernels back to back, as timed
    # above), one copy of the outputs out -- the headline e2e; (b) the host-buffer calls
    # sgemv_run_group_host / sgemv_run_host, whose copies sit between the
    # kernels.  Each step is captured once per packed copy into a CUDA
    # graph; a step is one replay on the benchmark's stream, a sync of that
    # stream and a host read of y.
    hgroups = layer_groups(gvs)
    # the step's activations in one page-locked buffer and its outputs in
    # one, so that each direction is one copy (views for the calls; every x
    # view starts on a 128-byte boundary: cols is a multiple of 64)
    xsz = {grp[0]: m * gvs[grp[0]].cols for grp in hgroups}
    ysz = [m * gv.rows for gv in gvs]
    xh_all = torch.empty(sum(xsz.values()), dtype=torch.float16).pin_memory()
    xd_all = torch.empty_like(xh_all, device=dev)
    yh_all = torch.empty(sum(ysz), dtype=torch.float16).pin_memory()
    yd_all = torch.empty_like(yh_all, device=dev)
    xh, xd, off = {}, {}, 0
    for i, n in xsz.items():
        xh[i] = xh_all[off:off + n].view(m, gvs[i].cols)
        xh[i].copy_(torch.from_numpy(gvs[i].x(m)))
        xd[i] = xd_all[off:off + n].view(m, gvs[i].cols)
        off += n
    yh, yd, off = [], [], 0
    for gv, n in zip(gvs, ysz):
        yh.append(yh_all[off:off + n].view(m, gv.rows))
        yd.append(yd_all[off:off + n].view(m, gv.rows))
        off += n
    h2d_bytes = xh_all.numel() * xh_all.element_size()
    d2h_bytes = yh_all.numel() * yh_all.element_size()
    lib = swo.load()
    e2e_steps = max(3, min(args.steps, 200))

    def e2e_issue_dev(st):
        xd_all.copy_(xh_all, non_blocking=True)
        for grp in hgroups:
            if len(grp) == 1:
                st[grp[0]].run(xd[grp[0]], yd[grp[0]], sptr)
            else:
                swo.run_group([st[i] for i in grp], xd[grp[0]], [yd[i] for i in grp], sptr)
        yh_all.copy_(yd_all, non_blocking=True)

    def e2e_issue_host(st):
        for grp in hgroups:
            if len(grp) == 1:
                i = grp[0]
                rc = lib.sgemv_run_host(st[i].handle, xh[i].data_ptr(), yh[i].data_ptr(), m, sptr)
                if rc:
                    raise RuntimeError(lib.sgemv_last_error().decode())
            else:
                swo.run_group_host([st[i] for i in grp], xh[grp[0]], [yh[i] for i in grp], sptr)

    def e2e_time(issue, graphed):
        """GB/s of e2e_steps steps, each ending in a stream sync and a read of y."""
        graphs = []
        if graphed:
            for c in range(copies):
                gh = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    with torch.cuda.graph(gh, stream=stream):
                        issue(sets[c])
                graphs.append(gh)

        yv = yh_all.numpy()   # the host read of y, without tensor indexing

        def one(k):
            if graphed:
                graphs[k % copies].replay()
            else:
                issue(sets[k % copies])
            stream.synchronize()
            return float(yv[0])

        # replay() launches on the current stream: make it the one each step
        # is synchronised on, for the whole timed loop
        with torch.cuda.stream(stream):
            for k in range(3):
                one(k)
            barrier(world)
            t0 = time.perf_counter()
            for k in range(e2e_steps):
                one(k)
            t = time.perf_counter() - t0
        t = max_over_ranks(t, world, dev)
        return sum_over_ranks(sb * e2e_steps, world, dev) / t / 1e9

    e2e_eager = e2e_time(e2e_issue_dev, False)
    e2e = e2e_eager
    e2e_mode = "one x copy in, sgemv_run_group / sgemv_run on device buffers, one y copy out; eager"
    e2e_host = None
    try:
        e2e = e2e_time(e2e_issue_dev, True)
        e2e_mode = ("one copy of the step's x in (pinned host -> device), run_group(q,k,v), "
                    "run(o), run_group(gate,up), run(down) on device buffers, one copy of its y "
                    "out; captured in a CUDA graph per packed copy, one replay + stream sync + "
                    "y read per step")
        e2e_host = e2e_time(e2e_issue_host, True)
    except Exception as exc:  # pragma: no cover - reported, the eager figure stands
        e2e_mode += f" (graph capture failed: {exc})"

    # CPU oracle on the host cores (rank 0 only), ~10 s bounded sample
    cpu = None
    cpu_all = None
    oracle_pack = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        from oracle import Packed
        packed = []
        for gv, c in zip(gvs, canon):
            packed.append((gv, Packed(gv.rows, gv.cols, gv.n_keep, gv.group, *c),
                           gv.x(m)))
        b, t, rows = oracle_time(packed, args.cpu_seconds)
        cpu = {"value": b / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{rows} rows of the layer set in blocks of 1/64 of a "
                         f"matrix, {t:.1f} s single-threaded"}
        threads = os.cpu_count() or 1
        b, t, rows = oracle_time_threads(packed, args.cpu_seconds, threads)
        cpu_all = {"value": b / t / 1e9, "unit": "GB/s", "cores": threads,
                   "kind": "oracle, row blocks on a thread pool",
                   "sample": f"{rows} rows of the layer set in blocks of 1/64 of a "
                             f"matrix, {t:.1f} s wall on {threads} threads"}
        # the oracle's pack (prune, quantise, encode) of one matrix, timed apart
        gk = next(g for g in gvs if g.name == "k")
        Wk = gk.weight()
        t0 = time.perf_counter()
        oracle.pack(Wk, gk.n_keep, gk.group)
        oracle_pack = {"matrix": f"k {gk.rows}x{gk.cols} {gk.n_keep}:4 g{gk.group}",
                       "seconds": round(time.perf_counter() - t0, 3), "cores": 1}
        del Wk

    peak, peak_src = read_peak()
    traffic = read_traffic("sgemv_layerset_m1")
    achieved = sb / (t_local / args.steps) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "us_per_call": 1e3 * ms_step / len(gvs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": WORKLOAD, "m": m, "seed": args.seed,
            "matrices": [[g.name, g.rows, g.cols, f"{g.n_keep}:4", g.group]
                         for g in gvs],
            "bytes_per_step": sb,
            "l2": f"inputs larger than L2: rotation over {copies} packed copies "
                  f"({copies * wbytes / 1e6:.0f} MB > 4 x L2 {l2 / 1e6:.0f} MB)",
            "parallelism": f"replicas x{world}",
            "timing": "CUDA graphs on one stream, CUDA events",
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic["bytes_per_step"] if traffic else None},
        "e2e": {"value": e2e, "unit": "GB/s",
                "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes,
                "api": e2e_mode, "eager_value": e2e_eager,
                "host_api_value": e2e_host,
                "host_api": "sgemv_run_group_host(q,k,v), sgemv_run_host(o), "
                            "sgemv_run_group_host(gate,up), sgemv_run_host(down) (copies between "
                            "the kernels), graph per packed copy"},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "oracle_pack": oracle_pack,
        "clocks": clocks.summary(),
        "gpu_launches": launches,
        "timing": repeat_info,
        "graph_200_launches": graph200,
        "per_matrix": per,
        "dense_fp16_us_per_step": dense_us,
        "speedup_vs_dense_fp16": (dense_us / (1e3 * ms_step)
                                  if isinstance(dense_us, float) else None),
        "pack_seconds": round(t_pack, 3),
        "batch_m": batch,
        "batch_m_layerset": batch_mixed,
        "row_groups": rowg,
        "gemv_sweep": sweep,
        "copies_identical_y": same,
        "launch_mode": ("grouped calls: run_group(q,k,v), run(o), run_group(gate,up), "
                        "run(down)" if grouped else "per-matrix calls"),
        "other_launch_mode": other,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def layer_groups(gvs):
    """Index groups of matrices that share x in a decoder layer (q/k/v,
    gate/up; the others alone), by name, for the matrices present."""
    pos = {g.name: i for i, g in enumerate(gvs)}
    groups, seen = [], set()
    for grp in GROUPS:
        idx = [pos[n] for n in grp if n in pos]
        if idx:
            groups.append(idx)
            seen.update(idx)
    groups += [[i] for i in range(len(gvs)) if i not in seen]
    return groups


def run_batch_sweep(args, swo, dev, stream, l2, gvs=None, ms=None):
    """us and GB/s per M for the config-4 set (seven 2:4 g128 matrices), or
    for the given matrices and M values: the grouped step (run_group over
    q/k/v and gate/up, as the decode step) and, beside it, one call per
    matrix (us_per_step_calls)."""
    import torch
    gvs = synth.config4(args.seed) if gvs is None else gvs
    ms = synth.CONFIG4_M if ms is None else ms
    mmax = max(ms)
    hs0 = []
    for gv in gvs:
        W = gv.weight()
        h = swo.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, max_m=mmax,
                           device=dev.index)
        h.pack(W)
        del W
        hs0.append(h)
    canon = [h.export_canonical() for h in hs0]
    wbytes = sum(g.packed_bytes() for g in gvs)
    copies = max(2, math.ceil(4 * l2 / wbytes) + 1)
    sets = [hs0]
    for _ in range(copies - 1):
        cp = []
        for gv, c in zip(gvs, canon):
            h = swo.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, max_m=mmax,
                               device=dev.index)
            h.import_canonical(*c)
            cp.append(h)
        sets.append(cp)
    sptr = stream.cuda_stream
    groups = layer_groups(gvs)
    out = {}
    for m in ms:
        xs = [None] * len(gvs)
        for grp in groups:
            x0 = torch.from_numpy(gvs[grp[0]].x(m)).to(dev)
            for i in grp:
                xs[i] = x0
        ys = [torch.empty((m, gv.rows), dtype=torch.float16, device=dev) for gv in gvs]

        def step(st, grouped):
            if grouped:
                for grp in groups:
                    if len(grp) == 1:
                        st[grp[0]].run(xs[grp[0]], ys[grp[0]], sptr)
                    else:
                        swo.run_group([st[i] for i in grp], xs[grp[0]],
                                      [ys[i] for i in grp], sptr)
            else:
                for h, x, y in zip(st, xs, ys):
                    h.run(x, y, sptr)

        res = {}
        for grouped in (True, False):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                step(sets[0], grouped)
                with torch.cuda.graph(g, stream=stream):
                    for k in range(copies):
                        step(sets[k], grouped)
            g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            reps = 5
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            res[grouped] = e0.elapsed_time(e1) * 1e3 / (reps * copies)
            del g
        us = res[True]
        b = step_bytes(gvs, m)
        fl = sum(gv.flops(m) for gv in gvs)
        out[str(m)] = {"us_per_step": round(us, 3), "gbs": round(b / us / 1e3, 1),
                       "tflops": round(fl / us / 1e6, 2),
                       "launches_per_step": len(groups),
                       "us_per_step_calls": round(res[False], 3)}
    for st in sets:
        for h in st:
            h.close()
    return out


def run_gemv_sweep(args, swo, dev, stream, l2, peak):
    """M = 1, one GEMV at a time, for the single-layer workloads (4096x4096
    2:4 g128; 4096x4096 with outliers at 1:4 g256 and 2:4 g64) and the large
    layers (8192x8192, 28672x8192, 8192x28672, g128): us per call, GB/s,
    fraction of the HBM peak, and cuBLAS dense binary16 on the same shape."""
    import torch
    sptr = stream.cuda_stream
    out = []
    for gv in synth.config1(args.seed) + synth.config2(args.seed) + synth.config5(args.seed):
        W = gv.weight()
        h0 = swo.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, device=dev.index)
        h0.pack(W)
        del W
        canon = h0.export_canonical()
        pb = gv.packed_bytes()
        copies = max(2, math.ceil(4 * l2 / pb) + 1)
        hs = [h0]
        for _ in range(copies - 1):
            h = swo.SparseGemv(gv.rows, gv.cols, gv.n_keep, gv.group, device=dev.index)
            h.import_canonical(*canon)
            hs.append(h)
        del canon
        x = torch.from_numpy(gv.x(1)).to(dev)
        y = torch.empty((1, gv.rows), dtype=torch.float16, device=dev)

        def timed(fn, reps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                fn(0)
                with torch.cuda.graph(g, stream=stream):
                    for k in range(reps):
                        fn(k)
            g.replay()
            torch.cuda.synchronize()
            # median of 10 timed replays of the whole rotation
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(10)]
            with torch.cuda.stream(stream):
                for a, b in ev:
                    a.record(stream)
                    g.replay()
                    b.record(stream)
            torch.cuda.synchronize()
            return float(np.median([a.elapsed_time(b) for a, b in ev])) * 1e3 / reps

        us = timed(lambda k: hs[k % copies].run(x, y, sptr), 4 * copies)
        for h in hs:
            h.close()
        del hs
        dense = None
        try:
            db = 2 * gv.rows * gv.cols
            dc = max(2, math.ceil(4 * l2 / db) + 1)
            dws = [torch.randn(gv.rows, gv.cols, device=dev, dtype=torch.float16)
                   for _ in range(dc)]
            dense = timed(lambda k: torch.matmul(x, dws[k % dc].t(), out=y), 2 * dc)
            del dws
        except Exception:  # pragma: no cover - reported as missing
            dense = None
        b = gv.bytes(1)
        out.append({"name": gv.name, "shape": [gv.rows, gv.cols],
                    "n_keep": gv.n_keep, "group": gv.group, "bytes": b,
                    "us": round(us, 3), "gbs": round(b / us / 1e3, 1),
                    "frac_of_peak": round(b / us / 1e3 / peak, 3),
                    "frac_of_nominal_8tbs": round(b / us / 1e3 / NOMINAL_HBM_GBS, 3),
                    "dense_fp16_us": round(dense, 3) if dense else None,
                    "speedup_vs_dense_fp16": round(dense / us, 2) if dense else None})
        torch.cuda.empty_cache()
    return out


def run_rowgroup_case(args, swo, dev, stream, l2):
    """M = 1 on an 11008 x 4096 2:4 layer with a seeded group size per row
    (64 / 128 / 256), next to the same layer with one group size."""
    import torch
    rows, cols = 11008, 4096
    W = synth.weight_normal(args.seed + 101, rows, cols, 0.02)
    rg = synth.row_groups(args.seed, rows)
    x = torch.from_numpy(synth.activations(args.seed + 102, 1, cols)).to(dev)
    y = torch.empty((1, rows), dtype=torch.float16, device=dev)
    sptr = stream.cuda_stream
    out = {"shape": [rows, cols], "n_keep": 2,
           "rows_per_group": {str(g): int((rg == g).sum()) for g in (64, 128, 256)}}
    for name, kw in (("per_row", {"row_group": rg}), ("g64", {}), ("g128", {})):
        group = None if kw else int(name[1:])
        h0 = swo.SparseGemv(rows, cols, 2, group, device=dev.index, **kw)
        h0.pack(W)
        canon = h0.export_canonical()
        pb = h0.packed_bytes()
        copies = max(2, math.ceil(4 * l2 / pb) + 1)
        hs = [h0]
        for _ in range(copies - 1):
            h = swo.SparseGemv(rows, cols, 2, group, device=dev.index, **kw)
            h.import_canonical(*canon)
            hs.append(h)
        g = torch.cuda.CUDAGraph()
        reps = 4 * copies
        with torch.cuda.stream(stream):
            hs[0].run(x, y, sptr)
            with torch.cuda.graph(g, stream=stream):
                for k in range(reps):
                    hs[k % copies].run(x, y, sptr)
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(5):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (5 * reps)
        b = pb + 2 * cols + 2 * rows
        out[name] = {"us": round(us, 3), "bytes": b, "gbs": round(b / us / 1e3, 1)}
        del g
        for h in hs:
            h.close()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--repeats", type=int, default=10,
                    help="timed repetitions of the K-step region (median reported)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ungrouped", action="store_true",
                    help="time one call per matrix instead of the grouped calls")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the one-GEMV-at-a-time sweep over the single and large layers")
    ap.add_argument("--no-batch", action="store_true",
                    help="skip the small-M (config 4) sweep")
    ap.add_argument("--step-only", action="store_true",
                    help="time the headline step region alone and stop (profiling)")
    ap.add_argument("--batch-only", type=int, default=0, metavar="M",
                    help="run only the verification-batch layer set at M rows (profiling)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="write the DRAM record of one step from an ncu CSV log and stop")
    ap.add_argument("--traffic-out", default=os.path.join(ROOT, "profiles", "traffic.json"))
    ap.add_argument("--traffic-command", default="",
                    help="the ncu command that produced the CSV (kept in the record)")
    args = ap.parse_args(argv)
    if args.record_traffic:
        return record_traffic(args.record_traffic, args.traffic_out, args.traffic_command)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.repeats < 1:
        ap.error("--repeats must be at least 1")
    rank, world, local = dist_init()
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        if args.batch_only:
            return run_batch_only(args, local)
        return run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
