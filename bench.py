"""Benchmark: fused decode + GEMV over entropy-coded weights on one GB300.

Step = one pass of the hot path over one batch: fused decode + GEMV (batch 1)
of every matrix of one Mistral-7B-shaped layer of 4-bit codes (q, k, v, o,
gate, up, down; one Huffman table per matrix), through the C ABI.  Metric:
coded bytes read per step / step time (GB/s), reported against the measured
HBM copy bandwidth; also the dense-equivalent effective bandwidth (2 bytes
per weight / time, "Software-Defined Bandwidth Expansion" eq. (1)), and the
same step on the fixed-width twin and on an uncompressed BF16 GEMV (cuBLAS).

The layer's coded bytes (~80 MB) fit in L2, so every step reads a different
device copy of the layer, rotating over enough copies to exceed 4x L2.

`--impl reference` times the CPU oracle instead (decode + dequant + fp64 GEMV
on a bounded sample of the same workload, on every host core at once, with
the one-core figure beside it).
Prints one JSON line (rank 0).
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused decode+GEMV coded GB/s vs HBM peak; dense-equiv eff. bandwidth, batch 1"
WORKLOAD = "mistral7b_layer_q4_batch1"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--only", default="", help="comma list of matrix names (profiling)")
    p.add_argument("--copies", type=int, default=0, help="layer copies to rotate (0 = auto)")
    p.add_argument("--twin", action="store_true",
                   help="time the fixed-width twin in the main loop instead (profiling)")
    p.add_argument("--workload", default="mistral",
                   choices=["mistral", "tiny", "phi3", "llama_mlp", "stack", "stack_bf16mlp"],
                   help="mistral: the headline line; the others print one line each with "
                        "per-batch rows (coded, twin and dense BF16 times)")
    p.add_argument("--batches", default="",
                   help="comma list of batch sizes for --workload sweeps (default: the workload's)")
    p.add_argument("--keep", type=float, default=1.0,
                   help="fraction of each matrix's 64-row strips to compute through a tile-skip "
                        "launch list (lw_decode_gemm_strips; seeded random strips); 1 = all")
    p.add_argument("--ungrouped", action="store_true",
                   help="one launch per matrix instead of one per group of independent matrices")
    p.add_argument("--no-extras", action="store_true",
                   help="skip twin / bf16 / cpu baseline / e2e legs (profiling)")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self._stop = threading.Event()
        self._t = None

    def _one(self):
        try:
            out = subprocess.run(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=5).stdout.strip()
            if out:
                self.rows.append([c.strip() for c in out.split(",")])
        except Exception:  # noqa: BLE001
            pass

    def _run(self):
        while not self._stop.is_set():
            self._one()
            self._stop.wait(0.05)

    def start(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def stop(self):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)
        if not self.rows:
            self._one()
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


# ----------------------------------------------------------------------------
# the CPU oracle on a bounded sample (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------

def layer_matrices():
    from decode_gemv_gb300 import inputs
    out = []
    for i, s in enumerate(inputs.workload_specs(inputs.MISTRAL_LAYER)):
        out.append((s, inputs.make_matrix(inputs.MISTRAL_LAYER, s, 0, i)))
    return out


def oracle_sample_setup(mats, target_weights: int):
    """Sample = the first row strips of every matrix of the layer, about
    `target_weights` weights in all, coded by the oracle's own encoder."""
    import oracle
    per = max(1, target_weights // len(mats))
    jobs = []
    for s, m in mats:
        rows = max(64, min(s.rows, (per // s.cols) // 64 * 64))
        sub = dict(codes=m["codes"][:rows], scales=m["scales"][:rows], mins=m["mins"][:rows],
                   x=m["x"])
        ob = oracle.encode(oracle.Q4, sub["codes"])
        coded = (ob["words"].nbytes + ob["tile_off"].nbytes + ob["lane_bits"].nbytes + 1024
                 + sub["scales"].nbytes + sub["mins"].nbytes + sub["x"].nbytes)
        jobs.append((rows, s.cols, ob, sub, coded))
    return jobs


def oracle_sample_step(jobs):
    """One oracle pass: decode every lane, dequantise, fp64 GEMV."""
    import oracle
    out = []
    for rows, cols, ob, sub, _ in jobs:
        packed = oracle.decode(oracle.Q4, rows, cols, ob["code_len"], ob["words"], ob["tile_off"])
        w = oracle.dequant_q4(oracle.unpack_q4(packed), sub["scales"], sub["mins"])
        out.append(oracle.gemm(w, sub["x"]))
    return out


def oracle_rate(mats):
    """Weights per second of one oracle pass on a small sample (calibration)."""
    jobs = oracle_sample_setup(mats, 1_000_000)
    w = sum(j[0] * j[1] for j in jobs)
    t0 = time.perf_counter()
    oracle_sample_step(jobs)
    return w / (time.perf_counter() - t0)


def host_cores() -> int:
    """Host cores this process may run on (its affinity mask where the OS
    keeps one)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_shares(mats, target_weights: int, n: int):
    """The sample of oracle_sample_setup (the first row strips of every
    matrix, about `target_weights` weights) cut into 64-row strips and dealt
    to at most n workers, largest strip first to the least loaded worker.
    Per worker: a list of sub-matrices (codes, scales, mins of its strips of
    one matrix, and that matrix's x)."""
    per = max(1, target_weights // len(mats))
    units = []
    for j, (s, _) in enumerate(mats):
        rows = max(64, min(s.rows, (per // s.cols) // 64 * 64))
        units += [(64 * s.cols, j, r0) for r0 in range(0, rows, 64)]
    units.sort(key=lambda u: (-u[0], u[1], u[2]))
    load = [0] * n
    picked = [dict() for _ in range(n)]
    for w, j, r0 in units:
        i = load.index(min(load))
        load[i] += w
        picked[i].setdefault(j, []).append(r0)
    shares = []
    for by in picked:
        share = []
        for j in sorted(by):
            m = mats[j][1]
            idx = np.concatenate([np.arange(r0, r0 + 64) for r0 in sorted(by[j])])
            share.append(dict(codes=np.ascontiguousarray(m["codes"][idx]),
                              scales=np.ascontiguousarray(m["scales"][idx]),
                              mins=np.ascontiguousarray(m["mins"][idx]), x=m["x"]))
        if share:
            shares.append(share)
    return shares


def _oracle_share_worker(path, barrier, steps, warmup, out):
    """One host core's part of the all-cores oracle run: load its strips
    from `path`, encode them with the oracle (untimed), then warm-up + timed
    passes, each started together with the other workers at a barrier.
    Sends back its coded bytes, weights and the seconds of every timed
    pass."""
    import oracle
    jobs = []
    with np.load(path) as f:
        share = [{k: f[f"{i}_{k}"] for k in ("codes", "scales", "mins", "x")}
                 for i in range(int(f["n"]))]
    for sub in share:
        rows, cols = sub["codes"].shape
        ob = oracle.encode(oracle.Q4, sub["codes"])
        coded = (ob["words"].nbytes + ob["tile_off"].nbytes + ob["lane_bits"].nbytes + 1024
                 + sub["scales"].nbytes + sub["mins"].nbytes + sub["x"].nbytes)
        jobs.append((rows, cols, ob, sub, coded))
    times = []
    for i in range(warmup + steps):
        barrier.wait(timeout=300)
        t0 = time.perf_counter()
        oracle_sample_step(jobs)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    out.put((sum(j[4] for j in jobs), sum(j[0] * j[1] for j in jobs), times))


def oracle_all_cores(mats, target_weights: int, steps: int, warmup: int, cores: int = 0):
    """The oracle on every host core at once: the sample split into strips
    over one spawned process per core (spawned, never forked: the parent
    may hold a CUDA context; the strips go through files, so a worker that
    fails early cannot stall the parent).  A pass's time is the slowest
    worker's; the result is coded bytes of the whole sample / mean pass
    time."""
    import multiprocessing as mp
    import queue
    import tempfile

    from oracle import oracle as oracle_impl
    oracle_impl._load()                  # build (if stale) and load it once, before the workers do
    shares = oracle_shares(mats, target_weights, cores or host_cores())
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory() as tmp:
        paths = []
        for w, share in enumerate(shares):
            path = os.path.join(tmp, f"share{w}.npz")
            np.savez(path, n=len(share), **{f"{i}_{k}": sub[k] for i, sub in enumerate(share)
                                            for k in ("codes", "scales", "mins", "x")})
            paths.append(path)
        barrier, out = ctx.Barrier(len(shares)), ctx.Queue()
        procs = [ctx.Process(target=_oracle_share_worker, args=(path, barrier, steps, warmup, out),
                             daemon=True) for path in paths]
        res, deadline = [], time.monotonic() + 1200
        try:
            for p in procs:
                p.start()
            while len(res) < len(procs):
                try:
                    res.append(out.get(timeout=1.0))
                except queue.Empty:
                    if any(p.exitcode not in (None, 0) for p in procs):
                        raise RuntimeError("an oracle worker failed")
                    if time.monotonic() > deadline:
                        raise RuntimeError("oracle workers did not finish in time")
        finally:
            for p in procs:
                if p.pid is not None:
                    p.join(timeout=10)
                    if p.is_alive():
                        p.terminate()
                        p.join(timeout=10)
    coded = sum(r[0] for r in res)
    weights = sum(r[1] for r in res)
    per_pass = [max(r[2][i] for r in res) for i in range(steps)]
    dt = sum(per_pass) / max(1, steps)
    return {"value": coded / dt / 1e9, "unit": "GB/s", "cores": len(shares), "weights": weights,
            "coded_bytes": coded, "seconds_per_pass": dt}


def cpu_baseline_entry(pairs, seconds: float = 5.0):
    """The oracle on the host for a JSON line: every host core at once (the
    value) and one core alone, each on the first row strips of every matrix
    of the layer -- one core's sample is about `seconds` of its work (at
    most 30 M weights), all cores together take one such sample per core
    (at most the whole layer)."""
    rate = oracle_rate(pairs)
    target = int(min(30_000_000, rate * seconds))
    jobs = oracle_sample_setup(pairs, target)
    coded = sum(j[4] for j in jobs)
    wts = sum(j[0] * j[1] for j in jobs)
    reps = 2
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_sample_step(jobs)
    dt = (time.perf_counter() - t0) / reps
    single = {"value": coded / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
              "sample": f"first row strips of every matrix of the layer: {wts} weights, "
                        f"{coded} coded bytes; decode + dequant + fp64 GEMV, {reps} timed passes"}
    layer = sum(sp.rows * sp.cols for sp, _ in pairs)
    try:
        allc = oracle_all_cores(pairs, int(min(layer, wts * host_cores())), reps, 1)
    except Exception as e:  # noqa: BLE001 -- the one-core figure still stands
        return dict(single, note=f"all-cores run unavailable: {e}")
    return {"value": allc["value"], "unit": "GB/s", "cores": allc["cores"], "kind": "oracle",
            "sample": f"first row strips of every matrix of the layer: {allc['weights']} weights, "
                      f"{allc['coded_bytes']} coded bytes, cut into 64-row strips over "
                      f"{allc['cores']} spawned processes (one per host core, started together "
                      f"each pass); decode + dequant + fp64 GEMV, {reps} timed passes",
            "single_core": single}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    mats = layer_matrices()
    # one core: size each step so that its warm-up + timed steps take about
    # 45 s of CPU time; all cores: one such sample per core, each step
    # started together on every core (about 45 s of wall time)
    rate = oracle_rate(mats)
    per_step = 45.0 / max(1, args.steps + args.warmup)
    target = int(min(30_000_000, max(64 * 4096 * 7, rate * per_step)))
    jobs = oracle_sample_setup(mats, target)
    coded = sum(j[4] for j in jobs)
    weights = sum(j[0] * j[1] for j in jobs)
    for _ in range(max(0, args.warmup)):
        oracle_sample_step(jobs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(jobs)
    dt1 = (time.perf_counter() - t0) / max(1, args.steps)
    single = {"value": coded / dt1 / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
              "ms_per_step": dt1 * 1e3,
              "sample": f"first row strips of all 7 matrices of the layer: {weights} weights, "
                        f"{coded} coded bytes per step; decode + dequant + fp64 GEMV"}
    layer = sum(sp.rows * sp.cols for sp, _ in mats)
    try:
        allc = oracle_all_cores(mats, int(min(layer, weights * host_cores())), max(1, args.steps),
                                max(0, args.warmup))
        sample = (f"first row strips of all 7 matrices of the layer: {allc['weights']} weights, "
                  f"{allc['coded_bytes']} coded bytes per step, cut into 64-row strips over "
                  f"{allc['cores']} spawned processes (one per host core, started together each "
                  f"step); decode + dequant + fp64 GEMV")
    except Exception as e:  # noqa: BLE001 -- the one-core run still stands as the value
        allc = {"value": single["value"], "seconds_per_pass": dt1, "cores": 1,
                "weights": weights}
        sample = single["sample"] + f" (all-cores run unavailable: {e})"
    gbs, dt = allc["value"], allc["seconds_per_pass"]
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_weights": allc["weights"]},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": allc["cores"], "kind": "oracle",
                             "sample": sample, "single_core": single},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

# ----------------------------------------------------------------------------
# replicas (one process per GPU, no data-path collective)
# ----------------------------------------------------------------------------

def max_over_ranks(ms, device=None):
    """The slowest rank's time (every rank gets it); `ms` unchanged with one
    process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank, world, t_max_ms):
    """Every rank's bytes over the slowest rank's time (weak scaling)."""
    return bytes_per_rank * world / (t_max_ms * 1e-3) / 1e9


# matrices of a decoder layer that read the same input and do not depend on
# one another: each set is one grouped launch (q, k, v read the normalised
# hidden state; gate and up read the normalised attention output)
LAYER_GROUPS = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]


def layer_groups(names, ungrouped=False):
    """Index lists, in layer order, of the launches of one step."""
    if ungrouped:
        return [[i] for i in range(len(names))]
    out = []
    for g in LAYER_GROUPS:
        idx = [names.index(n) for n in g if n in names]
        if idx:
            out.append(idx)
    assert sorted(i for g in out for i in g) == list(range(len(names)))
    return out


def listed_bytes(hb, strips, cols):
    """Bundle bytes the product reads for the listed strips: their tiles'
    coded words, tile offsets, lane bits and mids, scales/mins, plus the
    table."""
    tk = cols // 256
    toff = hb.view("tile_off", np.uint32).astype(np.int64)
    per_tile = 64 + 64 + (len(hb.sections.get("qparams", b"")) // max(1, len(toff) - 1))
    words = sum(int(toff[(s + 1) * tk] - toff[s * tk]) * 128 for s in strips)
    # tile offsets read: each listed tile's start and end entries
    offsets = set()
    for s in strips:
        offsets.update(range(int(s) * tk, (int(s) + 1) * tk + 1))
    return words + len(strips) * tk * per_tile + 4 * len(offsets) + 1024


def build_layer(names):
    from decode_gemv_gb300 import lw
    mats = []
    for s, m in layer_matrices():
        if names and s.name not in names:
            continue
        hb = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"])
        tw = lw.lw_encode_bundle(lw.LW_FMT_Q4_PAIR, m["codes"], m["scales"], m["mins"], twin=True)
        mats.append(dict(spec=s, m=m, hb=hb, tw=tw))
    return mats


def per_call_ms(torch, stream, calls_by_copy, reps=8):
    """Average duration of each call, one graph per call, events between
    replays, rotating over the given copies."""
    graphs = []
    for calls in calls_by_copy:
        row = []
        for f in calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                f()
            row.append(g)
        graphs.append(row)
    n = len(calls_by_copy[0])
    out = np.zeros(n)
    for r in range(reps + 2):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        for j, g in enumerate(graphs[r % len(graphs)]):
            ev[j].record(stream)
            g.replay()
        ev[n].record(stream)
        torch.cuda.synchronize()
        if r >= 2:
            out += [ev[j].elapsed_time(ev[j + 1]) for j in range(n)]
    return out / reps


KERNEL_SOURCES = ("lw_qlut.cuh", "lw_lutdec.cuh", "lw_lut.h", "lw_qkern.cuh", "lw_dev.cuh", "lw_qlut.cu")


def kernel_source_digest():
    """sha256 over the sources of the table-driven product kernel and its launcher."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_gemv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def kernel_counters():
    """The committed ncu counters of the table-driven kernel (per-launch DRAM
    bytes of this step, instruction and issue counts of the gate matrix) --
    only while the kernel's sources are the ones that were profiled, else
    None."""
    try:
        with open(os.path.join(ROOT, "profiles", "q_lut_kernel_counters.json")) as f:
            d = json.load(f)
    except Exception:  # noqa: BLE001
        return None
    return d if d.get("source_sha256") == kernel_source_digest() else None


def measured_traffic(names, launches):
    """DRAM bytes (read + write) per launch of the fused kernel on this step
    (mean over the step's launches, and each launch's), from the committed
    capture, or (None, None) when the kernel or the launches differ."""
    d = kernel_counters()
    if d is None or names or d.get("launches") != launches:
        return None, None
    per = d["traffic_per_launch_bytes"]
    return sum(per.values()) / len(per), per


def issue_roofline(achieved_gbs, bytes_per_pair, sm_mhz, sms):
    """The instruction-issue roof of the decode: warp-instructions per pair
    symbol (per lane) from the committed capture of the gate matrix, the
    coded GB/s that count allows at one instruction per cycle on each of the
    SM's four schedulers, and the fraction of it achieved."""
    d = kernel_counters()
    if d is None or not sm_mhz:
        return None
    ipp = d["gate"]["warp_inst_per_pair"]
    ceiling = sms * 4 * sm_mhz * 1e6 * 32 / ipp * bytes_per_pair / 1e9
    return {"warp_inst_per_pair": ipp, "issue_active_pct": d["gate"]["issue_active_pct"],
            "ceiling_gbs": ceiling, "achieved_gbs": achieved_gbs, "frac": achieved_gbs / ceiling,
            "hbm_frac_at_ceiling": None,
            "basis": "ceiling = SMs x 4 schedulers x SM clock (median sampled in the timed region) "
                     "x 32 lanes / warp-instructions per pair x coded bytes per pair of the step; "
                     "counts from the committed one-kernel capture of the gate matrix"}


def dequant_bf16(m):
    import torch
    s = np.repeat(m["scales"].view(np.float16).astype(np.float32), 256, axis=1)
    mi = np.repeat(m["mins"].view(np.float16).astype(np.float32), 256, axis=1)
    w = torch.from_numpy(s * m["codes"].astype(np.float32) + mi)
    return w.to(torch.bfloat16)


def step_graph(torch, lw, calls, stream):
    """The library calls of a step captured once as a CUDA graph of the
    library's own (lw.StepGraph: nothing but the calls is replayed), after
    one eager run."""
    for f in calls:
        f()
    torch.cuda.synchronize()
    g = lw.StepGraph(stream)
    with g.capture():
        for f in calls:
            f()
    torch.cuda.synchronize()
    return g


def layer_graph(torch, calls):
    """One CUDA graph holding the given calls in order (after one eager run)."""
    for f in calls:
        f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in calls:
            f()
    torch.cuda.synchronize()
    return g


def time_steps(torch, stream, step_fn, steps, warmup, copies):
    for i in range(warmup):
        step_fn(i % copies)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step_fn(i % copies)
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / steps


def percentiles(samples):
    """p10, median and p90 of per-step times (linear interpolation between
    order statistics, numpy's default)."""
    a = np.asarray(samples, dtype=np.float64)
    p10, med, p90 = np.percentile(a, [10, 50, 90])
    return {"p10": float(p10), "median": float(med), "p90": float(p90), "steps": int(a.size)}


def per_step_ms(torch, stream, step_fn, steps, copies):
    """Each step timed alone: an event pair around every step on `stream`
    (after the timed region; it does not enter `value`)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        step_fn(i % copies)
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_ours(args):
    import torch
    from decode_gemv_gb300 import lw

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lw.load()
    names = [n for n in args.only.split(",") if n]
    mats = build_layer(names)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layer_coded = sum(x["tw" if args.twin else "hb"].stats.coded_bytes for x in mats)
    copies = args.copies or max(2, math.ceil(4 * l2 / layer_coded))
    # device copies of the layer (distinct addresses), activations, outputs
    key = "tw" if args.twin else "hb"
    dbs = [[lw.DeviceBundle.upload(x[key], dev) for x in mats] for _ in range(copies)]
    xs = [torch.from_numpy(x["m"]["x"][0]).to(dev) for x in mats]
    ys = [torch.empty(x["spec"].rows, dtype=torch.float32, device=dev) for x in mats]
    keep = args.keep < 1.0 and not args.twin
    groups = layer_groups([x["spec"].name for x in mats], args.ungrouped or args.twin or keep)
    wsb = max([lw.lw_workspace_bytes(d, 1) for d in dbs[0]] +
              [lw.lw_workspace_bytes_group([dbs[0][j] for j in g]) for g in groups if len(g) > 1])
    ws = torch.zeros(wsb // 4 + 64, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    x_bytes = sum(t.numel() * 4 for t in xs)
    coded_step = layer_coded + x_bytes          # every byte the step must read
    strip_lists = None
    if keep:
        # tile-skip launch lists: a seeded random `keep` fraction of each
        # matrix's strips; the step then reads only their tiles
        rk = np.random.default_rng(1234)
        strip_lists, coded_keep = [], 0
        for x in mats:
            ns = x["spec"].rows // 64
            lst = np.sort(rk.choice(ns, max(1, int(round(args.keep * ns))), replace=False))
            strip_lists.append(torch.from_numpy(lst.astype(np.int32)).to(dev))
            coded_keep += listed_bytes(x["hb"], lst, x["spec"].cols)
        coded_step = coded_keep + x_bytes
    weights = sum(x["spec"].rows * x["spec"].cols for x in mats)

    def call(c, j):
        if args.twin:
            lw.lw_twin_gemv(dbs[c][j], xs[j], ys[j], ws, st)
        elif strip_lists is not None:
            lw.lw_decode_gemm_strips(dbs[c][j], strip_lists[j], xs[j], 1, ys[j], ws, st)
        else:
            lw.lw_decode_gemv(dbs[c][j], xs[j], ys[j], ws, st)

    def launch(c, g):
        if len(g) == 1:
            call(c, g[0])
        else:
            lw.lw_decode_gemv_group([dbs[c][j] for j in g], [xs[j] for j in g],
                                    [ys[j] for j in g], ws, st)

    for c in range(copies):
        for g in groups:
            launch(c, g)
    torch.cuda.synchronize()
    # one CUDA graph per layer copy (its fused launches, one per group of
    # independent matrices), captured by the library's step-graph calls: the
    # host only replays graphs, so the timed region measures the device (the
    # pages' runtime also captures each pass in CUDA graphs)
    cap = torch.cuda.Stream(dev)
    graphs = []
    for c in range(copies):
        sg = lw.StepGraph(cap)
        with sg.capture():
            for g in groups:
                launch(c, g)
        graphs.append(sg)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    n_mat = len(mats)

    if world > 1:
        torch.distributed.barrier()
    for i in range(args.warmup):
        graphs[i % copies].launch(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        graphs[i % copies].launch(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    ms = ev0.elapsed_time(ev1) / args.steps
    t_max = max_over_ranks(ms, dev)
    status = int(st.item())
    # spread of the step time: every step timed alone, over as many steps
    # as the timed region (at most 2000)
    spread = percentiles(per_step_ms(torch, stream, lambda c: graphs[c].launch(stream),
                                     max(1, min(args.steps, 2000)), copies))
    # diagnostic: each matrix's call alone (one graph per call, events around)
    per_mat = per_call_ms(torch, stream, [[(lambda c=c, j=j: call(c, j)) for j in range(n_mat)]
                                          for c in range(min(copies, 4))])

    value = whole_job_gbs(coded_step, world, t_max)
    peak, peak_kind = peaks()
    launches_per_step = len(groups)      # one fused kernel per group
    # dominant kernel (the fused decode+GEMV launch, 97 % of the step's GPU
    # time): algorithmic bytes per launch over its average duration in the
    # timed region, i.e. the step time shared over its launches
    mean_call_ms = t_max / launches_per_step
    mean_call_bytes = coded_step / launches_per_step
    achieved = mean_call_bytes / (mean_call_ms * 1e-3) / 1e9
    traffic_mean, traffic_per = measured_traffic(
        names, [[mats[j]["spec"].name for j in g] for g in groups])
    issue = issue_roofline(achieved, coded_step / (weights / 2), clocks.get("sm_mhz"),
                           torch.cuda.get_device_properties(dev).multi_processor_count)
    if issue is not None:
        issue["hbm_frac_at_ceiling"] = issue["ceiling_gbs"] / peak
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD + (f"_keep{args.keep:g}" if keep else ""),
                       "matrices": [x["spec"].name for x in mats],
                       "weights": weights, "coded_bytes_per_step": coded_step,
                       "bits_per_weight": 8 * layer_coded / weights, "batch": 1,
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": f"rotate {copies} device copies of the layer "
                             f"({copies * layer_coded / 1e6:.0f} MB > 4x L2 {l2 / 1e6:.0f} MB)"},
            "b_eff_gbs": 2.0 * weights * world / (t_max * 1e-3) / 1e9,
            "hbm_frac_of_nominal_8tbs": value / world / 8000.0,
            "step_ms_spread": dict(spread, note="each step timed alone with its own event pair, "
                                                "after the timed region (not part of value)"),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic_mean,
                         "traffic_per_launch": traffic_per,
                         "peak_kind": peak_kind,
                         "kernel": "q_lut_kernel (table-driven fused decode + GEMV + ordered split-K "
                                   "reduction), "
                                   + ("one launch per matrix" if len(groups) == n_mat else
                                      "one launch per group " + "/".join(
                                          "+".join(mats[j]["spec"].name for j in g) for g in groups)),
                         "issue": issue,
                         "per_matrix_ms": {x["spec"].name: float(v) for x, v in zip(mats, per_mat)},
                         "per_matrix_note": "each call alone, one graph per call (diagnostic)",
                         "note": "bound in practice by instruction issue, not HBM: the decode's "
                                 "warp-instructions per pair symbol (roofline.issue) cap the coded "
                                 "bytes per second far below the HBM peak"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks, "device_status": status}
    if keep:
        line["config"]["tile_skip"] = (f"each matrix computes a seeded random {args.keep:g} of its "
                                       f"64-row strips through lw_decode_gemm_strips; value counts "
                                       f"the listed tiles' bytes only")
    if rank == 0 and not args.no_extras and not keep:
        extras(args, torch, lw, dev, mats, copies, xs, ys, ws, st, stream, line, coded_step,
               weights, t_max, groups, dbs)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def extras(args, torch, lw, dev, mats, copies, xs, ys, ws, st, stream, line, coded_step,
           weights, t_ours, groups, dbs):
    """Comparators and the end-to-end leg (outside the timed region above)."""
    steps = max(10, min(args.steps, 400))

    # fixed-width twin, same rotation, one graph per matrix call
    ntw = max(2, math.ceil(copies * 0.75))
    twins = [[lw.DeviceBundle.upload(x["tw"], dev) for x in mats] for _ in range(ntw)]
    tcalls = [[(lambda d=d, x=x, y=y: lw.lw_twin_gemv(d, x, y, ws, st))
               for d, x, y in zip(twins[c], xs, ys)] for c in range(ntw)]
    # the twin step makes the same launches as the coded step (one per group)
    tsteps = [[(lambda c=c, g=g: lw.lw_twin_gemv_group([twins[c][j] for j in g], [xs[j] for j in g],
                                                       [ys[j] for j in g], ws, st))
               if len(g) > 1 else tcalls[c][g[0]] for g in groups] for c in range(ntw)]
    cap = torch.cuda.Stream(dev)
    tg = [step_graph(torch, lw, calls, cap) for calls in tsteps]

    def tstep(c):
        tg[c].launch(stream)
    t_twin = time_steps(torch, stream, tstep, steps, 5, ntw)
    tw_ms = per_call_ms(torch, stream, tcalls[: min(ntw, 4)])
    del tg, twins, tcalls, tsteps
    # uncompressed BF16 GEMV (cuBLAS) on the dequantised weights, graphed
    wb = [dequant_bf16(x["m"]).to(dev) for x in mats]
    xb = [x.to(torch.bfloat16) for x in xs]
    yb = [torch.empty(w.shape[0], dtype=torch.bfloat16, device=dev) for w in wb]
    bg = layer_graph(torch, [(lambda w=w, x=x, y=y: torch.mv(w, x, out=y)) for w, x, y in zip(wb, xb, yb)])

    def bstep(c):
        bg.replay()
    t_bf16 = time_steps(torch, stream, bstep, steps, 5, 1)
    del bg, wb
    twin_bytes = sum(x["tw"].stats.coded_bytes for x in mats) + sum(x.numel() * 4 for x in xs)
    line["twin"] = {"ms_per_step": t_twin, "speedup_of_coded": t_twin / t_ours,
                    "gbs": twin_bytes / (t_twin * 1e-3) / 1e9,
                    "per_matrix_ms": {x["spec"].name: float(v) for x, v in zip(mats, tw_ms)}}
    line["bf16_dense"] = {"ms_per_step": t_bf16, "speedup_of_coded": t_bf16 / t_ours,
                          "kind": "torch.mv on bf16 weights (cuBLAS), one CUDA graph per layer"}
    # end to end through the public API: every step copies the layer's
    # activations in from pinned host memory (one packed copy) and its
    # results out (one packed copy), on the device copies the timed loop
    # rotates over
    xo = np.cumsum([0] + [x.numel() for x in xs])
    yo = np.cumsum([0] + [y.numel() for y in ys])
    hx = torch.cat([x.cpu() for x in xs]).pin_memory()
    hy = torch.empty(int(yo[-1]), dtype=torch.float32).pin_memory()
    dx = torch.empty(int(xo[-1]), dtype=torch.float32, device=dev)
    dy = torch.empty(int(yo[-1]), dtype=torch.float32, device=dev)
    xv = [dx[int(a):int(b)] for a, b in zip(xo[:-1], xo[1:])]
    yv = [dy[int(a):int(b)] for a, b in zip(yo[:-1], yo[1:])]

    # the step's library calls with their arguments marshalled once (one C
    # call per launch, as a C caller would make them)
    prepared = [[lw.PreparedGemv([dbs[c][j] for j in g], [xv[j] for j in g], [yv[j] for j in g],
                                 ws, st, twin=args.twin) for g in groups] for c in range(copies)]

    def e2e_step(c):
        dx.copy_(hx, non_blocking=True)
        for call in prepared[c]:
            call()          # the current stream (the capture stream under a graph capture)
        hy.copy_(dy, non_blocking=True)
    for i in range(3):
        e2e_step(i % copies)
        torch.cuda.synchronize()
    e_steps = max(10, min(args.steps, 400))
    t0 = time.perf_counter()
    for i in range(e_steps):
        e2e_step(i % copies)
        torch.cuda.synchronize()
        _ = float(hy[0])
    dt = (time.perf_counter() - t0) / e_steps
    # the same step captured once in a CUDA graph per layer copy (copies in,
    # library calls, copies out), replayed and synchronised every step: the
    # form the pages' runtime takes (each pass captured in a CUDA graph)
    egraphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_step(c)
        egraphs.append(g)
    for i in range(3):
        egraphs[i % copies].replay()
        torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e_steps):
        egraphs[i % copies].replay()
        torch.cuda.synchronize()
        _ = float(hy[0])
    dtg = (time.perf_counter() - t0) / e_steps
    del egraphs
    line["e2e_graph"] = {"value": coded_step / dtg / 1e9, "unit": "GB/s", "ms_per_step": dtg * 1e3,
                         "note": "the e2e step captured once per layer copy in a CUDA graph; wall "
                                 "clock per replay incl. the H2D/D2H copies and a stream sync"}
    line["e2e"] = {"value": coded_step / dt / 1e9, "unit": "GB/s",
                   "h2d_bytes_per_step": int(hx.numel() * 4),
                   "d2h_bytes_per_step": int(hy.numel() * 4),
                   "ms_per_step": dt * 1e3,
                   "note": f"wall clock per step: one packed H2D of the activations, the step's "
                           f"{len(groups)} library calls, one packed D2H of the results, a stream "
                           f"sync; rotating over the {copies} device copies of the layer"}
    # the oracle on the host, bounded samples (a few seconds of work per
    # core); one process per GPU shares the host's cores, so only at N = 1
    if int(os.environ.get("WORLD_SIZE", "1")) == 1:
        line["cpu_baseline"] = cpu_baseline_entry([(x["spec"], x["m"]) for x in mats])


# ----------------------------------------------------------------------------
# Per-workload sweeps (--workload): every synthetic workload, each batch
# ----------------------------------------------------------------------------

SWEEPS = {
    # name: (workload id, label, batches, layers)
    "tiny": (0, "tiny_q4_256x1024", [1], 1),
    "phi3": (2, "phi3mini_layer_q6", [1, 2, 4, 8], 1),
    "llama_mlp": (3, "llama31_8b_mlp_bf16exp", [1, 4, 16, 64], 1),
    "stack": (4, "stack32_mistral_q4", [1, 2, 4, 8, 16, 32], 32),
    "stack_bf16mlp": (4, "stack32_q4attn_bf16exp_mlp", [1, 2, 4, 8, 16, 32], 32),
}


def _fmt_of(spec_fmt):
    from decode_gemv_gb300 import lw
    return {1: lw.LW_FMT_Q4_PAIR, 2: lw.LW_FMT_Q6, 3: lw.LW_FMT_BF16_EXP}[spec_fmt]


def _encode_job(job):
    """Spawned worker: draw one matrix and encode it (coded and twin);
    returns picklable bundle descriptions."""
    workload, layer, index, spec = job
    sys.path.insert(0, ROOT)
    from decode_gemv_gb300 import inputs, lw
    m = inputs.make_matrix(workload, spec, layer, index)
    fmt = _fmt_of(spec.fmt)
    payload = m["bits"] if spec.fmt == inputs.BF16 else m["codes"]
    out = {}
    for twin in (False, True):
        hb = lw.lw_encode_bundle(fmt, payload, m.get("scales"), m.get("mins"), twin=twin)
        out[twin] = (fmt, twin, spec.rows, spec.cols, hb.sections, hb.stats.max_tile_rows,
                     hb.stats.min_len, hb.stats.max_len, hb.stats.coded_bytes)
    return spec, out


def sweep_specs(name):
    from decode_gemv_gb300 import inputs
    wid, _, _, layers = SWEEPS[name]
    jobs = []
    for layer in range(layers):
        specs = inputs.workload_specs(wid)
        if name == "stack_bf16mlp":
            # attention projections 4-bit as the stack; MLP as the BF16 workload
            mlp = inputs.workload_specs(inputs.LLAMA_MLP_BF16)
            jobs += [(wid, layer, i, s) for i, s in enumerate(specs[:4])]
            jobs += [(inputs.LLAMA_MLP_BF16, layer, i, s) for i, s in enumerate(mlp)]
        else:
            jobs += [(wid, layer, i, s) for i, s in enumerate(specs)]
    return jobs


def sweep_groups(mats, lw):
    """Launch groups of a sweep at batch 1: the 4-/6-bit matrices of one layer
    that share an input (LAYER_GROUPS) and a format; every other matrix alone.
    Index lists in the order of each group's first matrix."""
    groups, seen = [], set()
    for i, m in enumerate(mats):
        if i in seen:
            continue
        g = [i]
        if m["fmt"] != lw.LW_FMT_BF16_EXP:
            for names in LAYER_GROUPS:
                if m["spec"].name in names:
                    g = [j for j, o in enumerate(mats) if o["layer"] == m["layer"]
                         and o["spec"].name in names and o["fmt"] == m["fmt"]][:8]
        seen.update(g)
        groups.append(g)
    return groups


def run_sweep(args):
    """Time the coded path, the fixed-width twin and a dense BF16 GEMV/GEMM
    (cuBLAS, same shapes) for every batch of one workload."""
    import multiprocessing as mp
    wid, label, batches, layers = SWEEPS[args.workload]
    if args.batches:
        batches = [int(b) for b in args.batches.split(",") if b]
    jobs = sweep_specs(args.workload)
    names = [n for n in args.only.split(",") if n]
    if names:
        jobs = [j for j in jobs if j[3].name in names]
    t_prep = time.perf_counter()
    if len(jobs) > 8:
        with mp.get_context("spawn").Pool(min(16, os.cpu_count() or 4)) as pool:
            built = pool.map(_encode_job, jobs, chunksize=1)
    else:
        built = [_encode_job(j) for j in jobs]
    t_prep = time.perf_counter() - t_prep
    import torch
    from decode_gemv_gb300 import lw
    lw.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    coded_total = sum(o[False][8] for _, o in built)
    copies = max(1, math.ceil(4 * l2 / coded_total)) if coded_total < 4 * l2 else 1
    mats = []
    for job, (spec, o) in zip(jobs, built):
        mats.append(dict(spec=spec, fmt=o[False][0], layer=job[1],
                         db=[lw.DeviceBundle(*o[False][:8], device=dev, coded_bytes=o[False][8])
                             for _ in range(copies)],
                         tw=[lw.DeviceBundle(*o[True][:8], device=dev, coded_bytes=o[True][8])
                             for _ in range(copies)]))
    del built
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    # dense comparator: random bf16 weights of the same shapes (cuBLAS time
    # depends on the shape only), as many copies as the coded layer
    dense = [[torch.randn(m["spec"].rows, m["spec"].cols, device=dev, generator=gen,
                          dtype=torch.bfloat16) for m in mats] for _ in range(copies)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = peaks()
    weights = sum(m["spec"].rows * m["spec"].cols for m in mats)
    # tiny layers: each CUDA graph holds `group` consecutive steps (each on
    # the next copy), so the host's replay cost does not dominate
    group = 64 if copies >= 128 else 1
    ngraph = max(1, copies // group)

    last = {}

    def timed(calls_of_copy, steps=None):
        graphs = [layer_graph(torch, [f for c in range(g * group, (g + 1) * group)
                                      for f in calls_of_copy(c)]) for g in range(ngraph)]
        if steps is None:
            one = time_steps(torch, stream, lambda i: graphs[i].replay(), 3, 2, ngraph) / group
            steps = max(10, min(args.steps, int(2000.0 / max(one, 1e-3))))
        reps = max(3, steps // group)
        t = time_steps(torch, stream, lambda i: graphs[i].replay(), reps, 5, ngraph) / group
        # spread: every replay timed alone afterwards (per step of the graph)
        last["spread"] = percentiles([v / group for v in per_step_ms(
            torch, stream, lambda i: graphs[i].replay(), reps, ngraph)])
        del graphs
        return t, steps

    groups = sweep_groups(mats, lw)
    # decode buffers of the full-decode comparator (all-BF16 workloads only;
    # one per matrix, rewritten every step)
    wdec = None
    if all(m["fmt"] == lw.LW_FMT_BF16_EXP for m in mats):
        wdec = [torch.empty(m["spec"].rows, m["spec"].cols, device=dev, dtype=torch.bfloat16)
                for m in mats]
    rows_out = []
    clk = ClockSampler(0)
    clk.start()
    for B in batches:
        xs, ys = [], []
        for m in mats:
            dt = torch.bfloat16 if m["fmt"] == lw.LW_FMT_BF16_EXP else torch.float32
            xs.append(torch.randn(B, m["spec"].cols, device=dev, generator=gen).to(dt))
            ys.append(torch.empty(B, m["spec"].rows, device=dev, dtype=torch.float32))
        wsb = max(lw.lw_workspace_bytes(m["db"][0], B) for m in mats)
        # one launch per group of a layer's independent 4-/6-bit matrices while
        # the batch stays on the CUDA cores (up to 5 rows: from 6 the large
        # matrices take the tensor cores, one launch each)
        grouped = B <= 5 and any(len(g) > 1 for g in groups)
        if grouped:
            wsb = max([wsb] + [lw.lw_workspace_bytes_group([mats[j]["db"][0] for j in g])
                               for g in groups if len(g) > 1])
        ws = torch.zeros(wsb // 4 + 64, dtype=torch.float32, device=dev)
        x_bytes = sum(x.numel() * x.element_size() for x in xs)
        coded_step = sum(m["db"][0].coded_bytes for m in mats) + x_bytes
        twin_step = sum(m["tw"][0].coded_bytes for m in mats) + x_bytes
        def step_calls(c, key, one, group):
            # batch 1: one launch per group of a layer's independent
            # 4-/6-bit matrices; otherwise one call per matrix
            if not grouped:
                return [(lambda d=m[key][c], x=x, y=y: one(d, x, B, y, ws, st))
                        for m, x, y in zip(mats, xs, ys)]
            return [(lambda g=g: group([mats[j][key][c] for j in g], [xs[j] for j in g],
                                       [ys[j] for j in g], ws, st)) if len(g) > 1 else
                    (lambda d=mats[g[0]][key][c], x=xs[g[0]], y=ys[g[0]]: one(d, x, B, y, ws, st))
                    for g in groups]
        gc = lambda d, x, y, w, s_: lw.lw_decode_gemm_group(d, x, B, y, w, s_)
        gt = lambda d, x, y, w, s_: lw.lw_twin_gemm_group(d, x, B, y, w, s_)
        t_coded, steps = timed(lambda c: step_calls(c, "db", lw.lw_decode_gemm, gc))
        spread_coded = last["spread"]
        t_twin, _ = timed(lambda c: step_calls(c, "tw", lw.lw_twin_gemm, gt), steps)
        xb = [x.to(torch.bfloat16) for x in xs]
        yb = [torch.empty(B, m["spec"].rows, device=dev, dtype=torch.bfloat16) for m in mats]
        t_bf16, _ = timed(lambda c: [(lambda w=w, x=x, y=y: torch.matmul(x, w.t(), out=y))
                                     for w, x, y in zip(dense[c], xb, yb)], steps)
        # the pages' "full decode" pipeline (BF16 exponent bundles): restore
        # the weights into HBM with lw_decode, then one cuBLAS product
        t_full = None
        if wdec is not None:
            t_full, _ = timed(lambda c: [f for m, x, y, w in zip(mats, xb, yb, wdec) for f in (
                (lambda d=m["db"][c], w=w: lw.lw_decode(d, w, st)),
                (lambda w=w, x=x, y=y: torch.matmul(x, w.t(), out=y)))], steps)
        gbs = coded_step / (t_coded * 1e-3) / 1e9
        rows_out.append({"batch": B, "calls": len(groups) if grouped else len(mats),
                         "ms_per_step": t_coded, "coded_gbs": gbs,
                         "frac_of_hbm": gbs / peak, "b_eff_gbs": 2.0 * weights / (t_coded * 1e-3) / 1e9,
                         "twin_ms": t_twin, "twin_gbs": twin_step / (t_twin * 1e-3) / 1e9,
                         "speedup_vs_twin": t_twin / t_coded, "ms_spread": spread_coded,
                         "bf16_ms": t_bf16, "speedup_vs_bf16": t_bf16 / t_coded,
                         "coded_bytes_per_step": coded_step, "steps": steps})
        if t_full is not None:
            rows_out[-1]["decode_cublas_ms"] = t_full
            rows_out[-1]["speedup_vs_decode_cublas"] = t_full / t_coded
    clocks = clk.stop()
    line = {"metric": METRIC, "workload": label, "value": rows_out[0]["coded_gbs"], "unit": "GB/s",
            "n_gpus": 1, "higher_is_better": True, "dtype": "f32" if mats[0]["fmt"] != lw.LW_FMT_BF16_EXP else "bf16",
            "data": "synthetic", "peak_gbs": peak, "peak_kind": peak_kind,
            "config": {"workload": label, "layers": layers, "matrices": len(mats), "weights": weights,
                       "calls": "library calls per step (rows[].calls): batch 1..5 one per group of a "
                                "layer's independent 4-/6-bit matrices (q+k+v, gate+up; coded and twin "
                                "alike), else one per matrix; a call on the CUDA cores is one kernel launch "
                                "per pass, a tensor-core call the product and, when its K range is split "
                                "over CTAs, the split-K sum",
                       "l2": (f"rotate {copies} device copies ({group} steps per CUDA graph)"
                              if copies > 1 else "working set > 4x L2"),
                       "dense_comparator": "torch.matmul on random bf16 weights of the same shapes (cuBLAS)",
                       "host_prep_s": round(t_prep, 1)},
            "rows": rows_out, "clocks": clocks, "device_status": int(st.item())}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "mistral":
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
