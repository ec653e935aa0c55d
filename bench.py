"""Benchmark of the exact ternary weight apply on one GB300 (or N replicas).

Headline: the batch-1 ternary GEMV of the ffn_up workload (N=6912, K=2560,
128-weight groups, int8 activations, int64 outputs), in microseconds per GEMV
and effective weight GB/s (packed masks + group scales / time).

One step is a decode sweep of GEMVS_PER_STEP batch-1 GEMV calls through the C
ABI, each on the next of R distinct device copies of the packed weights; the
copies together exceed 4x the L2 cache, so no call finds its weights in L2.
The step's calls are captured once into a CUDA graph and the graph is replayed
per step, so host launch overhead does not enter the device-timed value (the
e2e figure makes the same calls eagerly from the host). Inputs are resident in
HBM before the timed region. Timing: W warm-up steps, then exactly K steps
between CUDA events on the launching stream, bracketed by a barrier and a
device synchronise; with several ranks the slowest rank's time is used and
every rank runs its own replica (weak scaling, no collective on the data path).

Also reported on the same line:
  e2e          the same metric with the step's activations copied in from
               pinned host memory, every call made eagerly through the public
               API, and all outputs read back, every step;
  e2e_graph    the same, with the calls replayed from CUDA graphs captured
               once before the timed region (the copies stay inside it);
  wall_us      µs per call: back to back from the graph (with and without the
               constant-weights flag) and one call at a time (200 reps:
               median, p10, p90);
  roofline     the GEMV kernel's algorithmic bytes per launch / its average
               launch time, against the measured HBM copy bandwidth;
  cpu_baseline the CPU oracle timed on a bounded sample on the host cores;
  rows         the other hot-path calls (LNS8 both routes, lm_head both paths,
               batched M=64, Q1_0, the floor shift and int64 activations at
               batch 1), each timed alone
               (skip with --no-rows);
  clocks       nvidia-smi SM clocks and throttle reasons during the timed region.

--impl reference times the CPU oracle on the same workload and metric.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "batch-1 ternary GEMV µs and effective weight GB/s as % of GB300 HBM peak"
WORKLOAD = ("ffn_up batch-1 ternary GEMV, N=6912 K=2560, 128-weight groups, int8 x from "
            "N(0,40^2), int32 group scales, int64 y")
GEMVS_PER_STEP = 1024
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 7900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row figures")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--quick", action="store_true", help="= --no-rows --no-cpu (for profiler runs)")
    ap.add_argument("--sweep", default=None, choices=["lns8_routes", "gemv_m", "lns8_purelns", "ffn_up_graph"],
                    help="run a measurement sweep instead of the bench and exit (ffn_up_graph: only the "
                         "headline's CUDA graph of back-to-back calls, replayed warmup + steps times, as a "
                         "profiler target)")
    ap.add_argument("--gemvs-per-step", type=int, default=GEMVS_PER_STEP,
                    help="batch-1 GEMV calls in one step's graph (the headline uses 1024)")
    ap.add_argument("--row", default=None,
                    help="time only these rows (comma list of tiny, lns8, lm_head, batched, q1, x64) and exit")
    a = ap.parse_args()
    if a.quick:
        a.no_rows = a.no_cpu = True
    a.warmup = max(a.warmup, 3)
    return a


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}",
                   "--format=csv,noheader,nounits", "-lms", "20"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    stamp = parts[0]
                    whole, _, frac = stamp.partition(".")
                    ts = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts + (float("0." + frac) if frac else 0.0), parts[1:]))
                except Exception:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [p for t, p in rows if self.t0 - 0.05 <= t <= self.t1 + 0.05]
        use = inside if inside else [p for _, p in rows]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [v for v in (num(p[0]) for p in use) if v is not None]
        smax = [v for v in (num(p[1]) for p in use) if v is not None]
        reasons = set()
        for p in use:
            for n, v in zip(self.REASONS, p[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use),
                "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------

def weight_bytes_ffn(w):
    N, K = w["t"].shape
    return N * K // 4 + N * (K // 128) * 4


def oracle_gemv_rate(w, seconds: float, reps_max: int = 10_000, threads: int = 1):
    """Effective weight GB/s of the CPU oracle on the ffn_up GEMV: whole GEMVs
    for about `seconds`, each split into `threads` contiguous row slices that
    run the unchanged oracle call concurrently (ctypes releases the GIL during
    the call). Returns (GB/s, GEMVs, seconds)."""
    import concurrent.futures as cf
    import oracle
    wbytes = weight_bytes_ffn(w)
    N = w["t"].shape[0]
    cuts = [N * i // threads for i in range(threads + 1)]
    slices = [(w["t"][a:b], w["d"][a:b]) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    x = w["x"]
    n = 0
    with cf.ThreadPoolExecutor(max_workers=len(slices)) as ex:
        t0 = time.perf_counter()
        while n < reps_max:
            if len(slices) == 1:
                oracle.gemv_i8(slices[0][0], slices[0][1], x)
            else:
                list(ex.map(lambda td: oracle.gemv_i8(td[0], td[1], x), slices))
            n += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    return n * wbytes / dt / 1e9, n, dt


def host_description():
    """The host's architecture (uname -m), CPU model and logical core count."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"uname_m": platform.machine(), "cpu_model": model or "unknown", "logical_cores": os.cpu_count()}


def cpu_baseline_record(w, seconds_single: float, seconds_parallel: float):
    """cpu_baseline: the oracle row-parallel over every host core (the value), with
    the single-threaded figure and the host description beside it."""
    cores = os.cpu_count() or 1
    g1, n1, s1 = oracle_gemv_rate(w, seconds_single, threads=1)
    gp, n_p, sp = oracle_gemv_rate(w, seconds_parallel, threads=cores)
    return {"value": round(gp, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_p} full ffn_up GEMVs in {sp:.1f} s, each as {cores} row slices of the plain C "
                      "oracle on concurrent threads",
            "single_thread": {"value": round(g1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} full ffn_up GEMVs in {s1:.1f} s"},
            "host": host_description()}


def run_reference(args):
    """--impl reference: the CPU oracle, timed on the same workload and metric."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import concurrent.futures as cf
    import oracle
    w = W.ffn_up()
    wbytes = weight_bytes_ffn(w)
    cores = os.cpu_count() or 1
    N = w["t"].shape[0]
    cuts = [N * i // cores for i in range(cores + 1)]
    slices = [(w["t"][a:b], w["d"][a:b]) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]

    def gemv():   # one whole GEMV: the unchanged oracle on row slices, concurrently
        list(ex.map(lambda td: oracle.gemv_i8(td[0], td[1], w["x"]), slices))

    with cf.ThreadPoolExecutor(max_workers=len(slices)) as ex:
        for _ in range(args.warmup):
            gemv()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            gemv()
        dt = time.perf_counter() - t0
    gbs = args.steps * wbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemvs_per_step": 1,
                   "us_per_gemv": round(dt / args.steps * 1e6, 1)},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": len(slices), "kind": "oracle",
                         "sample": f"{args.steps} full ffn_up GEMVs (one per step), each as {len(slices)} row "
                                   "slices of the plain C oracle on concurrent threads",
                         "host": host_description()},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def kernel_source_hash(name):
    with open(os.path.join(ROOT, "bit_decode_gemv_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_file, workload):
    """dram bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_sha256_16") != kernel_source_hash(kernel_file):
        return None
    return e.get("dram_bytes_per_launch")


def capture_graph(torch, fn, count):
    """CUDA graph of `count` calls fn(i, stream_handle), captured on a side stream."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(min(count, 4)):
            fn(i, side.cuda_stream)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(count):
            fn(i, h)
    torch.cuda.synchronize()
    return g


def event_time(torch, fn, reps, stream):
    """Seconds for reps calls of fn, between CUDA events on `stream` (a torch.cuda.Stream)."""
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def isolated_call_stats(torch, stream, call, reps=200, spacer_cycles=200_000):
    """Device time of one call at a time, in µs: before each rep the stream runs
    a short spin kernel (about 0.1 ms), behind which the host queues the rep's
    two events and its call, so that the interval between the events holds the
    call alone, with no host submission gap; median, p10 and p90 over the reps.
    call(i) makes rep i's call (rotate the weights there to keep them out of L2)."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    spin = getattr(torch.cuda, "_sleep", None)   # torch's own spin kernel; without it the reps may include host gaps
    torch.cuda.synchronize()
    for i in range(reps):
        if spin is not None:
            spin(spacer_cycles)
        a, b = evs[i]
        a.record(stream)
        call(i)
        b.record(stream)
    torch.cuda.synchronize()
    us = np.array([a.elapsed_time(b) * 1e3 for a, b in evs])
    out = {"median": round(float(np.median(us)), 3), "p10": round(float(np.quantile(us, 0.1)), 3),
           "p90": round(float(np.quantile(us, 0.9)), 3), "reps": reps}
    if spin is None:
        out["note"] = "no spin kernel available: the reps include the host's submission gap"
    return out


def _copies_for(nbytes):
    return max(1, int(math.ceil(4 * L2_BYTES / nbytes)))


def row_lns8(tg, torch, stream, dev):
    """LNS8 eight-phase GEMV, N = K = 4096, weights rotated over copies > 4x L2."""
    hbm, _ = measured_peaks()
    w = W.lns8()
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    R = min(_copies_for(blob.size), 128)
    wd = [dev(blob) for _ in range(R)]
    xa = dev(w["xa"])
    A = torch.empty((L.N, 8), dtype=torch.int64, device="cuda")
    S = torch.empty((L.N,), dtype=torch.float64, device="cuda")
    alg = L.mask_bytes + L.N * L.G + L.K + L.N * 8 * 8 + L.N * 8
    out = {}
    for key, flags in (("lns8", 0), ("lns8_stateset", tg.TG_FLAG_LNS8_STATE_SET),
                       ("lns8_purelns_f4", tg.TG_FLAG_LNS8_PURE_LNS)):
        Lr = tg.tg_layout.from_buffer_copy(L)
        Lr.flags = flags
        Lr.frac = 4 if flags == tg.TG_FLAG_LNS8_PURE_LNS else 0
        g = capture_graph(torch, lambda i, h: tg.tg_gemv_lns8_phase(Lr, wd[i % R], xa, A, S, h), R)
        g.replay()
        t = event_time(torch, lambda i: g.replay(), 4, stream) / (4 * R)
        route = {0: "direct route", tg.TG_FLAG_LNS8_STATE_SET: "state-population route",
                 tg.TG_FLAG_LNS8_PURE_LNS: "pure fractional-LNS route, F = 4 (approximate)"}[flags]
        out[key] = {"workload": "N=4096 K=4096 LNS8 eight-phase, " + route,
                    "us": round(t * 1e6, 3), "alg_bytes": int(alg), "gbs": round(alg / t / 1e9, 1),
                    "frac_hbm": round(alg / t / 1e9 / hbm, 4), "bound": "alu", "copies": R,
                    "us_one_call": isolated_call_stats(
                        torch, stream, lambda i: tg.tg_gemv_lns8_phase(Lr, wd[i % R], xa, A, S, stream.cuda_stream))}
        del g
    # the same direct route with activation codes over the whole range (about a
    # fifth of the lanes near an end, so most (row, group) pairs need the exact
    # clamp correction)
    xf = dev(W.lns8_activations_full_range(0, L.K))
    g = capture_graph(torch, lambda i, h: tg.tg_gemv_lns8_phase(L, wd[i % R], xf, A, S, h), R)
    g.replay()
    t = event_time(torch, lambda i: g.replay(), 4, stream) / (4 * R)
    out["lns8_full_range_codes"] = {"workload": "N=4096 K=4096 LNS8 eight-phase, direct route, activation codes "
                                                "uniform over 1..127 (10% zero)",
                                    "us": round(t * 1e6, 3), "alg_bytes": int(alg), "gbs": round(alg / t / 1e9, 1),
                                    "frac_hbm": round(alg / t / 1e9 / hbm, 4), "bound": "alu", "copies": R}
    del g
    return out


def row_lm_head(tg, torch, stream, dev):
    """lm_head, N=128256, K=2560, k=200: both paths (657 MB of weights, > L2 by itself)."""
    hbm, _ = measured_peaks()
    out = {}
    w = W.lm_head()
    blob, L = tg.tg_pack_weights(tg.TG_PLANES8, w["planes"], w["s"])
    del w["planes"]
    wdl = dev(blob)
    del blob
    xd = dev(w["x"])
    k = w["k"]
    wsb = tg.tg_lmhead_workspace_bytes(L, k)
    ws = torch.empty((wsb,), dtype=torch.uint8, device="cuda")
    logits = torch.empty((L.N,), dtype=torch.int64, device="cuda")
    am = torch.empty((1,), dtype=torch.int32, device="cuda")
    ids = torch.empty((k,), dtype=torch.int32, device="cuda")
    sc = torch.empty((k,), dtype=torch.int64, device="cuda")
    nc = torch.empty((1,), dtype=torch.int32, device="cuda")
    for full in (False, True):
        lg = logits if full else None
        g = capture_graph(torch, lambda i, h: tg.tg_lmhead_argmax_topk(L, wdl, xd, k, lg, am, ids, sc,
                                                                        nc, ws, wsb, h), 10)
        g.replay()
        t = event_time(torch, lambda i: g.replay(), 3, stream) / 30
        if full:
            alg = L.mask_bytes + L.aux_bytes + L.scale_bytes + L.K + L.N * 8
        else:
            alg = L.mask_bytes + L.scale_bytes + L.aux2_bytes + L.K + int(nc.item()) * L.K
        key = "lm_head_full" if full else "lm_head_two_stage"
        out[key] = {"workload": "N=128256 K=2560 8 base-3 planes, k=200", "us": round(t * 1e6, 2),
                    "alg_bytes": int(alg), "gbs": round(alg / t / 1e9, 1),
                    "frac_hbm": round(alg / t / 1e9 / hbm, 4), "bound": "hbm",
                    "candidates": int(nc.item()),
                    "us_one_call": isolated_call_stats(
                        torch, stream, lambda i: tg.tg_lmhead_argmax_topk(L, wdl, xd, k, lg, am, ids, sc, nc, ws,
                                                                          wsb, stream.cuda_stream))}
        del g
    return out


def row_batched(tg, torch, stream, dev):
    """Batched M=64, N=13824, K=5120 ternary GEMM, weights rotated over copies."""
    w = W.batched()
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    R = min(_copies_for(blob.size), 32)
    wd = [dev(blob) for _ in range(R)]
    xd = dev(w["x"])
    y = torch.empty((64, L.N), dtype=torch.int64, device="cuda")
    g = capture_graph(torch, lambda i, h: tg.tg_gemv_i8(L, wd[i % R], xd, 64, y, h), R)
    g.replay()
    t = event_time(torch, lambda i: g.replay(), 2, stream) / (2 * R)
    alg = L.mask_bytes + L.scale_bytes + 64 * L.K + 64 * L.N * 8
    macs = 64 * L.N * L.K
    iso = isolated_call_stats(torch, stream, lambda i: tg.tg_gemv_i8(L, wd[i % R], xd, 64, y, stream.cuda_stream))
    return {"batched_m64": {"workload": "M=64 N=13824 K=5120 ternary GEMM", "us": round(t * 1e6, 2),
                            "alg_bytes": int(alg), "gbs": round(alg / t / 1e9, 1),
                            "tops_int": round(2 * macs / t / 1e12, 2), "copies": R, "us_one_call": iso}}


def _gemv_m1_row(tg, torch, stream, dev, kind, w, frac):
    """Per-call time of one batch-1 GEMV shape, weights rotated over copies, PDL on."""
    hbm, _ = measured_peaks()
    blob, L = tg.tg_pack_weights(kind, w["t"], w["d"])
    L.frac = frac
    L.flags |= tg.TG_FLAG_CONST_WEIGHTS
    R = min(_copies_for(blob.size), 512)
    wd = [dev(blob) for _ in range(R)]
    xd = dev(w["x"])
    y = torch.empty((1, L.N), dtype=torch.int64, device="cuda")
    g = capture_graph(torch, lambda i, h: tg.tg_gemv_i8(L, wd[i % R], xd, 1, y, h), R)
    g.replay()
    t = event_time(torch, lambda i: g.replay(), 4, stream) / (4 * R)
    alg = L.mask_bytes + L.scale_bytes + L.K + L.N * 8
    Lplain = tg.tg_layout.from_buffer_copy(L)
    Lplain.flags &= ~tg.TG_FLAG_CONST_WEIGHTS
    iso = isolated_call_stats(torch, stream, lambda i: tg.tg_gemv_i8(Lplain, wd[i % R], xd, 1, y, stream.cuda_stream))
    return {"us": round(t * 1e6, 3), "alg_bytes": int(alg), "gbs": round(alg / t / 1e9, 1),
            "frac_hbm": round(alg / t / 1e9 / hbm, 4), "bound": "hbm", "copies": R, "us_one_call": iso}


def row_tiny(tg, torch, stream, dev):
    """The tiny GEMV (N=256, K=512, batch 1; 36 KB of weights): launch-latency
    bound, reported in µs per call -- back to back from a CUDA graph with the
    weights flagged constant and without the flag, and one call at a time (200
    reps, each queued behind a short spin kernel: median, p10 and p90)."""
    w = W.tiny()
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    R = 64
    wd = [dev(blob) for _ in range(R)]
    xd = dev(w["x"])
    y = torch.empty((1, L.N), dtype=torch.int64, device="cuda")
    out = {"workload": "N=256 K=512 ternary, batch 1, x uniform [-127, 127] (launch-latency bound)",
           "alg_bytes": int(L.mask_bytes + L.scale_bytes + L.K + L.N * 8), "bound": "launch latency"}
    Lc = tg.tg_layout.from_buffer_copy(L)
    Lc.flags |= tg.TG_FLAG_CONST_WEIGHTS
    for key, lay in (("us_back_to_back_const_weights", Lc), ("us_back_to_back", L)):
        g = capture_graph(torch, lambda i, h: tg.tg_gemv_i8(lay, wd[i % R], xd, 1, y, h), 512)
        g.replay()
        out[key] = round(event_time(torch, lambda i: g.replay(), 8, stream) / (8 * 512) * 1e6, 3)
        del g
    iso = isolated_call_stats(torch, stream, lambda i: tg.tg_gemv_i8(L, wd[i % R], xd, 1, y, stream.cuda_stream))
    out["us_single_call"] = iso["median"]
    out["us_single_call_p10_p90"] = [iso["p10"], iso["p90"]]
    out["single_call_reps"] = iso["reps"]
    out["us"] = out["us_back_to_back_const_weights"]
    return {"tiny": out}


def row_x64(tg, torch, stream, dev):
    """int64 fixed-point activations on the ffn_up shape, batch 1: Q.16 values
    (three digit planes) and full-range values (eight)."""
    hbm, _ = measured_peaks()
    out = {}
    w = W.ffn_up()
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    L.flags |= tg.TG_FLAG_X_INT64
    R = min(_copies_for(blob.size), 512)
    wd = [dev(blob) for _ in range(R)]
    y = torch.empty((1, L.N), dtype=torch.int64, device="cuda")
    for key, x in (("x64_q16_ffn_up", W.x_fixed64(0, (1, L.K), frac_bits=16)),
                   ("x64_full_ffn_up", W.x_int64_full(0, (1, L.K)))):
        xd = dev(x)
        g = capture_graph(torch, lambda i, h: tg.tg_gemv_i8(L, wd[i % R], xd, 1, y, h), R)
        g.replay()
        t = event_time(torch, lambda i: g.replay(), 4, stream) / (4 * R)
        alg = L.mask_bytes + L.scale_bytes + 8 * L.K + L.N * 8
        out[key] = {"workload": "N=6912 K=2560 ternary, batch 1, int64 activations "
                                + ("rint(N(0,1) 2^16)" if "q16" in key else "uniform over int64"),
                    "us": round(t * 1e6, 3), "alg_bytes": int(alg), "gbs": round(alg / t / 1e9, 1),
                    "frac_hbm": round(alg / t / 1e9 / hbm, 4), "copies": R,
                    "us_one_call": isolated_call_stats(
                        torch, stream, lambda i: tg.tg_gemv_i8(L, wd[i % R], xd, 1, y, stream.cuda_stream))}
        del g
    return out


def row_q1(tg, torch, stream, dev):
    """Q1_0 binary weights and the per-group floor shift on the ffn_up shape, batch 1."""
    out = {}
    r = _gemv_m1_row(tg, torch, stream, dev, tg.TG_TERNARY_I8, W.ffn_up(), 0)
    out["ternary_ffn_up"] = {"workload": "N=6912 K=2560 ternary, batch 1 (same timing as below)", **r}
    r = _gemv_m1_row(tg, torch, stream, dev, tg.TG_BINARY_Q1, W.ffn_up_q1(), 0)
    out["q1_ffn_up"] = {"workload": "N=6912 K=2560 Q1_0 binary, batch 1", **r}
    r = _gemv_m1_row(tg, torch, stream, dev, tg.TG_TERNARY_I8, W.ffn_up(), 4)
    out["ternary_ffn_up_frac4"] = {"workload": "N=6912 K=2560 ternary, batch 1, frac=4", **r}
    return out


ROWS = {"tiny": row_tiny, "lns8": row_lns8, "lm_head": row_lm_head, "batched": row_batched, "q1": row_q1,
        "x64": row_x64}


def measure_rows(tg, torch, stream, dev, names=None):
    """Per-call time of the other hot-path entry points, each on its own workload."""
    out = {}
    for name in names or ROWS:
        out.update(ROWS[name](tg, torch, stream, dev))
        torch.cuda.empty_cache()
    return out


def _lns8_route_point(tg, torch, stream, dev, w):
    """Per-call µs of both LNS8 routes on one workload (weights rotated over
    copies, each route from its own CUDA graph); the two routes' A must agree."""
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    R = min(_copies_for(blob.size), 256)
    wd = [dev(blob) for _ in range(R)]
    xa = dev(w["xa"])
    A = [torch.empty((L.N, 8), dtype=torch.int64, device="cuda") for _ in range(2)]
    S = torch.empty((L.N,), dtype=torch.float64, device="cuda")
    us = []
    for k, flags in enumerate((0, tg.TG_FLAG_LNS8_STATE_SET)):
        Lr = tg.tg_layout.from_buffer_copy(L)
        Lr.flags = flags
        g = capture_graph(torch, lambda i, h: tg.tg_gemv_lns8_phase(Lr, wd[i % R], xa, A[k], S, h), R)
        g.replay()
        reps = max(2, min(20, int(2e5 / R)))
        us.append(event_time(torch, lambda i: g.replay(), reps, stream) / (reps * R) * 1e6)
        del g
    if not torch.equal(A[0], A[1]):
        raise SystemExit("LNS8 routes disagree")
    states = [len(set((w["xa"][g * 128:(g + 1) * 128] & 0x7F).tolist()) - {0}) for g in range(L.G)]
    return {"direct_us": round(us[0], 3), "stateset_us": round(us[1], 3),
            "stateset_over_direct": round(us[1] / us[0], 3),
            "states_per_group": round(float(np.mean(states)), 1), "weight_copies": R}


def run_sweep_lns8_routes(args):
    """The reuse sweep (rows sharing one activation vector), the activation
    state-cardinality sweep and the ternary zero-density sweep of the two LNS8
    routes, one JSON line per point."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300 import build as tgbuild
    tgbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    K = 4096
    for N in (1, 8, 32, 128, 512, 2048, 4096, 16384):
        r = _lns8_route_point(tg, torch, stream, dev, W.lns8(seed=1, N=N, K=K))
        print(json.dumps({"sweep": "reuse", "N": N, "K": K, **r}), flush=True)
        torch.cuda.empty_cache()
    for n in (1, 2, 4, 8, 16, 32, 64, 127):
        w = W.lns8(seed=2, N=4096, K=K)
        w["xa"] = W.lns8_activations_states(n, K, n)
        r = _lns8_route_point(tg, torch, stream, dev, w)
        print(json.dumps({"sweep": "cardinality", "N": 4096, "K": K, "code_set": n, **r}), flush=True)
        torch.cuda.empty_cache()
    for z in (0.0, 1 / 3, 0.9):
        w = W.lns8(seed=3, N=4096, K=K)
        w["t"] = W.trits_sparse(3, (4096, K), z)
        r = _lns8_route_point(tg, torch, stream, dev, w)
        print(json.dumps({"sweep": "zero_density", "N": 4096, "K": K, "zero_frac": round(z, 3), **r}),
              flush=True)
        torch.cuda.empty_cache()


def run_sweep_lns8_purelns(args):
    """Error study of the pure fractional-LNS route against the exact direct
    route by internal precision F, and its per-call time (N = K = 4096): the
    LNS8 workload (signed sums) and the same rows with every term positive."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300 import build as tgbuild
    tgbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    for name in ("signed", "positive"):
        w = W.lns8()
        if name == "positive":
            w["t"] = np.abs(w["t"])
            w["xa"] = w["xa"] & 0x7F
        blob, L = tg.tg_pack_weights(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
        R = min(_copies_for(blob.size), 128)
        wd = [dev(blob) for _ in range(R)]
        xa = dev(w["xa"])
        A = torch.empty((L.N, 8), dtype=torch.int64, device="cuda")
        S_exact = torch.empty((L.N,), dtype=torch.float64, device="cuda")
        tg.tg_gemv_lns8_phase(L, wd[0], xa, A, S_exact)
        S = torch.empty((L.N,), dtype=torch.float64, device="cuda")
        for F in range(1, 7):
            Lp = tg.tg_layout.from_buffer_copy(L)
            Lp.flags = tg.TG_FLAG_LNS8_PURE_LNS
            Lp.frac = F
            g = capture_graph(torch, lambda i, h: tg.tg_gemv_lns8_phase(Lp, wd[i % R], xa, A, S, h), R)
            g.replay()
            t = event_time(torch, lambda i: g.replay(), 3, stream) / (3 * R)
            del g
            tg.tg_gemv_lns8_phase(Lp, wd[0], xa, A, S)
            torch.cuda.synchronize()
            se, sp = S_exact.cpu().numpy(), S.cpu().numpy()
            nz = se != 0
            rel = np.abs(sp[nz] / se[nz] - 1.0)
            print(json.dumps({"sweep": "lns8_purelns", "terms": name, "F": F, "N": L.N, "K": L.K,
                              "us": round(t * 1e6, 3),
                              "rel_err_median": float(np.median(rel)), "rel_err_p90": float(np.quantile(rel, 0.9)),
                              "rel_err_p99": float(np.quantile(rel, 0.99)), "rel_err_max": float(rel.max()),
                              "sign_mismatch_rows": int(np.sum(np.sign(sp) != np.sign(se))),
                              "rows": int(L.N)}), flush=True)
        del wd
        torch.cuda.empty_cache()


def run_sweep_gemv_m(args):
    """Per-call time of tg_gemv_i8 against the token count M on the ffn_up and
    batched shapes (weights rotated over copies), one JSON line per point."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300 import build as tgbuild
    tgbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    hbm, _ = measured_peaks()

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    for name, N, K in (("ffn_up", 6912, 2560), ("batched", 13824, 5120)):
        w = W.batched(seed=5, M=64, N=N, K=K)
        blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
        R = min(_copies_for(blob.size), 128)
        wd = [dev(blob) for _ in range(R)]
        Lc = tg.tg_layout.from_buffer_copy(L)
        Lc.flags |= tg.TG_FLAG_CONST_WEIGHTS
        for M in (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64):
            xd = dev(w["x"][:M])
            y = torch.empty((M, N), dtype=torch.int64, device="cuda")
            times = []
            for lay in (L, Lc):
                g = capture_graph(torch, lambda i, h: tg.tg_gemv_i8(lay, wd[i % R], xd, M, y, h), R)
                g.replay()
                reps = max(2, min(20, int(4e4 / R)))
                times.append(event_time(torch, lambda i: g.replay(), reps, stream) / (reps * R))
                del g
            t, tc = times
            wbytes = L.mask_bytes + L.scale_bytes
            print(json.dumps({"sweep": "gemv_m", "shape": name, "N": N, "K": K, "M": M,
                              "us": round(t * 1e6, 3), "us_const_weights": round(tc * 1e6, 3),
                              "us_per_token": round(tc * 1e6 / M, 3),
                              "weight_gbs": round(wbytes / tc / 1e9, 1),
                              "frac_hbm": round(wbytes / tc / 1e9 / hbm, 4)}), flush=True)
        del wd
        torch.cuda.empty_cache()


def run_ffn_up_graph(args):
    """--sweep ffn_up_graph: only the headline's CUDA graph of back-to-back
    batch-1 GEMVs (weights flagged constant, rotated over copies > 4x L2),
    replayed --warmup then --steps times. A profiler target: the graph is the
    only thing this mode launches after the 4 warm-up calls made while it is
    captured, so `ncu --graph-profiling graph -s <4 + warmup>` lands on the
    first timed replay."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300 import build as tgbuild
    tgbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    w = W.ffn_up()
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    L.flags |= tg.TG_FLAG_CONST_WEIGHTS
    calls = args.gemvs_per_step
    R = max(int(math.ceil(2 * L2_BYTES / blob.size)), 1)
    wd = [dev(blob) for _ in range(R)]
    xd = dev(w["x"])
    y = torch.empty((1, L.N), dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    g = capture_graph(torch, lambda j, h: tg.tg_gemv_i8(L, wd[j % R], xd, 1, y, h), calls)
    for _ in range(args.warmup):
        g.replay()
    t = event_time(torch, lambda i: g.replay(), args.steps, stream)
    alg = L.mask_bytes + L.scale_bytes + L.K + L.N * 8
    per = t / (args.steps * calls)
    print(json.dumps({"sweep": "ffn_up_graph", "calls_per_graph": calls, "weight_copies": R,
                      "us_per_gemv": round(per * 1e6, 3), "alg_bytes_per_call": int(alg),
                      "achieved_gbs": round(alg / per / 1e9, 1)}), flush=True)


def run_row_only(args):
    """--row NAME: time one of the other hot-path calls alone (for profiler runs)."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300 import build as tgbuild
    tgbuild.build()
    torch.cuda.set_device(0)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    print(json.dumps(measure_rows(tg, torch, torch.cuda.current_stream(), dev,
                                  args.row.split(","))), flush=True)


def run_ours(args):
    import torch
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300 import build as tgbuild

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # one rank compiles the in-tree library (when it is stale) before the others
    # load it, so that no two compilers write the same files
    if rank == 0:
        tgbuild.build()
    barrier()
    if rank != 0:
        tgbuild.build()
    stream = torch.cuda.current_stream()
    s_handle = stream.cuda_stream

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    # workload and rotating weight copies
    w = W.ffn_up(seed=rank)
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    wbytes = L.mask_bytes + L.scale_bytes
    alg_bytes = wbytes + L.K + L.N * 8
    R = int(math.ceil(4 * L2_BYTES / blob.size))
    R = 1 << int(math.ceil(math.log2(R)))
    wd = [dev(blob) for _ in range(R)]
    xd = dev(w["x"])
    y = torch.empty((1, L.N), dtype=torch.int64, device="cuda")

    # parity guard on the timed configuration (checked against the oracle unless --no-cpu)
    tg.tg_gemv_i8(L, wd[0], xd, 1, y, s_handle)
    torch.cuda.synchronize()
    if not args.no_cpu:
        import oracle
        if not np.array_equal(y.cpu().numpy(), oracle.gemv_i8(w["t"], w["d"], w["x"])):
            raise SystemExit("parity failure on the bench workload")

    # The weights are constant during decode, so the calls may overlap their
    # weight streaming with the previous call's tail (TG_FLAG_CONST_WEIGHTS).
    # The same sweep without the flag is timed too and reported in the config.
    Lp = tg.tg_layout.from_buffer_copy(L)
    Lp.flags |= tg.TG_FLAG_CONST_WEIGHTS
    calls = args.gemvs_per_step
    graph_plain = capture_graph(torch, lambda j, h: tg.tg_gemv_i8(L, wd[j % R], xd, 1, y, h), calls)
    graph_plain.replay()
    t_plain = event_time(torch, lambda i: graph_plain.replay(), 3, stream) / (3 * calls)
    del graph_plain
    graph = capture_graph(torch, lambda j, h: tg.tg_gemv_i8(Lp, wd[j % R], xd, 1, y, h), calls)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    try:
        gpu_id = str(torch.cuda.get_device_properties(local).uuid)
        gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    clocks.start()

    barrier()
    torch.cuda.synchronize()
    clocks.mark("t0")
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier()
    dt = e0.elapsed_time(e1) / 1e3
    clk = clocks.stop()
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([dt], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dt = float(t.item())
    del graph

    launches = args.steps * calls
    per_gemv = dt / launches
    value = world * launches * wbytes / dt / 1e9
    hbm, peak_kind = measured_peaks()
    achieved = alg_bytes / per_gemv / 1e9

    # e2e: per step, activations in from pinned host memory, every call made
    # eagerly through the public API, outputs read back. The caller's buffers
    # (per-call views of the staging tensors) exist before the loop, as in a
    # serving loop; the outputs go back in chunks on a second stream as soon as
    # their calls are done, so the read-back overlaps the remaining calls.
    xs_host = torch.from_numpy(np.tile(w["x"], (GEMVS_PER_STEP, 1))).pin_memory()
    xs_dev = torch.empty(xs_host.shape, dtype=xs_host.dtype, device="cuda")
    ys_dev = torch.empty((GEMVS_PER_STEP, L.N), dtype=torch.int64, device="cuda")
    ys_host = torch.empty((GEMVS_PER_STEP, L.N), dtype=torch.int64).pin_memory()
    # the calls take device addresses (the binding accepts tensors or plain
    # integers); a decode loop resolves its buffers' addresses once, not per call
    x_views = [xs_dev[j].data_ptr() for j in range(GEMVS_PER_STEP)]
    y_views = [ys_dev[j].data_ptr() for j in range(GEMVS_PER_STEP)]
    w_views = [wd[j % R].data_ptr() for j in range(GEMVS_PER_STEP)]
    readback_chunk = 128
    assert GEMVS_PER_STEP % readback_chunk == 0
    copy_stream = torch.cuda.Stream()
    chunk_done = [torch.cuda.Event() for _ in range(GEMVS_PER_STEP // readback_chunk)]

    def e2e_step():
        xs_dev.copy_(xs_host, non_blocking=True)
        for c in range(0, GEMVS_PER_STEP, readback_chunk):
            for j in range(c, c + readback_chunk):
                tg.tg_gemv_i8(Lp, w_views[j], x_views[j], 1, y_views[j], s_handle)
            ev = chunk_done[c // readback_chunk]
            ev.record(stream)
            copy_stream.wait_event(ev)
            with torch.cuda.stream(copy_stream):
                ys_host[c:c + readback_chunk].copy_(ys_dev[c:c + readback_chunk], non_blocking=True)
        torch.cuda.synchronize()

    for _ in range(2):
        e2e_step()
    e2e_steps = max(3, min(args.steps, 10))
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_dt = time.perf_counter() - t0
    if not np.array_equal(ys_host[0].numpy(), y[0].cpu().numpy()):
        raise SystemExit("e2e result differs from the device-timed result")
    e2e_val = world * e2e_steps * GEMVS_PER_STEP * wbytes / e2e_dt / 1e9

    # The same step with each chunk's calls replayed from a CUDA graph captured
    # once before the timed region, as a decode loop does: the activations still
    # come in from pinned host memory and every output goes back, every step.
    chunk_graphs = [capture_graph(torch, lambda j, h, c=c: tg.tg_gemv_i8(Lp, w_views[c + j], x_views[c + j], 1,
                                                                         y_views[c + j], h), readback_chunk)
                    for c in range(0, GEMVS_PER_STEP, readback_chunk)]

    def e2e_graph_step():
        xs_dev.copy_(xs_host, non_blocking=True)
        for ci, gch in enumerate(chunk_graphs):
            gch.replay()
            ev = chunk_done[ci]
            ev.record(stream)
            copy_stream.wait_event(ev)
            c = ci * readback_chunk
            with torch.cuda.stream(copy_stream):
                ys_host[c:c + readback_chunk].copy_(ys_dev[c:c + readback_chunk], non_blocking=True)
        torch.cuda.synchronize()

    for _ in range(2):
        e2e_graph_step()
    ys_host.zero_()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_graph_step()
    e2e_graph_dt = time.perf_counter() - t0
    if not np.array_equal(ys_host[-1].numpy(), y[0].cpu().numpy()):
        raise SystemExit("graph e2e result differs from the device-timed result")
    e2e_graph_val = world * e2e_steps * GEMVS_PER_STEP * wbytes / e2e_graph_dt / 1e9
    del chunk_graphs

    # one call at a time (the plain call, no dependent launch), weights rotated
    iso = isolated_call_stats(torch, stream, lambda i: tg.tg_gemv_i8(L, wd[i % R], xd, 1, y, s_handle))

    if rank != 0:
        return

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "seed": rank,
                   "inputs_sha256_16": hashlib.sha256(blob.tobytes() + np.ascontiguousarray(w["x"]).tobytes())
                   .hexdigest()[:16],
                   "gemvs_per_step": calls, "weight_copies": R,
                   "weight_copy_bytes": int(blob.size),
                   "l2": f"weights rotated over {R} copies ({R * blob.size / 2**20:.0f} MiB > 4x L2)",
                   "launch": "each step's calls replayed from one CUDA graph; weights flagged "
                             "constant (programmatic dependent launch between calls)",
                   "us_per_gemv_without_const_flag": round(t_plain * 1e6, 3),
                   "us_per_gemv": round(per_gemv * 1e6, 3),
                   "pct_hbm_peak": round(100 * value / world / hbm, 2),
                   "pct_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(xs_host.numel()),
                "d2h_bytes_per_step": int(ys_host.numel() * 8)},
        "e2e_graph": {"value": round(e2e_graph_val, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": int(xs_host.numel()),
                      "d2h_bytes_per_step": int(ys_host.numel() * 8),
                      "launch": f"each chunk of {readback_chunk} calls replayed from a CUDA graph captured "
                                "before the timed region; copies in and out inside it"},
        "wall_us": {"graph_back_to_back": round(per_gemv * 1e6, 3),
                    "graph_back_to_back_without_const_flag": round(t_plain * 1e6, 3),
                    "one_call_at_a_time": iso},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": profiled_traffic("gemv_i8.cu", "ffn_up"),
                     "kernel": "gemv_i8_m1_kernel", "alg_bytes_per_launch": int(alg_bytes),
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "clocks": clk,
    }
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_record(w, 8.0, 8.0)
    del wd
    torch.cuda.empty_cache()
    if not args.no_rows:
        line["rows"] = measure_rows(tg, torch, stream, dev)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.sweep == "lns8_routes":
        run_sweep_lns8_routes(args)
    elif args.sweep == "gemv_m":
        run_sweep_gemv_m(args)
    elif args.sweep == "lns8_purelns":
        run_sweep_lns8_purelns(args)
    elif args.sweep == "ffn_up_graph":
        run_ffn_up_graph(args)
    elif args.row:
        run_row_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
