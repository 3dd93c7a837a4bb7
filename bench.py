"""Benchmark of the fused dequantize-and-multiply hot path on GB300.

Default workload (one step): the one-token BF16 GEMV and the one-token F16
GEMV at k = n = 4096 (weights ~N(0, 0.02) rounded to 16 bits, x ~ N(0, 1),
seed 2), i.e. 2 x 33,554,432 weight bytes per step. Metric: effective weight
GB/s = weight bytes / time (x and y bytes excluded). Inputs are resident in
HBM; every step reads a different one of several distinct weight copies whose
total is > 3x the L2 size, so each step streams W from HBM.

The JSON line also carries the other workloads measured the same way
(Q4_0 / Q4_K / Q6_K / Q8_0 / Q5_0 GEMVs, the expert-indexed products, the
gated pairs, the affine GEMVs and N = 512 products, the backward-input cases,
and the Q4_K N-token product in TFLOP/s at N = 1, 8, 64, 512 on both paths),
the roofline of the dominant kernel against the measured HBM copy bandwidth,
an end-to-end figure through the host-buffer C entry point (qmm_matmul_host:
W and x copied in, y copied out, every step), SM clocks sampled during the
timed region, and the oracle timed on the host's cores as a CPU baseline.

--case <workload> times one workload alone (for profiling one kernel).

--impl reference times the oracle (plain C, one host core) on the same
workload: each step is the full oracle product of both weight matrices.
Under torchrun (N > 1) every rank runs its own replica (weak scaling); the
time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qmm_synth  # noqa: E402

# the workload every arm of the bench reports (the same string in each line)
HEADLINE_WORKLOAD = "bf16+f16 GEMV k=n=4096, 1 token (one step = both GEMVs)"


def headline_config(ws: int, wbytes_step: int, l2_bytes: int) -> dict:
    """The `config` of the headline line, the same in both arms."""
    ncop = max(1, min(64, -(-3 * l2_bytes // max(wbytes_step // 2, 1))))
    return {"workload": HEADLINE_WORKLOAD, "weight_bytes_per_step": int(wbytes_step),
            "l2": f"inputs larger than L2: {ncop} distinct copies of each weight matrix rotate "
                  f"(> 3x L2 of {l2_bytes >> 20} MiB)",
            "parallelism": f"replicas x{ws}"}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES_DEFAULT = 129 * 1024 * 1024


# ------------------------------------------------------------ utilities ----

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity at world size 1)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_weight_gguf_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the kernel sources as they are now."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ------------------------------------------------------------ reference ----

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    fmts = [qmm_synth.workload("bf16_gemv"), qmm_synth.workload("f16_gemv")]
    wbytes = sum(w.size for _, _, _, w, _ in fmts)
    n = fmts[0][2]
    rb = [w.size // nn for _, _, nn, w, _ in fmts]
    state = {"off": 0}

    def step(rows):
        # rows [off, off + rows) of both matrices (rotating), through the oracle
        o = state["off"]
        done = 0
        for (fmt, k, _, w, x), r in zip(fmts, rb):
            m = min(rows, n - o)
            oracle.matmul(fmt, np.ascontiguousarray(w[o * r:(o + m) * r]), x, k, m)
            done += m * r
        state["off"] = 0 if o + rows >= n else o + rows
        return done

    # a whole step is both full products; when warm-up plus the timed steps
    # would take more than about a minute that way, each step is a block of
    # rows of both matrices instead, sized to fit the minute
    t0 = time.perf_counter()
    step(n)
    full = time.perf_counter() - t0
    total = args.steps + args.warmup
    rows = n
    if total * full > 60.0:
        rows = max(8, min(n, int(n * 60.0 / (total * full)) // 8 * 8))
    for _ in range(args.warmup):
        step(rows)
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += step(rows)
    elapsed = time.perf_counter() - t0
    dt = elapsed / args.steps
    value = done / elapsed / 1e9
    sample = ("full oracle product of both 4096x4096 weight matrices per step" if rows == n else
              f"{rows} of the 4096 rows of both 4096x4096 weight matrices per step, the rows "
              f"rotating through the matrices (a whole step would take {full:.2f} s)")
    line = {"impl": "reference", "metric": "effective weight GB/s", "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(ws, wbytes, L2_BYTES_DEFAULT),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- native ----

def _oracle_share(job):
    """One worker of the all-core CPU baseline: rows [i*n/P, (i+1)*n/P) of
    both 4096x4096 GEMVs through the oracle, repeated until `seconds` pass."""
    i, parts, seconds = job
    import oracle
    fmts = [qmm_synth.workload("bf16_gemv"), qmm_synth.workload("f16_gemv")]
    shares = []
    for fmt, k, n, w, x in fmts:
        r0, r1 = i * n // parts, (i + 1) * n // parts
        rb = w.size // n
        shares.append((fmt, k, r1 - r0, np.ascontiguousarray(w[r0 * rb:r1 * rb]), x))
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for fmt, k, m, ws, x in shares:
            oracle.matmul(fmt, ws, x, k, m)
            done += ws.size
    return done, time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def cpu_baseline(seconds: float = 10.0):
    """The oracle as it stands on the host: single-threaded, and row-partitioned
    over every core (one spawned process per core; spawn, since the CUDA
    context of this process must not be forked)."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    fmts = [qmm_synth.workload("bf16_gemv"), qmm_synth.workload("f16_gemv")]
    done = 0
    single_s = max(1.0, seconds / 2)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < single_s:
        for fmt, k, n, w, x in fmts:
            oracle.matmul(fmt, w, x, k, n)
            done += w.size
    dt = time.perf_counter() - t0
    single = {"value": done / dt / 1e9, "unit": "GB/s", "cores": 1,
              "sample": f"bf16+f16 4096x4096 GEMVs repeated for {dt:.1f} s ({done / 1e6:.0f} MB)"}
    cores = max(1, os.cpu_count() or 1)
    try:
        with mp.get_context("spawn").Pool(cores) as pool:
            res = pool.map(_oracle_share, [(i, cores, seconds) for i in range(cores)])
        total = sum(r[0] for r in res)
        wall = max(r[1] for r in res)
        return {"value": total / wall / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"oracle (plain C, f64 sums) on the bf16+f16 4096x4096 GEMVs, rows split "
                          f"over {cores} processes, repeated for {wall:.1f} s "
                          f"({total / 1e6:.0f} MB of weights)",
                "cpu_model": cpu_model(),
                "single_core": single}
    except Exception as e:  # a pool that cannot start: report the single-core figure
        single.update({"kind": "oracle", "note": f"all-core run unavailable: {e}"})
        return single


class Runner:
    """Device-resident inputs with rotation over distinct weight copies."""

    def __init__(self, torch, q, device):
        self.torch, self.q, self.dev = torch, q, device
        self.stream = torch.cuda.current_stream(device)
        try:
            self.l2 = torch.cuda.get_device_properties(device).L2_cache_size
        except Exception:
            self.l2 = L2_BYTES_DEFAULT

    def copies_for(self, nbytes: int) -> int:
        return max(1, min(64, -(-3 * self.l2 // max(nbytes, 1))))

    def weights(self, w_np, copies):
        base = self.torch.from_numpy(w_np).to(self.dev)
        return [base] + [base.clone() for _ in range(copies - 1)]


def queue_ahead(torch, stream, ms=1.0):
    """Keep the device busy for about `ms` (a spin of torch's, outside any
    timed region) so that the launches that follow are all queued before the
    first one runs: the device-timed region then holds the K steps back to
    back and not the host's latency to issue the first of them."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(min(ms, 5.0) * 2.1e6))


def time_loop(torch, launch, steps, warmup, ncopies, stream, inner_events=None):
    """Time `steps` calls of launch(i) (i rotates the weight copy) with CUDA
    events on `stream`; returns seconds per call."""
    for i in range(warmup):
        launch(i % ncopies)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    queue_ahead(torch, stream, 0.5 + 0.02 * steps)
    start.record(stream)
    for i in range(steps):
        launch(i % ncopies)
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3 / steps


def run_native(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    import quantized_weight_gguf_gb300 as q
    from quantized_weight_gguf_gb300 import build_lib
    if not os.path.exists(q.LIB_PATH):
        build_lib.build()
    lib = q.load()
    r = Runner(torch, q, device)
    stream = r.stream
    sptr = stream.cuda_stream
    hbm_peak, tc_peak, tc_sust, peak_src = peaks()

    # ---------------- headline: bf16 + f16 GEMV, k = n = 4096 ----------------
    work = [qmm_synth.workload("bf16_gemv"), qmm_synth.workload("f16_gemv")]
    wbytes_each = work[0][3].size
    ncop = r.copies_for(wbytes_each)
    wcopies = [r.weights(w, ncop) for (_, _, _, w, _) in work]
    xs = [torch.from_numpy(x).to(device) for (*_, x) in work]
    ys = [torch.empty((1, n), device=device) for (_, _, n, _, _) in work]
    flags = 0 if args.no_overlap else (q.FLAG_OVERLAP_PREV | q.FLAG_X_READY)
    argsets = [[q.make_args(fmt, wc[c], xs[i], ys[i], k, n, 1, stream=stream, flags=flags)
                for c in range(ncop)] for i, ((fmt, k, n, _, _), wc) in enumerate(zip(work, wcopies))]
    import ctypes
    refs = [[ctypes.byref(a) for a in al] for al in argsets]
    mm = lib.qmm_matmul_ex

    def step(c):
        if mm(refs[0][c]) or mm(refs[1][c]):
            raise RuntimeError(q.qmm_last_error())

    for i in range(max(args.warmup, 3)):
        step(i % ncop)
    torch.cuda.synchronize()
    q.qmm_device_status(stream)
    K = args.steps
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.25)
        # timed region: K steps back to back, events only at its ends (an event
        # between launches would stop each GEMV from overlapping the previous one)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        queue_ahead(torch, stream, 0.5 + 0.02 * K)
        start.record(stream)
        for i in range(K):
            step(i % ncop)
        end.record(stream)
        end.synchronize()
        # dominant kernel alone: average launch duration of the BF16 GEMV over a
        # back-to-back loop of it (same flags, same rotation)
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        KR = max(K, 500)
        queue_ahead(torch, stream, 0.5 + 0.01 * KR)
        r0.record(stream)
        for i in range(KR):
            if mm(refs[0][i % ncop]):
                raise RuntimeError(q.qmm_last_error())
        r1.record(stream)
        r1.synchronize()
        # the same kernel as plain stream-ordered launches (no programmatic
        # overlap: what a dependent chain of products gets)
        fmt0, k0, n0 = work[0][:3]
        plain = [q.make_args(fmt0, wcopies[0][c], xs[0], ys[0], k0, n0, 1, stream=stream, flags=0)
                 for c in range(ncop)]
        prefs = [ctypes.byref(a) for a in plain]
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        queue_ahead(torch, stream, 0.5 + 0.01 * KR)
        p0.record(stream)
        for i in range(KR):
            if mm(prefs[i % ncop]):
                raise RuntimeError(q.qmm_last_error())
        p1.record(stream)
        p1.synchronize()
        time.sleep(0.25)
    torch.cuda.synchronize()
    barrier(ws)
    elapsed = start.elapsed_time(end) / 1e3
    elapsed = max_over_ranks(elapsed, ws, device)
    q.qmm_device_status(stream)
    t_bf16 = r0.elapsed_time(r1) / 1e3 / KR
    t_bf16_plain = p0.elapsed_time(p1) / 1e3 / KR
    ms_per_step = elapsed / K * 1e3
    value = ws * 2 * wbytes_each / (elapsed / K) / 1e9
    clocks = clk.summary()

    # ---------------- e2e: host buffers through qmm_matmul_host ----------------
    e2e = None
    try:
        hw = [torch.from_numpy(w).pin_memory() for (_, _, _, w, _) in work]
        hx = [torch.from_numpy(x).pin_memory() for (*_, x) in work]
        hy = [torch.empty((1, n)).pin_memory() for (_, _, n, _, _) in work]
        dw = [wc[0] for wc in wcopies]
        hargs = [q.make_args(fmt, hw[i], hx[i], hy[i], k, n, 1, stream=stream)
                 for i, (fmt, k, n, _, _) in enumerate(work)]

        def e2e_step():
            for i in range(2):
                q.qmm_matmul_host(hargs[i], dw[i], xs[i], ys[i])
            stream.synchronize()   # y must be on the host at the end of the step

        for _ in range(3):
            e2e_step()
        ek = max(5, K // 4)
        t0 = time.perf_counter()
        for _ in range(ek):
            e2e_step()
        et = max_over_ranks((time.perf_counter() - t0) / ek, ws, device)
        h2d = sum(w.size + x.nbytes for (_, _, _, w, x) in work)
        d2h = sum(4 * n for (_, _, n, _, _) in work)
        e2e = {"value": ws * 2 * wbytes_each / et / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": et * 1e3,
               "note": "qmm_matmul_host: pinned host W and x copied in, y copied out, stream synchronized, every step"}
    except Exception as ex:  # pragma: no cover - reported, not hidden
        e2e = {"value": None, "unit": "GB/s", "error": str(ex)[:200]}

    # ---------------- other workloads of the path ----------------
    others = {}
    if ws == 1 and not args.quick:
        # single-GPU runs only: the tensor-core cases use cluster-shared x
        # tile copies, which stay within one GPU's own memory
        others = measure_other_workloads(torch, q, lib, r, stream, hbm_peak, tc_peak)

    # roofline of the dominant kernel (bf16 GEMV)
    achieved = wbytes_each / t_bf16 / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": recorded_traffic("gemv_bf16_4096x4096"),
            "kernel": "gemv_kernel<BF16> (k=n=4096)", "peak_source": f"{peak_src} hbm_gbs",
            "duration_us": t_bf16 * 1e6,
            "duration_from": f"CUDA events around {KR} back-to-back launches of this kernel alone",
            "stream_ordered": {"duration_us": t_bf16_plain * 1e6,
                               "achieved": wbytes_each / t_bf16_plain / 1e9,
                               "frac": wbytes_each / t_bf16_plain / 1e9 / hbm_peak,
                               "note": "the same kernel launched without QMM_FLAG_OVERLAP_PREV "
                                       "(each launch waits for the previous one to finish)"}}

    line = {"metric": "effective weight GB/s", "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
            "data": "synthetic",
            "config": headline_config(ws, 2 * wbytes_each, r.l2),
            "timing": {"launch": ("stream-ordered" if args.no_overlap else
                                  "programmatic dependent launch (QMM_FLAG_OVERLAP_PREV | "
                                  "QMM_FLAG_X_READY): consecutive GEMVs on the same x; each streams "
                                  "its weights and computes while the previous one finishes, and "
                                  "stores y after it"),
                       "queue": "a device-side sleep (torch.cuda._sleep) precedes the start event, "
                                "so that the K steps are queued before the first one runs: the "
                                "host's latency to issue them is outside the device-timed region "
                                "(it is inside e2e)",
                       "rotation": f"{ncop} copies per format"},
            "roofline": roof, "e2e": e2e, "clocks": clocks,
            "gpu_launches": 2 * K,
            "other_workloads": others}
    if rank == 0 and not args.quick:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_other_workloads(torch, q, lib, r, stream, hbm_peak, tc_peak):
    import ctypes
    out = {}
    mm = lib.qmm_matmul_ex
    dev = r.dev

    def gemv_case(name, tiles=1, reps=50):
        fmt, k, n, w, x = qmm_synth.workload(name)
        ncop = r.copies_for(w.size)
        wc = r.weights(w, ncop)
        xd = torch.from_numpy(x).to(dev)
        yd = torch.empty((1, n), device=dev)
        tile = n // tiles
        al = [[ctypes.byref(q.make_args(fmt, wc[c], xd, yd, k, n, 1, j_start=t * tile,
                                        j_end=(t + 1) * tile, accumulate=False, stream=stream,
                                        flags=q.FLAG_OVERLAP_PREV | q.FLAG_X_READY))
               for t in range(tiles)] for c in range(ncop)]
        keep = al  # noqa: F841

        def launch(c):
            for a in al[c]:
                if mm(a):
                    raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 5, ncop, stream)
        q.qmm_device_status(stream)
        gbs = w.size / dt / 1e9
        return {"us": dt * 1e6, "weight_gbs": gbs, "frac_hbm": gbs / hbm_peak,
                "weight_bytes": int(w.size), "launches_per_call": tiles}

    out["q4_0_gemv"] = gemv_case("q4_0_gemv", reps=200)
    out["q4_0_gemv"]["note"] = ("73,728 weight bytes: every rotated copy fits in L2, so this is the "
                                "L2-resident figure; launch-latency bound, fraction not meaningful")
    out["q4_k_gemv"] = gemv_case("q4_k_gemv")
    out["q6_k_head_8_tiles"] = gemv_case("q6_k_head", tiles=8, reps=20)
    out["q6_k_head_untiled"] = gemv_case("q6_k_head", tiles=1, reps=20)
    out["q8_0_gemv"] = gemv_case("q8_0_gemv")
    out["q5_0_gemv"] = gemv_case("q5_0_gemv")

    # expert-indexed product: each (position, slot) multiplies by the slice its
    # id selects; the bytes are the selected slices (one read per pair)
    ex = lib.qmm_matmul_experts

    def expert_case(name, n_pos, reps=50, path=q.PATH_AUTO):
        fmt, k, n, n_exp, w, x, ids = qmm_synth.expert_workload(name, n_pos=n_pos)
        slice_bytes = w.size // n_exp
        pairs = ids.size
        touched = len(np.unique(ids)) * slice_bytes
        ncop = r.copies_for(touched)
        wc = r.weights(w, ncop)
        xd = torch.from_numpy(x).to(dev)
        idd = torch.from_numpy(ids).to(dev)
        yd = torch.empty((pairs, n), device=dev)
        args = [q.make_args(fmt, wc[c], xd, yd, k, n, n_pos, stream=stream, path=path,
                            flags=q.FLAG_OVERLAP_PREV | q.FLAG_X_READY) for c in range(ncop)]
        need = q.qmm_experts_workspace_bytes(args[0], n_exp, ids.shape[1])
        wsb = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        if need:
            for a in args:
                a.workspace, a.workspace_bytes = wsb.data_ptr(), need
        al = [ctypes.byref(a) for a in args]
        ip = ctypes.c_void_p(idd.data_ptr())

        def launch(c):
            if ex(al[c], ip, n_exp, ids.shape[1]):
                raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 5, ncop, stream)
        q.qmm_device_status(stream)
        res = {"us": dt * 1e6, "pairs": int(pairs), "distinct_bytes": int(touched),
               "form": "grouped tensor-core" if need else "one GEMV per pair"}
        if need:
            # grouped: each selected slice is decoded once per token tile
            fl = 2.0 * pairs * k * n
            res.update({"tflops": fl / dt / 1e12, "frac_bf16_peak": fl / dt / 1e12 / tc_peak,
                        "distinct_weight_gbs": touched / dt / 1e9, "launches_per_call": 3})
        else:
            gbs = pairs * slice_bytes / dt / 1e9
            res.update({"weight_gbs": gbs, "frac_hbm": gbs / hbm_peak,
                        "weight_bytes": int(pairs * slice_bytes), "launches_per_call": 1})
        return res

    for name in sorted(qmm_synth.EXPERT_WORKLOADS):
        out[f"{name}_pos1"] = expert_case(name, 1)
        out[f"{name}_pos4"] = expert_case(name, 4)
        out[f"{name}_pos64_gemv"] = expert_case(name, 64, reps=20, path=q.PATH_GEMV)
        out[f"{name}_pos64_grouped"] = expert_case(name, 64, reps=20, path=q.PATH_MMA)

    exa = lib.qmm_matmul_experts_affine

    def expert_affine_case(bits, n_pos, reps=50):
        # affine experts of the same shape: k=2048, n=768, 64 experts, top 8
        k, n, n_exp, top_k = 2048, 768, 64, 8
        rng = np.random.default_rng(20 + bits)
        w, sc, bi = qmm_synth.gen_affine(bits, k, n * n_exp, rng)
        x = qmm_synth.gen_x(n_pos, k, rng)
        ids = qmm_synth.gen_ids(n_pos, top_k, n_exp, rng)
        slice_bytes = (w.size + sc.nbytes + bi.nbytes) // n_exp
        pairs = ids.size
        ncop = r.copies_for(len(np.unique(ids)) * slice_bytes)
        wc = r.weights(w, ncop)
        scd = torch.from_numpy(sc.view(np.int16)).to(dev)
        bid = torch.from_numpy(bi.view(np.int16)).to(dev)
        xd = torch.from_numpy(x).to(dev)
        idd = torch.from_numpy(ids).to(dev)
        yd = torch.empty((pairs, n), device=dev)
        al = [ctypes.byref(q.make_args(f"affine{bits}", wc[c], xd, yd, k, n, n_pos, stream=stream,
                                       flags=q.FLAG_OVERLAP_PREV | q.FLAG_X_READY))
              for c in range(ncop)]
        ip, sp, bp = (ctypes.c_void_p(t.data_ptr()) for t in (idd, scd, bid))

        def launch(c):
            if exa(al[c], ip, n_exp, top_k, sp, bp):
                raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 5, ncop, stream)
        q.qmm_device_status(stream)
        gbs = pairs * slice_bytes / dt / 1e9
        return {"us": dt * 1e6, "weight_gbs": gbs, "frac_hbm": gbs / hbm_peak,
                "weight_bytes": int(pairs * slice_bytes), "pairs": int(pairs),
                "note": "scale and bias arrays of the code words rotate with one copy (L2-resident)",
                "launches_per_call": 1}

    out["affine4_experts_pos1"] = expert_affine_case(4, 1)

    # MLX-style affine matrices: bytes = codes + bf16 scales + bf16 biases
    aff = lib.qmm_matmul_affine

    def affine_case(name, n_tokens=None, reps=50):
        bits, k, n, w, sc, bi, x = qmm_synth.affine_workload(name, n_tokens=n_tokens)
        nt = x.shape[0]
        total = w.size + sc.nbytes + bi.nbytes
        ncop = r.copies_for(total)
        wc = r.weights(w, ncop)
        sc_c = r.weights(sc.view(np.int16), ncop)
        bi_c = r.weights(bi.view(np.int16), ncop)
        xd = torch.from_numpy(x).to(dev)
        yd = torch.empty((nt, n), device=dev)
        fl = q.FLAG_OVERLAP_PREV | q.FLAG_X_READY if nt == 1 else 0
        a0 = q.make_args(f"affine{bits}", wc[0], xd, yd, k, n, nt, stream=stream, flags=fl)
        need = q.qmm_workspace_bytes(a0)
        wsb = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        al = [q.make_args(f"affine{bits}", wc[c], xd, yd, k, n, nt, stream=stream, flags=fl,
                          workspace=wsb if need else None, workspace_bytes=need)
              for c in range(ncop)]
        refs = [(ctypes.byref(al[c]), ctypes.c_void_p(sc_c[c].data_ptr()),
                 ctypes.c_void_p(bi_c[c].data_ptr())) for c in range(ncop)]

        def launch(c):
            if aff(*refs[c]):
                raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 5, ncop, stream)
        q.qmm_device_status(stream)
        gbs = total / dt / 1e9
        res = {"us": dt * 1e6, "weight_gbs": gbs, "frac_hbm": gbs / hbm_peak,
               "weight_bytes": int(total), "launches_per_call": 1 if nt == 1 else 2}
        if nt > 1:
            fl_ = 2.0 * nt * k * n
            res.update({"tflops": fl_ / dt / 1e12, "frac_bf16_peak": fl_ / dt / 1e12 / tc_peak})
        return res

    # gated pair (SwiGLU) on the Q4_K FFN shape: gate and up matrices, one
    # fused launch; bytes = both matrices
    glu = lib.qmm_matmul_glu

    def glu_case(name, act, reps=50):
        fmt, k, n, w, x = qmm_synth.workload(name)
        w2 = qmm_synth.gen_weights(fmt, k, n, np.random.default_rng(77))
        ncop = r.copies_for(2 * w.size)
        wg, wu = r.weights(w, ncop), r.weights(w2, ncop)
        xd = torch.from_numpy(x).to(dev)
        yd = torch.empty((1, n), device=dev)
        al = [ctypes.byref(q.make_args(fmt, wg[c], xd, yd, k, n, 1, stream=stream,
                                       flags=q.FLAG_OVERLAP_PREV | q.FLAG_X_READY))
              for c in range(ncop)]
        ups = [ctypes.c_void_p(wu[c].data_ptr()) for c in range(ncop)]

        def launch(c):
            if glu(al[c], ups[c], act):
                raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 5, ncop, stream)
        q.qmm_device_status(stream)
        gbs = 2 * w.size / dt / 1e9
        return {"us": dt * 1e6, "weight_gbs": gbs, "frac_hbm": gbs / hbm_peak,
                "weight_bytes": int(2 * w.size), "launches_per_call": 1}

    out["q4_k_swiglu_pair"] = glu_case("q4_k_gemv", q.ACT_SWIGLU)
    out["q8_0_geglu_pair"] = glu_case("q8_0_gemv", q.ACT_GEGLU)

    def glu_tokens_case(nt, act, reps=20):
        # several tokens: the gate product into scratch, then the up product
        # whose epilogue writes act(gate) * up
        fmt, k, n, w, x = qmm_synth.workload("q4_k_prefill", n_tokens=nt)
        w2 = qmm_synth.gen_weights(fmt, k, n, np.random.default_rng(78))
        ncop = r.copies_for(2 * w.size)
        wg, wu = r.weights(w, ncop), r.weights(w2, ncop)
        xd = torch.from_numpy(x).to(dev)
        yd = torch.empty((nt, n), device=dev)
        a0 = q.make_args(fmt, wg[0], xd, yd, k, n, nt, stream=stream)
        need = q.qmm_glu_workspace_bytes(a0)
        wsb = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        al = [ctypes.byref(q.make_args(fmt, wg[c], xd, yd, k, n, nt, stream=stream, workspace=wsb,
                                       workspace_bytes=need)) for c in range(ncop)]
        ups = [ctypes.c_void_p(wu[c].data_ptr()) for c in range(ncop)]

        def launch(c):
            if glu(al[c], ups[c], act):
                raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 3, ncop, stream)
        q.qmm_device_status(stream)
        fl = 4.0 * nt * k * n
        return {"us": dt * 1e6, "tflops": fl / dt / 1e12, "frac_bf16_peak": fl / dt / 1e12 / tc_peak,
                "launches_per_call": 4,
                "note": "gate product into scratch; the up product's epilogue applies act(gate)"}

    out["q4_k_swiglu_pair_N64"] = glu_tokens_case(64, q.ACT_SWIGLU)
    out["q4_k_swiglu_pair_N512"] = glu_tokens_case(512, q.ACT_SWIGLU)

    out["affine4_gemv"] = affine_case("affine4_gemv")
    out["affine8_gemv"] = affine_case("affine8_gemv")
    out["affine4_prefill_512"] = affine_case("affine4_prefill", reps=20)
    out["affine8_prefill_512"] = affine_case("affine8_prefill", reps=20)

    # backward with respect to the input, dx = W^T dy: the output head in 8
    # sum-axis tiles (first writes, the rest accumulate), and the Q4_K FFN shape
    bw = lib.qmm_matmul_backward_input

    def back_case(name, tiles=1, reps=20):
        fmt, k, n, w, _ = qmm_synth.workload(name)
        ncop = r.copies_for(w.size)
        wc = r.weights(w, ncop)
        dyd = torch.from_numpy(np.random.default_rng(4).standard_normal(n).astype(np.float32)).to(dev)
        dxd = torch.empty(k, device=dev)
        tile = n // tiles
        al = [[q.make_args(fmt, wc[c], dyd, dxd, k, n, 1, j_start=t * tile, j_end=(t + 1) * tile,
                           accumulate=t > 0, stream=stream,
                           flags=q.FLAG_OVERLAP_PREV | q.FLAG_X_READY)
               for t in range(tiles)] for c in range(ncop)]
        need = max(q.qmm_backward_input_workspace_bytes(a) for a in al[0])
        wsb = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        for row in al:
            for a in row:
                a.workspace, a.workspace_bytes = wsb.data_ptr(), need
        refs = [[ctypes.byref(a) for a in row] for row in al]

        def launch(c):
            for a in refs[c]:
                if bw(a):
                    raise RuntimeError(q.qmm_last_error())
        dt = time_loop(torch, launch, reps, 3, ncop, stream)
        q.qmm_device_status(stream)
        gbs = w.size / dt / 1e9
        return {"us": dt * 1e6, "weight_gbs": gbs, "frac_hbm": gbs / hbm_peak,
                "weight_bytes": int(w.size), "launches_per_call": 2 * tiles}

    out["q6_k_head_backward_input_8_tiles"] = back_case("q6_k_head", tiles=8)
    out["q4_k_backward_input"] = back_case("q4_k_gemv", reps=50)

    # Q4_K N-token product: both paths at N = 1, 8, 64, 512
    fmt, k, n, w, _ = qmm_synth.workload("q4_k_prefill", n_tokens=1)
    ncop = r.copies_for(w.size)
    wc = r.weights(w, ncop)
    pre = {}
    for nt in (1, 8, 64, 512):
        _, _, _, _, x = qmm_synth.workload("q4_k_prefill", n_tokens=nt)
        xd = torch.from_numpy(x).to(dev)
        yd = torch.empty((nt, n), device=dev)
        ws_bytes = 0
        row = {}
        for pname, path in (("gemv", q.PATH_GEMV), ("mma", q.PATH_MMA)):
            if pname == "gemv" and nt > 64:
                continue
            a0 = q.make_args(fmt, wc[0], xd, yd, k, n, nt, path=path, stream=stream)
            need = q.qmm_workspace_bytes(a0)
            wsb = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
            al = [q.make_args(fmt, wc[c], xd, yd, k, n, nt, path=path, workspace=wsb if need else None,
                              workspace_bytes=need, stream=stream) for c in range(ncop)]
            refs = [ctypes.byref(a) for a in al]

            def launch(c, refs=refs):
                if mm(refs[c]):
                    raise RuntimeError(q.qmm_last_error())
            reps = 20 if nt >= 64 else 50
            dt = time_loop(torch, launch, reps, 5, ncop, stream)
            q.qmm_device_status(stream)
            flops = 2.0 * nt * k * n
            row[pname] = {"us": dt * 1e6, "tflops": flops / dt / 1e12,
                          "frac_bf16_peak": flops / dt / 1e12 / tc_peak,
                          "weight_gbs": w.size / dt / 1e9}
        pre[f"N={nt}"] = row
    out["q4_k_prefill"] = pre
    return out


def run_case(args):
    """One workload alone, for profiling: warmup + steps calls, per-call time printed."""
    import ctypes
    import torch
    import quantized_weight_gguf_gb300 as q
    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    lib = q.load()
    r = Runner(torch, q, device)
    stream = r.stream
    name = args.case
    nt = 1
    path = q.PATH_AUTO
    if name.startswith("q4_k_prefill"):
        nt = int(name.split("N")[-1]) if "N" in name else 512
        base = "q4_k_prefill"
        if name.endswith("_gemv"):
            path = q.PATH_GEMV
    else:
        base = name
    if name.endswith("_backward_input"):
        return run_case_backward(args, torch, q, lib, r, name[:-len("_backward_input")])
    if "_experts_pos" in name:
        return run_case_experts(args, torch, q, lib, r, name)
    if "_pair" in name:
        return run_case_glu(args, torch, q, lib, r, name)
    if name in qmm_synth.AFFINE_WORKLOADS:
        return run_case_affine(args, torch, q, lib, r, name)
    fmt, k, n, w, x = qmm_synth.workload(base, n_tokens=nt)
    ncop = 1 if args.no_rotate else r.copies_for(w.size)
    wc = r.weights(w, ncop)
    xd = torch.from_numpy(x).to(device)
    yd = torch.empty((x.shape[0], n), device=device)
    a0 = q.make_args(fmt, wc[0], xd, yd, k, n, x.shape[0], path=path, stream=stream)
    need = q.qmm_workspace_bytes(a0)
    wsb = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    flags = 0 if args.no_overlap else (q.FLAG_OVERLAP_PREV | (0 if args.x_wait else q.FLAG_X_READY))
    al = [q.make_args(fmt, wc[c], xd, yd, k, n, x.shape[0], path=path,
                      workspace=wsb if need else None, workspace_bytes=need, stream=stream,
                      flags=flags)
          for c in range(ncop)]
    refs = [ctypes.byref(a) for a in al]

    def launch(c):
        if lib.qmm_matmul_ex(refs[c]):
            raise RuntimeError(q.qmm_last_error())
    with ClockSampler(0) as clk:
        dt = time_loop(torch, launch, args.steps, args.warmup, ncop, stream)
    q.qmm_device_status(stream)
    print(json.dumps({"case": name, "overlap": not args.no_overlap, "us_per_call": dt * 1e6, "weight_gbs": w.size / dt / 1e9,
                      "tflops": 2.0 * x.shape[0] * k * n / dt / 1e12, "copies": ncop,
                      "clocks": clk.summary()}), flush=True)
    return 0


def run_case_affine(args, torch, q, lib, r, name):
    """An affine workload alone (codes + bf16 scales and biases)."""
    import ctypes
    bits, k, n, w, sc, bi, x = qmm_synth.affine_workload(name)
    dev = r.dev
    nt = x.shape[0]
    total = w.size + sc.nbytes + bi.nbytes
    ncop = 1 if args.no_rotate else r.copies_for(total)
    wc = r.weights(w, ncop)
    sc_c = r.weights(sc.view(np.int16), ncop)
    bi_c = r.weights(bi.view(np.int16), ncop)
    xd = torch.from_numpy(x).to(dev)
    yd = torch.empty((nt, n), device=dev)
    fl = (q.FLAG_OVERLAP_PREV | q.FLAG_X_READY) if nt == 1 and not args.no_overlap else 0
    a0 = q.make_args(f"affine{bits}", wc[0], xd, yd, k, n, nt, stream=r.stream, flags=fl)
    need = q.qmm_workspace_bytes(a0)
    wsb = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    al = [q.make_args(f"affine{bits}", wc[c], xd, yd, k, n, nt, stream=r.stream, flags=fl,
                      workspace=wsb if need else None, workspace_bytes=need) for c in range(ncop)]
    refs = [(ctypes.byref(al[c]), ctypes.c_void_p(sc_c[c].data_ptr()),
             ctypes.c_void_p(bi_c[c].data_ptr())) for c in range(ncop)]

    def launch(c):
        if lib.qmm_matmul_affine(*refs[c]):
            raise RuntimeError(q.qmm_last_error())
    with ClockSampler(0) as clk:
        dt = time_loop(torch, launch, args.steps, args.warmup, ncop, r.stream)
    q.qmm_device_status(r.stream)
    print(json.dumps({"case": name, "us_per_call": dt * 1e6, "weight_gbs": total / dt / 1e9,
                      "tflops": 2.0 * nt * k * n / dt / 1e12, "copies": ncop,
                      "clocks": clk.summary()}), flush=True)
    return 0


def run_case_experts(args, torch, q, lib, r, name):
    """An expert workload at some positions: <workload>_pos<N>[_gemv|_grouped]."""
    import ctypes
    base, rest = name.split("_pos")
    parts = rest.split("_")
    n_pos = int(parts[0])
    path = {"gemv": q.PATH_GEMV, "grouped": q.PATH_MMA}.get(parts[1] if len(parts) > 1 else "",
                                                           q.PATH_AUTO)
    fmt, k, n, n_exp, w, x, ids = qmm_synth.expert_workload(base, n_pos=n_pos)
    dev, stream = r.dev, r.stream
    ncop = 1 if args.no_rotate else r.copies_for(w.size)
    wc = r.weights(w, ncop)
    xd = torch.from_numpy(x).to(dev)
    idd = torch.from_numpy(ids).to(dev)
    yd = torch.empty((ids.size, n), device=dev)
    al = [q.make_args(fmt, wc[c], xd, yd, k, n, n_pos, path=path, stream=stream)
          for c in range(ncop)]
    need = q.qmm_experts_workspace_bytes(al[0], n_exp, ids.shape[1])
    wsb = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if need:
        for a in al:
            a.workspace, a.workspace_bytes = wsb.data_ptr(), need
    refs = [ctypes.byref(a) for a in al]
    ip = ctypes.c_void_p(idd.data_ptr())

    def launch(c):
        if lib.qmm_matmul_experts(refs[c], ip, n_exp, ids.shape[1]):
            raise RuntimeError(q.qmm_last_error())
    dt = time_loop(torch, launch, args.steps, args.warmup, ncop, stream)
    q.qmm_device_status(stream)
    print(json.dumps({"case": name, "form": "grouped" if need else "gemv", "us_per_call": dt * 1e6,
                      "tflops": 2.0 * ids.size * k * n / dt / 1e12, "copies": ncop}), flush=True)
    return 0


def run_case_glu(args, torch, q, lib, r, name):
    """A gated pair: <gemv workload>_swiglu_pair / _geglu_pair (one token, the
    fused GEMV) or q4_k_swiglu_pair_N<tokens> (gate product, then the up
    product with the gated epilogue)."""
    import ctypes
    import re
    m = re.fullmatch(r"(\w+?)_(swiglu|geglu)_pair(?:_N(\d+))?", name)
    if not m:
        raise SystemExit(f"unknown gated-pair case {name}")
    act = q.ACT_SWIGLU if m.group(2) == "swiglu" else q.ACT_GEGLU
    nt = int(m.group(3)) if m.group(3) else 1
    if nt > 1:
        fmt, k, n, w, x = qmm_synth.workload("q4_k_prefill", n_tokens=nt)
        w2 = qmm_synth.gen_weights(fmt, k, n, np.random.default_rng(78))
    else:
        fmt, k, n, w, x = qmm_synth.workload(m.group(1) + "_gemv")
        w2 = qmm_synth.gen_weights(fmt, k, n, np.random.default_rng(77))
    dev, stream = r.dev, r.stream
    ncop = 1 if args.no_rotate else r.copies_for(2 * w.size)
    wg, wu = r.weights(w, ncop), r.weights(w2, ncop)
    xd = torch.from_numpy(x).to(dev)
    yd = torch.empty((nt, n), device=dev)
    flags = 0 if (args.no_overlap or nt > 1) else (q.FLAG_OVERLAP_PREV | q.FLAG_X_READY)
    al = [q.make_args(fmt, wg[c], xd, yd, k, n, nt, stream=stream, flags=flags) for c in range(ncop)]
    need = q.qmm_glu_workspace_bytes(al[0])
    wsb = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if need:
        for a in al:
            a.workspace, a.workspace_bytes = wsb.data_ptr(), need
    refs = [ctypes.byref(a) for a in al]
    ups = [ctypes.c_void_p(wu[c].data_ptr()) for c in range(ncop)]

    def launch(c):
        if lib.qmm_matmul_glu(refs[c], ups[c], act):
            raise RuntimeError(q.qmm_last_error())
    dt = time_loop(torch, launch, args.steps, args.warmup, ncop, stream)
    q.qmm_device_status(stream)
    print(json.dumps({"case": name, "us_per_call": dt * 1e6, "weight_gbs": 2 * w.size / dt / 1e9,
                      "tflops": 4.0 * nt * k * n / dt / 1e12, "copies": ncop}), flush=True)
    return 0


def run_case_backward(args, torch, q, lib, r, base):
    """dx = W^T dy over all rows of a workload's weights, timed alone."""
    import ctypes
    fmt, k, n, w, _ = qmm_synth.workload(base)
    dev = r.dev
    stream = r.stream
    ncop = 1 if args.no_rotate else r.copies_for(w.size)
    wc = r.weights(w, ncop)
    dyd = torch.from_numpy(np.random.default_rng(4).standard_normal(n).astype(np.float32)).to(dev)
    dxd = torch.empty(k, device=dev)
    flags = 0 if args.no_overlap else (q.FLAG_OVERLAP_PREV | q.FLAG_X_READY)
    al = [q.make_args(fmt, wc[c], dyd, dxd, k, n, 1, stream=stream, flags=flags)
          for c in range(ncop)]
    need = q.qmm_backward_input_workspace_bytes(al[0])
    wsb = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    for a in al:
        a.workspace, a.workspace_bytes = wsb.data_ptr(), need
    refs = [ctypes.byref(a) for a in al]

    def launch(c):
        if lib.qmm_matmul_backward_input(refs[c]):
            raise RuntimeError(q.qmm_last_error())
    dt = time_loop(torch, launch, args.steps, args.warmup, ncop, stream)
    q.qmm_device_status(stream)
    print(json.dumps({"case": args.case, "us_per_call": dt * 1e6, "weight_gbs": w.size / dt / 1e9,
                      "copies": ncop}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None,
                    help="profile one workload alone (bf16_gemv, f16_gemv, q4_0_gemv, q4_k_gemv, "
                         "q6_k_head, q4_k_prefill_N<tokens>[_gemv], <gemv workload>_backward_input, "
                         "<expert workload>_pos<N>[_gemv|_grouped], <format>_swiglu_pair, "
                         "<format>_geglu_pair, q4_k_swiglu_pair_N<tokens>)")
    ap.add_argument("--no-rotate", action="store_true")
    ap.add_argument("--x-wait", action="store_true",
                    help="overlap only the weight stream with the previous kernel (x read after it)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="plain stream-ordered launches (no programmatic dependent launch)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only (no other workloads, no CPU baseline)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
