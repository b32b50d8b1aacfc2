#!/usr/bin/env python3
"""Benchmark of the low-M split-K bf16 GEMM on GB300.

One step = one GEMM C[M,N] = A[M,K] . W[N,K]^T (the whole hot path: TMA
stream, tcgen05 MMA, TMEM epilogue, cluster mailbox reduction, bf16 store).
The default workload is M=4, N=6144, K=4096, split_k=2 (96 clusters of 2
CTAs); a second, wide-N line (M=4, N=49152, K=4096, split_k=2) is measured in
the same run and reported under "wide_n".

Timing: W warm-up steps, then exactly K steps between two CUDA events on the
launching stream, replayed from CUDA graphs of back-to-back launches (PDL
edges kept).  Each launch reads the next of R copies of W whose total is more
than twice the L2 size, so every launch streams W from HBM.  The metric is
algorithmic bytes (N*K*2 + M*K*2 + M*N*2) per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, all host cores) on the same
workload, each step a bounded column sample of it.  Multi-GPU runs (torchrun)
are independent replicas, one per GPU, with no data exchange (weak scaling).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "HBM GB/s (% of GB300 peak) and us/GEMM, bf16 M=4 N=6144 K=4096 split-K"
UNIT = "GB/s"
WORKLOAD = dict(M=4, N=6144, K=4096, split_k=2)
WIDE = dict(M=4, N=49152, K=4096, split_k=2)
# name -> (M, N, K, split_k); split_k 0 lets the tactic table choose (the M sweep)
OTHER_CONFIGS = [
    ("M4 N2304 K12288 split_k 4", (4, 2304, 12288, 4)),
    ("M16 N6144 K32768 split_k 4", (16, 6144, 32768, 4)),
    ("M1 N6144 K4096 auto", (1, 6144, 4096, 0)),
    ("M2 N6144 K4096 auto", (2, 6144, 4096, 0)),
    ("M8 N6144 K4096 auto", (8, 6144, 4096, 0)),
    ("M16 N6144 K4096 auto", (16, 6144, 4096, 0)),
    ("M32 N6144 K4096 auto", (32, 6144, 4096, 0)),
    ("M64 N6144 K4096 auto", (64, 6144, 4096, 0)),
    ("M96 N6144 K4096 auto", (96, 6144, 4096, 0)),
    ("M128 N6144 K4096 auto", (128, 6144, 4096, 0)),
]
FALLBACK_HBM_GBS = 6800.0
KERNEL_NAME = "lowm_splitk_kernel"


def algo_bytes(M, N, K):
    return N * K * 2 + M * K * 2 + M * N * 2


def workload_name(w):
    return "lowm_gemm_bf16 M%d N%d K%d split_k %d" % (w["M"], w["N"], w["K"], w["split_k"])


# ------------------------------------------------------------------ environment
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_sha():
    """Fingerprint of the device code (the kernels and their PTX wrappers)."""
    h = hashlib.sha256()
    for rel in ("split_bf16_gemm_swap_gb300/csrc/lowm_kernel.cuh", "split_bf16_gemm_swap_gb300/csrc/lowm_persistent.cuh",
                "split_bf16_gemm_swap_gb300/csrc/ptx.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload, tactic):
    """DRAM bytes per launch from the committed ncu summary of this workload, if it
    was taken on the current device code with the same tile width and ring."""
    path = os.path.join(ROOT, "profiles", "lowm_splitk_kernel_m%d_n%d_k%d.md" % (
        workload["M"], workload["N"], workload["K"]))
    try:
        fields = {}
        for line in open(path):
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
        if fields.get("kernel_sources_sha256_16") != kernel_sources_sha():
            return None
        if fields.get("workload") != workload_name(workload):
            return None
        if fields.get("ring") != "%d x %d" % (tactic["kb_per_stage"], tactic["stages"]):
            return None
        if fields.get("tile_n") != str(tactic["tile_n"]):
            return None
        return int(fields["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if t0 <= ts <= t1 + 0.15:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def max_over_ranks(x: float) -> float:
    """Largest value of x over the ranks of the default process group (x itself without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(bytes_per_step: int, steps: int, world: int, secs_max: float) -> float:
    """GB/s over all replicas: every rank did `steps` GEMMs; the job took the slowest rank's time."""
    return world * bytes_per_step * steps / secs_max / 1e9


# ------------------------------------------------------------------ our arm
class GraphSet:
    """CUDA graphs of back-to-back launches that cycle through the W copies.

    graph(n, start) holds n launches reading W copies start, start + 1, ...
    (mod R), so that a sequence of replays keeps the rotation going across
    graph boundaries; each (n, start mod R) is captured once.
    """

    def __init__(self, lowm, A, Ws, C, w, stream):
        self.lowm, self.A, self.Ws, self.C, self.w, self.stream = lowm, A, Ws, C, w, stream
        self.cache = {}

    def graph(self, n, start):
        key = (n, start % len(self.Ws))
        g = self.cache.get(key)
        if g is None:
            M, N, K, sk = self.w["M"], self.w["N"], self.w["K"], self.w["split_k"]
            flags = self.w.get("flags", 0)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(n):
                    st = self.lowm.lowm_gemm_bf16_ex(self.A, self.Ws[(key[1] + i) % len(self.Ws)], self.C, M, N, K,
                                                     sk, flags, self.stream)
                    if st != 0:
                        raise RuntimeError("lowm_gemm_bf16 failed during capture: %s" % self.lowm.status_string(st))
            self.cache[key] = g
        return g

    def plan(self, launches, start, per_graph):
        """The graphs that replay `launches` launches from W copy `start`: full graphs, then one tail."""
        out, done = [], 0
        while done < launches:
            n = min(per_graph, launches - done)
            out.append(self.graph(n, start + done))
            done += n
        return out


PER_GRAPH = 100


def launch_plan_text(steps):
    q, r = divmod(steps, PER_GRAPH)
    parts = []
    if q:
        parts.append("%d graph%s of %d" % (q, "s" if q > 1 else "", PER_GRAPH))
    if r:
        parts.append("%d graph of %d" % (1, r))
    return ("%s PDL launches, replayed back to back after the warm-up graphs with no host synchronization "
            "between warm-up and timed region" % " + ".join(parts))


def time_device(lowm, w, steps, warmup, device, seed=1234, sampler=None):
    """Return (seconds for exactly `steps` GEMMs, clocks summary or None, W copies).

    The warm-up graphs, the start event, the timed graphs and the stop event
    are queued on one stream without a host synchronization in between, so
    the timed region starts on a busy GPU in steady state (a synchronization
    there would start it from an idle GPU and charge a cold graph launch to
    the first steps).  The device status word is read once, after the stop
    event: a wait that gave up anywhere in warm-up or timed steps fails the run.
    """
    from split_bf16_gemm_swap_gb300 import inputs
    M, N, K = w["M"], w["N"], w["K"]
    A, W = inputs.make_problem(M, N, K, seed=seed)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    wbytes = N * K * 2
    R = max(2, math.ceil(2 * l2 / wbytes) + 1)
    Ad = A.to(device)
    Wd = W.to(device)
    Ws = [Wd] + [Wd.clone() for _ in range(R - 1)]
    C = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device=device)
    torch.cuda.synchronize(device)
    gs = GraphSet(lowm, Ad, Ws, C, w, stream)
    ramp = [gs.graph(PER_GRAPH, i * PER_GRAPH) for i in range(R)]
    warm = gs.plan(warmup, 0, PER_GRAPH)
    timed = gs.plan(steps, warmup, PER_GRAPH)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        # Untimed clock ramp (an idle GPU sits at its lowest clock).
        t_ramp = time.time()
        while time.time() - t_ramp < 0.3:
            for g in ramp:
                g.replay()
            stream.synchronize()
        # One more round without a synchronization: the GPU is busy with it
        # while the host queues the warm-up and timed graphs, so the timed
        # region does not wait on the host's graph submissions.
        for g in ramp:
            g.replay()
        for g in warm:
            g.replay()
        e0.record(stream)
        for g in timed:
            g.replay()
        e1.record(stream)
    e1.synchronize()
    t1 = time.time()
    st, detail = lowm.lowm_gemm_sync_status(stream)
    if st != 0:
        raise RuntimeError("kernel status after the warm-up and timed steps: %s (bits %#x)" % (
            lowm.status_string(st), detail))
    secs = e0.elapsed_time(e1) / 1e3
    clocks = sampler.summary(t_ramp, t1) if sampler is not None else None
    if clocks is not None:
        clocks["window"] = ("clock ramp (0.3 s of the same launches) + warm-up + timed region: %.3f ms "
                            "(the timed region alone, %.3f ms, can be shorter than the 100 ms sampling period)" % (
                                (t1 - t_ramp) * 1e3, secs * 1e3))
    del gs, ramp, warm, timed
    return secs, clocks, R


def time_e2e(lowm, w, steps, device, seed=1234):
    """Through lowm_gemm_bf16_host: pinned host A, W in; C out; copies inside the timed region."""
    from split_bf16_gemm_swap_gb300 import inputs
    M, N, K, sk = w["M"], w["N"], w["K"], w["split_k"]
    A, W = inputs.make_problem(M, N, K, seed=seed)
    Ah, Wh = A.pin_memory(), W.pin_memory()
    Ch = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    Ad = torch.empty((M, K), dtype=torch.bfloat16, device=device)
    Wd = torch.empty((N, K), dtype=torch.bfloat16, device=device)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device=device)
    for _ in range(3):
        assert lowm.lowm_gemm_bf16_host(Ah, Wh, Ch, Ad, Wd, Cd, M, N, K, sk, stream) == 0
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for _ in range(steps):
        st = lowm.lowm_gemm_bf16_host(Ah, Wh, Ch, Ad, Wd, Cd, M, N, K, sk, stream)
        if st != 0:
            raise RuntimeError("lowm_gemm_bf16_host: %s" % lowm.status_string(st))
    secs = time.perf_counter() - t0
    return secs, M * K * 2 + N * K * 2, M * N * 2


def run_ours(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from split_bf16_gemm_swap_gb300 import lowm
    lowm.lib()
    # The W copies are never written by any kernel, so the promise of
    # LOWM_FLAG_W_BEFORE_PDL_WAIT holds; --default-launch measures the plain
    # lowm_gemm_bf16 path instead (also reported under "variants").
    w = dict(WORKLOAD, flags=0 if args.default_launch else lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    st, tactic = lowm.lowm_gemm_query_tactic_ex(w["M"], w["N"], w["K"], w["split_k"], w["flags"])
    assert st == 0, lowm.status_string(st)
    peak, peak_kind = measured_peak()
    bytes_per = algo_bytes(w["M"], w["N"], w["K"])

    with ClockSampler(local) as sampler:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        secs, clocks, R = time_device(lowm, w, args.steps, args.warmup, device, sampler=sampler)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
    my_secs = secs
    secs = max_over_ranks(secs)
    per_step = my_secs / args.steps
    achieved = bytes_per / per_step / 1e9                  # this rank's kernel, for the roofline
    value = whole_job_rate(bytes_per, args.steps, world, secs)

    # wide-N line (same protocol, fewer steps)
    wide_steps = max(200, min(args.steps, 2000))
    wide_w = dict(WIDE, flags=w["flags"])
    wsecs, _, wR = time_device(lowm, wide_w, wide_steps, max(args.warmup, 3), device)
    wbytes = algo_bytes(WIDE["M"], WIDE["N"], WIDE["K"])
    _, wtactic = lowm.lowm_gemm_query_tactic_ex(WIDE["M"], WIDE["N"], WIDE["K"], WIDE["split_k"], w["flags"])
    wide = {"workload": workload_name(WIDE), "us_per_gemm": wsecs / wide_steps * 1e6, "tactic": wtactic,
            "traffic": committed_traffic(WIDE, wtactic),
            "gbs": wbytes * wide_steps / wsecs / 1e9, "steps": wide_steps,
            "frac": wbytes * wide_steps / wsecs / 1e9 / peak, "l2": "rotating %d W copies" % wR}

    # The same workload through the other launch path (default flags <-> the
    # W-before-PDL-wait flag), same protocol.
    variants = {}
    vw = dict(w, flags=0 if w["flags"] else lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT)
    vsteps = min(args.steps, 50000)
    vsecs, _, _ = time_device(lowm, vw, vsteps, max(args.warmup, 3), device)
    variants["default_flags" if vw["flags"] == 0 else "w_before_pdl_wait"] = {
        "us_per_gemm": vsecs / vsteps * 1e6, "gbs": bytes_per * vsteps / vsecs / 1e9,
        "frac": bytes_per * vsteps / vsecs / 1e9 / peak, "steps": vsteps,
        "entry_point": "lowm_gemm_bf16_ex(flags=%d)" % vw["flags"]}
    # GEMMs that share their input (A is not written by the preceding kernel
    # either, as for projections of the same activations): both promises.
    both = lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT | lowm.LOWM_FLAG_A_BEFORE_PDL_WAIT
    aw = dict(w, flags=both)
    asecs, _, _ = time_device(lowm, aw, vsteps, max(args.warmup, 3), device)
    variants["w_and_a_before_pdl_wait"] = {
        "us_per_gemm": asecs / vsteps * 1e6, "gbs": bytes_per * vsteps / asecs / 1e9,
        "frac": bytes_per * vsteps / asecs / 1e9 / peak, "steps": vsteps,
        "entry_point": "lowm_gemm_bf16_ex(flags=%d)" % both}

    # The other configurations of the method's workloads (split-K reduction
    # width, long K, the M sweep, M above 64), same protocol and launch flags,
    # shorter runs: reported alongside the headline, not part of `value`.
    others = {}
    osteps = max(200, min(args.steps, 5000))
    for name, (M, N, K, sk) in OTHER_CONFIGS:
        ow = dict(M=M, N=N, K=K, split_k=sk, flags=w["flags"])
        _, otactic = lowm.lowm_gemm_query_tactic_ex(M, N, K, sk, w["flags"])
        steps_o = osteps if N * K <= 64 << 20 else max(200, osteps // 5)
        osecs, _, _ = time_device(lowm, ow, steps_o, max(args.warmup, 3), device)
        ob = algo_bytes(M, N, K)
        others[name] = {"us_per_gemm": osecs / steps_o * 1e6, "gbs": ob * steps_o / osecs / 1e9,
                        "frac": ob * steps_o / osecs / 1e9 / peak, "steps": steps_o,
                        "tile_n": otactic["tile_n"], "split_k": otactic["split_k"],
                        "ring": "%d x %d" % (otactic["kb_per_stage"], otactic["stages"]),
                        "traffic": committed_traffic(dict(M=M, N=N, K=K, split_k=otactic["split_k"]), otactic)}

    e2e_steps = max(5, min(args.steps, 50))
    esecs, h2d, d2h = time_e2e(lowm, w, e2e_steps, device)
    e2e = {"value": bytes_per * e2e_steps / esecs / 1e9 * world, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": e2e_steps, "us_per_gemm": esecs / e2e_steps * 1e6,
           "path": "lowm_gemm_bf16_host (pinned host buffers, copies + launch + sync per step)"}

    if rank != 0:
        return
    cpu = None if args.no_cpu_baseline else cpu_baseline(w, seconds=args.cpu_seconds)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "us_per_gemm": per_step * 1e6,
        "pct_of_peak": 100.0 * achieved / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(w), "M": w["M"], "N": w["N"], "K": w["K"], "split_k": w["split_k"],
                   "inputs": "A, W ~ N(0,1)/sqrt(K) rounded to bf16, seed 1234",
                   "l2": "inputs larger than L2: %d rotating W copies (%.0f MB)" % (R, R * w["N"] * w["K"] * 2 / 1e6),
                   "tactic": tactic, "launch": launch_plan_text(args.steps),
                   "entry_point": "lowm_gemm_bf16_ex(flags=%d)" % w["flags"],
                   "w_before_pdl_wait": bool(w["flags"]),
                   "w_before_pdl_wait_note": "W is never written by a kernel here, so the flag's promise holds",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind if peak_kind == "measured"
                     else "fallback 6800 GB/s", "kernel": KERNEL_NAME,
                     "algorithmic_bytes_per_launch": bytes_per, "traffic": committed_traffic(w, tactic),
                     # the same protocol on the method's other workloads, compact (us/GEMM, fraction of
                     # peak, ncu DRAM bytes per launch or null); the full records follow under
                     # "wide_n" and "other_configs"
                     "workloads": dict(
                         [(workload_name(WIDE), {"us": round(wide["us_per_gemm"], 3), "frac": round(wide["frac"], 4),
                                                 "traffic": wide["traffic"]})] +
                         [(name, {"us": round(o["us_per_gemm"], 3), "frac": round(o["frac"], 4),
                                  "traffic": o["traffic"]}) for name, o in others.items()])},
        "wide_n": wide,
        "variants": variants,
        "other_configs": others,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the oracle as the CPU baseline
def oracle_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seconds=10.0):
    """The CPU oracle on the full workload, repeated for about `seconds`."""
    import oracle
    from split_bf16_gemm_swap_gb300 import inputs
    M, N, K = w["M"], w["N"], w["K"]
    A, W = inputs.make_problem(M, N, K, seed=1234)
    a, b = inputs.bits(A), inputs.bits(W)
    nth = oracle_threads()
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.gemm_bf16_f64(a, b, nthreads=nth, want_sum=False)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": runs * algo_bytes(M, N, K) / el / 1e9, "unit": UNIT, "cores": nth, "kind": "oracle",
            "sample": "%d full M%d N%d K%d GEMMs (fp64 dot products, %d host threads), %.1f s" % (
                runs, M, N, K, nth, el)}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return                                          # rank 0 alone times the oracle
    import oracle
    from split_bf16_gemm_swap_gb300 import inputs
    oracle.build()
    w = dict(WORKLOAD)
    M, N, K = w["M"], w["N"], w["K"]
    A, W = inputs.make_problem(M, N, K, seed=1234)
    a, b = inputs.bits(A), inputs.bits(W)
    nth = oracle_threads()
    # Calibrate: cost of a 64-column slice, then size each step's column sample so
    # that warm-up + timed steps take about `budget` seconds.
    t0 = time.perf_counter()
    oracle.gemm_bf16_f64(a, b[:64], nthreads=nth, want_sum=False)
    per64 = max(time.perf_counter() - t0, 1e-6)
    budget = min(120.0, 4.0 * (args.steps + args.warmup))
    cols = int(budget / (args.steps + args.warmup) / per64) * 64
    cols = max(64, min(N, cols))
    bsample = b[:cols]
    for _ in range(args.warmup):
        oracle.gemm_bf16_f64(a, bsample, nthreads=nth, want_sum=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_bf16_f64(a, bsample, nthreads=nth, want_sum=False)
    secs = time.perf_counter() - t0
    step_bytes = algo_bytes(M, cols, K)
    value = step_bytes * args.steps / secs / 1e9
    sample = "%d of %d output columns of M%d N%d K%d per step (fp64 dot products, %d host threads)" % (
        cols, N, M, N, K, nth)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(w), "M": M, "N": N, "K": K, "split_k": w["split_k"],
                   "inputs": "A, W ~ N(0,1)/sqrt(K) rounded to bf16, seed 1234"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nth, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """Plain launches of the workload for ncu: `warmup` + `steps` GEMMs, rotating W copies, no graphs,
    through lowm_gemm_bf16_ex with the flags the benchmark times (W-before-PDL unless --default-launch)."""
    import __graft_entry__
    __graft_entry__.build()
    from split_bf16_gemm_swap_gb300 import inputs, lowm
    w = dict(WIDE if args.wide else WORKLOAD)
    if args.config:
        M, N, K, sk = dict(OTHER_CONFIGS)[args.config]
        w = dict(M=M, N=N, K=K, split_k=sk)
    M, N, K, sk = w["M"], w["N"], w["K"], w["split_k"]
    device = torch.device("cuda", 0)
    A, W = inputs.make_problem(M, N, K, seed=1234)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    R = max(2, math.ceil(2 * l2 / (N * K * 2)) + 1)
    Ad = A.to(device)
    Ws = [W.to(device) for _ in range(R)]
    C = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    torch.cuda.synchronize()
    flags = 0 if args.default_launch else lowm.LOWM_FLAG_W_BEFORE_PDL_WAIT   # the launch the bench times
    for i in range(args.warmup + args.steps):
        st = lowm.lowm_gemm_bf16_ex(Ad, Ws[i % R], C, M, N, K, sk, flags, None)
        assert st == 0, lowm.status_string(st)
    st, detail = lowm.lowm_gemm_sync_status()
    assert st == 0, "kernel status bits %#x" % detail
    print("profile case done: %s, %d launches, %d W copies" % (workload_name(w), args.warmup + args.steps, R))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--default-launch", action="store_true",
                    help="time lowm_gemm_bf16 without LOWM_FLAG_W_BEFORE_PDL_WAIT (the headline uses the flag: "
                         "the W copies are never written by a kernel)")
    ap.add_argument("--profile-only", action="store_true",
                    help="plain launches of the workload for a profiler (no timing, no JSON line)")
    ap.add_argument("--wide", action="store_true", help="with --profile-only: the wide-N workload")
    ap.add_argument("--config", default=None, choices=[name for name, _ in OTHER_CONFIGS],
                    help="with --profile-only: one of the other configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.steps < 1:
        raise SystemExit("--steps must be positive")
    if args.profile_only:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
