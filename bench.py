"""Benchmark of the block-quantized MatMulNBits hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mnb|reference] [--sweep]

Headline (one JSON line on rank 0): the decode call -- M = 1, K = N = 4096,
INT4 block-32 weights with explicit uint8 zero points and a rank-32 FP16 LoRA
adapter -- as weight-stream GB/s (every byte the call must move: packed codes,
scales, zero points, adapter A and B, X and Y) against the HBM roofline.  One
step = one mnb_run call (one decode launch: base and adapter fused).  The prefill call
(M = 1024, same K, N, default zero point, rank 32) is reported in the same line
as TFLOP/s against the dense FP16 tensor roofline.

Inputs are seeded synthetic data of those shapes.  Each step reads its own copy
of the weights, rotating over enough copies to exceed 4x the L2 size, so no
step finds its weights in L2.  K steps are captured in a CUDA graph; the graph
is replayed at least 10 times, each replay timed with CUDA events on the
replay stream, and the median replay gives the time per step.  SM clocks are
sampled with nvidia-smi over every timed leg.  `--impl reference` times the CPU oracle (the reference arm).
Under torchrun every rank runs an independent replica on its own GPU (the
operation has no exchange step); rank 0 prints the aggregate.
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

METRIC = "M=1 weight-stream GB/s vs HBM peak; M=1024 TFLOP/s vs FP16 tensor peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DECODE = dict(M=1, K=4096, N=4096, bits=4, rank=32)
PREFILL = dict(M=1024, K=4096, N=4096, bits=4, rank=32)


# ----------------------------------------------------------------------------- helpers

def decode_bytes(M, K, N, bits, rank, zp=True):
    nb = K // 32
    b = N * K * bits // 8 + N * nb * 2 + (N * nb if zp else 0)
    if rank:
        b += K * rank * 2 + N * rank * 2
    return b + M * K * 2 + M * N * 2


def prefill_flops(M, K, N, rank):
    return 2.0 * M * N * K + (2.0 * M * rank * (K + N) if rank else 0.0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            bf = d.get("bf16_tflops")
            if hbm and bf:
                return float(hbm), float(bf), float(d.get("bf16_tflops_sustained") or bf), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu capture, if the kernel sources
    are unchanged since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(kernel_key)
        if not d:
            return None
        if source_sha(d["sources"]) != d["source_sha"]:
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is busy."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

class Workload:
    """Rotating device copies of one seeded problem (weights, adapter, X, Y, T)."""

    def __init__(self, torch, mnb, synth, cfg, copies, seed_offset=0, zp=True):
        self.torch, self.mnb = torch, mnb
        self.cfg = cfg
        M, K, N, bits, rank = cfg["M"], cfg["K"], cfg["N"], cfg["bits"], cfg["rank"]
        inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=synth.SEED_BASE + 1 + seed_offset,
                                zp_range=(0, 15) if zp else None, rank=rank)
        self.inp = inp

        def dev(a):
            if a is None:
                return None
            if a.dtype == np.uint16:
                return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()
            return torch.from_numpy(np.ascontiguousarray(a)).cuda()

        base = dict(X=dev(inp.X), Wq=dev(inp.Wq), S=dev(inp.scales), Z=dev(inp.zp), A=dev(inp.A), B=dev(inp.B))
        self.copies = []
        for i in range(copies):
            c = {k: (None if v is None else v.clone()) for k, v in base.items()}
            c["Y"] = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
            c["T"] = torch.empty((M, rank), dtype=torch.float16, device="cuda") if rank else None
            self.copies.append(c)
        # decode loops keep the weights constant: let each call stream them early
        self.h = mnb.mnb_create(N, K, bits, 32, 32, 0, 0, mnb.FLAG_EARLY_WEIGHTS)

    def launches_per_call(self, sms, rank=None):
        """Kernels one call launches: the matmul kernel, plus the LoRA down kernel
        where the plan runs one."""
        rank = self.cfg["rank"] if rank is None else rank
        return 1 + self.mnb.mnb_plan(self.h, 1, self.cfg["M"], rank, sms)["lora_kernel"]

    def step(self, i, rank=None):
        c = self.copies[i % len(self.copies)]
        rank = self.cfg["rank"] if rank is None else rank
        self.mnb.mnb_run(self.h, c["X"], c["Wq"], c["S"], c["Z"], c["A"] if rank else None,
                         c["B"] if rank else None, rank, c["Y"], c["T"] if rank else None, 1, self.cfg["M"])

    def graph(self, start, n, rank=None):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step(start, rank)  # warm the capture stream once outside the graph
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(start, start + n):
                self.step(i, rank)
        return g

    def close(self):
        self.mnb.mnb_destroy(self.h)


def replay_median(torch, graphs, replays, barrier=None):
    """Replay the captured graphs round robin, `replays` times in all, each
    replay timed on its own with CUDA events on the replay stream, and return
    the median replay time in seconds.  A barrier and a device synchronize
    bracket the timed region."""
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    if barrier:
        barrier()
    torch.cuda.synchronize()
    for i in range(replays):
        ev[i][0].record(st)
        graphs[i % len(graphs)].replay()
        ev[i][1].record(st)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3


def timed_steps(torch, wl, steps, warmup, rank=None, chunk=1000, barrier=None, min_replays=10):
    """Warm up with `warmup` calls, then time K = `steps` calls per measurement:
    a CUDA graph of G = min(steps, chunk) consecutive calls is replayed
    R = max(min_replays, ceil(steps / G)) times, each replay timed on its own.
    Graphs start at different weight copies (as many as it takes to cover the
    rotation once), so a replay never finds the previous replay's weights in
    L2.  Returns (median seconds per call, R, G)."""
    G = max(1, min(chunk, steps))
    ncop = len(wl.copies)
    graphs = [wl.graph(j * G, G, rank) for j in range(max(1, min(8, math.ceil(ncop / G))))]
    for i in range(max(1, math.ceil(warmup / G))):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    R = max(min_replays, math.ceil(steps / G))
    return replay_median(torch, graphs, R, barrier) / G, R, G


def e2e_decode(torch, wl, steps, chunk=240, lanes=1, min_replays=10):
    """Through the public call with host buffers, every step: pinned X ->
    device, mnb_run, Y -> pinned host; the copies are real copies each step.
    lanes == 1: one request after another on one stream (the end-to-end
    latency of a call).  lanes > 1: consecutive steps are independent requests
    on `lanes` streams round robin (each step's copy-in, call and copy-out stay
    in order on its stream; each lane has its own host buffers), a serving
    loop's throughput.  Recorded in CUDA graphs of `chunk` steps, replayed
    max(min_replays, steps / chunk) times, each replay timed on its own.
    Returns (median seconds per step, h2d bytes per step, d2h bytes per step,
    replays, steps per replay)."""
    M, K, N = wl.cfg["M"], wl.cfg["K"], wl.cfg["N"]
    x_host = [torch.from_numpy(wl.inp.X.view(np.float16).copy()).pin_memory() for _ in range(lanes)]
    y_host = [torch.empty((1, M, N), dtype=torch.float16).pin_memory() for _ in range(lanes)]
    side = [torch.cuda.Stream() for _ in range(lanes)]

    def one(i, st):
        c = wl.copies[i % len(wl.copies)]
        with torch.cuda.stream(st):
            c["X"].copy_(x_host[i % lanes], non_blocking=True)
            wl.step(i)
            y_host[i % lanes].copy_(c["Y"], non_blocking=True)

    def record(start, n):
        main = torch.cuda.current_stream()
        for st in side:
            st.wait_stream(main)
        for i in range(start, start + n):
            one(i, side[i % lanes])
        for st in side:
            main.wait_stream(st)

    G = max(1, min(chunk, steps))
    warm = torch.cuda.Stream()
    warm.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(warm):
        record(0, lanes)
    torch.cuda.current_stream().wait_stream(warm)
    torch.cuda.synchronize()
    graphs = []
    for j in range(max(1, min(8, math.ceil(len(wl.copies) / G)))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            record(j * G, G)
        graphs.append(g)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    R = max(min_replays, math.ceil(steps / G))
    return replay_median(torch, graphs, R) / G, M * K * 2, M * N * 2, R, G


def measure_copy_gbs(torch, nbytes=1 << 30, reps=10):
    """Device-to-device copy bandwidth of one 1 GiB buffer (bytes read + bytes
    written, median of `reps` copies timed with CUDA events): the practical HBM
    ceiling on this device, reported next to the roofline's peak."""
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    for _ in range(3):
        dst.copy_(src)
    st = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(st)
        dst.copy_(src)
        e1.record(st)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    del src, dst
    torch.cuda.empty_cache()
    ts.sort()
    return 2.0 * nbytes / ts[len(ts) // 2] / 1e9


def run_gpu_arm(args, dist_ctx):
    import torch

    from block_quantized_matmul_matmulnbits_gb300 import mnb, synth

    rank_id, world, barrier, reduce_max = dist_ctx
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    mnb.lib()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20
    hbm_peak, bf16_peak, bf16_sus, peak_src = load_peaks()

    cfg = DECODE
    step_bytes = decode_bytes(cfg["M"], cfg["K"], cfg["N"], cfg["bits"], cfg["rank"])
    copies = max(8, math.ceil(4 * l2 / step_bytes))
    wl = Workload(torch, mnb, synth, cfg, copies)
    launches_per_step = wl.launches_per_call(props.multi_processor_count)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    only = args.only
    nan = float("nan")
    c_decode = c_base = c_e2e = c_e2e4 = nan  # seconds per call (median replay / calls per replay)
    rep_decode = rep_e2e = (0, 0)
    h2d = d2h = 0
    e2e_steps = min(args.steps, 2000)
    base_bytes = decode_bytes(cfg["M"], cfg["K"], cfg["N"], cfg["bits"], 0)
    if only in ("all", "decode"):
        c, R, G = timed_steps(torch, wl, args.steps, args.warmup, barrier=barrier)
        c_decode, rep_decode = reduce_max(c), (R, G)
    if only in ("all", "decode_base"):
        # the decode kernel alone (empty adapter), same rotation, for the per-kernel roofline
        c_base = reduce_max(timed_steps(torch, wl, args.steps, args.warmup, rank=0, barrier=barrier)[0])
    if only == "all":
        c, h2d, d2h, R, G = e2e_decode(torch, wl, e2e_steps, lanes=1)
        c_e2e, rep_e2e = reduce_max(c), (R, G)
        c_e2e4 = reduce_max(e2e_decode(torch, wl, e2e_steps, lanes=4)[0])
    wl.close()
    del wl
    torch.cuda.empty_cache()

    # prefill leg
    prefill = None
    try:
        if only not in ("all", "prefill"):
            raise RuntimeError(f"skipped (--only {only})")
        pc = PREFILL
        pbytes = decode_bytes(pc["M"], pc["K"], pc["N"], pc["bits"], pc["rank"], zp=False)
        pcopies = max(4, math.ceil(4 * l2 / pbytes))
        pwl = Workload(torch, mnb, synth, pc, pcopies, seed_offset=1, zp=False)
        psteps = max(10, min(args.steps // 20, 400))
        c_p, pR, pG = timed_steps(torch, pwl, psteps, max(3, args.warmup // 20), barrier=barrier)
        c_p = reduce_max(c_p)
        fl = prefill_flops(pc["M"], pc["K"], pc["N"], pc["rank"])
        tflops = fl / c_p / 1e12 * world
        per_tf = fl / c_p / 1e12
        prefill = {
            "value": round(tflops, 2), "unit": "TFLOP/s", "steps": psteps,
            "ms_per_step": round(c_p * 1e3, 4),
            "timing": f"median of {pR} graph replays of {pG} calls, each replay timed on its own",
            "config": {"workload": "prefill GEMM M=1024 K=4096 N=4096 INT4 block-32, default zero point 8, "
                                   "rank-32 FP16 LoRA epilogue", "M": 1024, "K": 4096, "N": 4096, "bits": 4,
                       "rank": 32, "l2": f"inputs larger than L2: {pcopies} rotating weight+X copies "
                                         f"({pcopies * pbytes / 2 ** 20:.0f} MiB vs {l2 / 2 ** 20:.0f} MiB L2)"},
            "roofline": {"bound": "tensor", "achieved": round(per_tf, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(per_tf / bf16_peak, 4), "traffic": ncu_traffic("gemm"),
                         "peak_source": f"{peak_src} bf16 burst (fp16 dense rate = bf16 rate)"},
        }
        pwl.close()
    except Exception as e:  # a prefill failure is reported in the line, not raised
        prefill = {"unavailable": f"{type(e).__name__}: {e}"[:200]}

    sampler.stop()  # the clocks cover every timed leg, prefill included
    clocks = sampler.summary()
    copy_gbs = measure_copy_gbs(torch) if only == "all" else None

    def rate(nbytes, steps, t):
        return nbytes * steps / t / 1e9 if t == t and t > 0 else None

    def rnd(x, n=2):
        return None if x is None else round(x, n)

    gbs = job_rate(step_bytes, 1, c_decode, world) / 1e9
    per_gbs = job_rate(step_bytes, 1, c_decode, 1) / 1e9
    base_gbs = base_bytes / c_base / 1e9
    e2e_gbs = step_bytes / c_e2e / 1e9 * world
    e2e4_gbs = step_bytes / c_e2e4 / 1e9 * world
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(c_decode * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded)",
        "config": {"workload": "decode GEMV M=1 K=4096 N=4096 INT4 block-32, explicit uint8 zero points, "
                               "rank-32 FP16 LoRA (A,B ~ N(0,0.02))", "M": 1, "K": 4096, "N": 4096, "bits": 4,
                   "rank": 32, "bytes_per_step": step_bytes, "flags": "MNB_FLAG_EARLY_WEIGHTS",
                   "l2": f"inputs larger than L2: {copies} rotating weight copies "
                         f"({copies * step_bytes / 2 ** 20:.0f} MiB vs {l2 / 2 ** 20:.0f} MiB L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": f"median of {rep_decode[0]} graph replays of {rep_decode[1]} calls, each replay "
                             f"timed on its own with CUDA events"},
        "roofline": {"bound": "hbm", "achieved": round(per_gbs, 2), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(per_gbs / hbm_peak, 4), "traffic": ncu_traffic("decode"),
                     "kernel": "single-token decode kernel (base and fused adapter in one launch), per mnb_run call",
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "copy_ceiling": None if copy_gbs is None else {
                         "value": round(copy_gbs, 1), "unit": "GB/s", "frac": round(per_gbs / copy_gbs, 4),
                         "method": "1 GiB device-to-device copy on this GPU, read + write bytes, median of 10"}},
        "decode_base_only": {"value": round(base_gbs, 2), "unit": "GB/s", "bytes_per_step": base_bytes,
                             "ms_per_step": round(c_base * 1e3, 6),
                             "frac": round(base_gbs / hbm_peak, 4), "traffic": ncu_traffic("decode_base")},
        "prefill": prefill,
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": rep_e2e[1], "ms_per_step": round(c_e2e * 1e3, 5),
                "path": "one request at a time on one stream: pinned X host->device, mnb_run, Y device->host "
                        f"every step; median of {rep_e2e[0]} replays of a CUDA graph of {rep_e2e[1]} steps"},
        "e2e_4lane": {"value": round(e2e4_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": round(c_e2e4 * 1e3, 5),
                      "path": "the same steps as independent requests on 4 streams round robin (serving "
                              "throughput, not a latency)"},
        "gpu_launches": launches_per_step * rep_decode[0] * rep_decode[1],
        "gpu_launches_note": f"this library's kernels launched in the timed decode region: {rep_decode[0]} "
                             f"replays x {rep_decode[1]} calls x {launches_per_step} launch per call",
        "clocks": clocks,
    }
    return line


# ----------------------------------------------------------------------------- sweep

SWEEP_M = (1, 2, 4, 8, 16, 64, 256, 1024, 4096)


def run_sweep(args):
    """The lm_head shapes and the M sweep at K=4096, N=14336 (INT4, default
    zero point, adapter on and off), every route, per-call time = median of 10
    replays of a graph of back-to-back calls over weight copies larger than 4x
    L2.  Reports the decode/prefill crossover."""
    import torch

    from block_quantized_matmul_matmulnbits_gb300 import mnb, synth

    torch.cuda.set_device(0)
    mnb.lib()
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20
    hbm_peak, bf16_peak, _, peak_src = load_peaks()

    def dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def measure(M, K, N, bits, rank, zp_range, scale_range, mode, seed):
        inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=seed, zp_range=zp_range,
                                scale_range=scale_range or (0.005, 0.02), rank=rank)
        nbytes = decode_bytes(M, K, N, bits, rank, zp=zp_range is not None)
        copies = max(2, min(64, math.ceil(4 * l2 / nbytes)))
        base = dict(X=dev(inp.X), Wq=dev(inp.Wq), S=dev(inp.scales), Z=dev(inp.zp), A=dev(inp.A), B=dev(inp.B))
        cps = [{k: (None if v is None else v.clone()) for k, v in base.items()} for _ in range(copies)]
        Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda") if rank else None
        h = mnb.mnb_create(N, K, bits, 32, 32, mode, 0, mnb.FLAG_EARLY_WEIGHTS)
        try:
            def call(i):
                c = cps[i % copies]
                mnb.mnb_run(h, c["X"], c["Wq"], c["S"], c["Z"], c["A"], c["B"], rank, Y, T, 1, M)
            n = max(4, min(200, int(2e-3 / max(1e-6, 2 * M * N * K / 1e15))))  # about 2 ms of calls per graph
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                call(0)
            torch.cuda.current_stream().wait_stream(st)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    call(i)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            times = []
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) * 1e3 / n)
            if mnb.mnb_sync_status(h) != mnb.MNB_OK:
                raise RuntimeError("device timeout")
            route = mnb.mnb_last_route(h)
        finally:
            mnb.mnb_destroy(h)
        us = float(np.median(times))
        fl = prefill_flops(M, K, N, rank)
        return {"us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1), "TFps": round(fl / us / 1e6, 2),
                "hbm_frac": round(nbytes / us / 1e3 / hbm_peak, 4), "tensor_frac": round(fl / us / 1e6 / bf16_peak, 4),
                "route": {1: "gemv", 2: "gemm"}.get(route, str(route))}

    rows = []

    def wanted(name):
        return args.sweep_filter is None or args.sweep_filter in name

    for name, (K, N, zpr, scr) in {"lm_head K=576 N=49152 INT8": (576, 49152, (120, 136), (0.001, 0.01)),
                                   "lm_head K=896 N=151936 INT8": (896, 151936, (120, 136), (0.001, 0.01))}.items():
        if not wanted(name):
            continue
        r = measure(1, K, N, 8, 0, zpr, scr, mnb.MODE_AUTO, synth.SEED_BASE + 4)
        rows.append({"workload": name, "M": 1, "rank": 0, "mode": "auto", **r})
        print(json.dumps(rows[-1]), flush=True)
    cross = {}
    ms = SWEEP_M if args.sweep_m is None else tuple(int(v) for v in args.sweep_m.split(","))
    ranks = (0, 32) if args.sweep_rank is None else (args.sweep_rank,)
    modes = tuple((m, r) for m, r in (("gemv", mnb.MODE_FORCE_GEMV), ("gemm", mnb.MODE_FORCE_GEMM))
                  if args.sweep_mode in (None, m))
    for rank in (ranks if wanted("K=4096 N=14336 INT4") else ()):
        for M in ms:
            res = {}
            for mname, mode in modes:
                if mname == "gemv" and M > 64:
                    continue  # the decode kernel re-reads the weights per 16 tokens
                res[mname] = measure(M, 4096, 14336, 4, rank, None, None, mode, synth.SEED_BASE + 5)
                rows.append({"workload": "K=4096 N=14336 INT4", "M": M, "rank": rank, "mode": mname, **res[mname]})
                print(json.dumps(rows[-1]), flush=True)
            if "gemv" in res and "gemm" in res and res["gemm"]["us"] < res["gemv"]["us"] and rank not in cross:
                cross[rank] = M
    summary = {"sweep": "lm_head + K=4096 N=14336 M sweep", "peaks": {"hbm_GBps": hbm_peak, "tensor_TFps": bf16_peak,
                                                                     "source": peak_src},
               "crossover_M_gemm_faster": cross, "rows": len(rows)}
    print(json.dumps(summary), flush=True)
    return 0


def run_next_rows(args):
    """The rows beyond the core path, timed like the sweep (a graph of
    back-to-back calls over input copies larger than 4x L2, median of 10
    replays): FP16 vs INT8 adapters, int8 activations, 2-bit weights, a bias,
    the fused QKV call against three separate calls, prefill with INT8
    adapters.  GB/s counts every input byte once plus the output."""
    import torch

    from block_quantized_matmul_matmulnbits_gb300 import mnb, synth

    torch.cuda.set_device(0)
    mnb.lib()
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", 129 * 2 ** 20) or 129 * 2 ** 20
    hbm_peak, bf16_peak, _, peak_src = load_peaks()

    def dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def nb(*arrays):
        return sum(int(a.nbytes) for a in arrays if a is not None)

    def timed(tensors, nbytes, enqueue, handles, calls_per_graph):
        """tensors: dict of device tensors (inputs), cloned into rotating copies;
        enqueue(copy, i) issues call i."""
        copies = max(2, min(64, math.ceil(4 * l2 / max(1, nbytes))))
        cps = [{k: (None if v is None else v.clone()) for k, v in tensors.items()} for _ in range(copies)]
        n = calls_per_graph
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            enqueue(cps[0], 0)
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                enqueue(cps[i % copies], i)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / n)
        for h in handles:
            if mnb.mnb_sync_status(h) != mnb.MNB_OK:
                raise RuntimeError("device timeout")
        return float(np.median(times))

    rows = []
    flt = getattr(args, "next_filter", None)

    def want(workload):
        return not flt or flt in workload

    def report(workload, us, nbytes, flops=0.0, **extra):
        r = {"workload": workload, "us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
             "hbm_frac": round(nbytes / us / 1e3 / hbm_peak, 4)}
        if flops:
            r["TFps"] = round(flops / us / 1e6, 2)
            r["tensor_frac"] = round(flops / us / 1e6 / bf16_peak, 4)
        r.update(extra)
        rows.append(r)
        print(json.dumps(r), flush=True)

    def single(M, K, N, bits, zp, adapter, q8x=False, bias=False, seed=synth.SEED_BASE + 6, calls=200):
        """adapter: None, 'fp16' or 'int8'."""
        inp = synth.make_inputs(M=M, K=K, N=N, bits=bits, seed=seed, zp_range=zp, rank=32 if adapter == "fp16" else 0)
        ql = synth.make_qlora(K=K, N=N, seed=seed) if adapter == "int8" else None
        bvec = synth.make_bias(N, seed=seed) if bias else None
        t = dict(X=dev(inp.X), Wq=dev(inp.Wq), S=dev(inp.scales), Z=dev(inp.zp), A=dev(inp.A), B=dev(inp.B),
                 bias=dev(bvec))
        if ql is not None:
            t.update(Aq=dev(ql.Aq), As=dev(ql.A_scales), Az=dev(ql.A_zp), Bq=dev(ql.Bq), Bs=dev(ql.B_scales),
                     Bz=dev(ql.B_zp))
        nbytes = nb(inp.X, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, bvec) + M * N * 2
        if ql is not None:
            nbytes += nb(ql.Aq, ql.A_scales, ql.A_zp, ql.Bq, ql.B_scales, ql.B_zp)
        Y = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
        T = torch.empty((M, 32), dtype=torch.float16, device="cuda") if adapter else None
        h = mnb.mnb_create(N, K, bits, 32, 32, mnb.MODE_AUTO, 0, mnb.FLAG_EARLY_WEIGHTS)
        try:
            def enqueue(c, i):
                if adapter == "int8":
                    mnb.mnb_run_qlora(h, c["X"], c["Wq"], c["S"], c["Z"], c["Aq"], c["As"], c["Az"], c["Bq"], c["Bs"],
                                      c["Bz"], 32, c["bias"], Y, T, 1, M)
                elif q8x:
                    mnb.mnb_run_q8x(h, c["X"], c["Wq"], c["S"], c["Z"], c["A"], c["B"], 32 if adapter else 0,
                                    c["bias"], Y, T, 1, M)
                else:
                    mnb.mnb_run_bias(h, c["X"], c["Wq"], c["S"], c["Z"], c["A"], c["B"], 32 if adapter else 0,
                                     c["bias"], Y, T, 1, M)
            us = timed(t, nbytes, enqueue, [h], calls)
            route = {1: "gemv", 2: "gemm"}.get(mnb.mnb_last_route(h), "?")
        finally:
            mnb.mnb_destroy(h)
        return us, nbytes, prefill_flops(M, K, N, 32 if adapter else 0), route

    K = 4096
    for name, kw in (("INT4 zp, no adapter", dict(adapter=None)),
                     ("INT4 zp, FP16 rank-32 adapter", dict(adapter="fp16")),
                     ("INT4 zp, INT8 rank-32 adapter", dict(adapter="int8")),
                     ("INT4 zp, bias, no adapter", dict(adapter=None, bias=True)),
                     ("INT4 zp, int8 activations, no adapter", dict(adapter=None, q8x=True)),
                     ("INT4 zp, int8 activations, FP16 adapter", dict(adapter="fp16", q8x=True))):
        if want(f"M=1 K=4096 N=4096 {name}"):
            us, nbytes, _, route = single(1, K, 4096, 4, (0, 15), **kw)
            report(f"M=1 K=4096 N=4096 {name}", us, nbytes, route=route)
    if want("M=1 K=4096 N=4096 INT2 zp, no adapter"):
        us, nbytes, _, route = single(1, K, 4096, 2, (0, 3), None)
        report("M=1 K=4096 N=4096 INT2 zp, no adapter", us, nbytes, route=route)
    for bits, q8x in ((4, False), (4, True), (2, False), (8, False)):
        name = f"M=1 K=4096 N=14336 INT{bits}{' int8 activations' if q8x else ''}"
        if want(name):
            us, nbytes, _, route = single(1, K, 14336, bits, None, None, q8x=q8x)
            report(name, us, nbytes, route=route)
    for M in (4, 16, 64):
        name = f"M={M} K=4096 N=14336 INT4 int8 activations"
        if want(name):
            us, nbytes, fl, route = single(M, K, 14336, 4, None, None, q8x=True, calls=100)
            report(name, us, nbytes, fl, route=route)
    # int8 activations at a prefill size, next to the FP16 tensor-core path on the same shape
    for q8x in (True, False):
        name = f"M=1024 K=4096 N=4096 INT4 {'int8' if q8x else 'FP16'} activations, no adapter"
        if want(name):
            us, nbytes, fl, route = single(1024, K, 4096, 4, None, None, q8x=q8x, seed=synth.SEED_BASE + 2, calls=10)
            report(name, us, nbytes, fl, route=route)
    for adapter in ("fp16", "int8"):
        name = f"M=1024 K=4096 N=4096 INT4, {adapter.upper()} rank-32 adapter"
        if want(name):
            us, nbytes, fl, route = single(1024, K, 4096, 4, None, adapter, seed=synth.SEED_BASE + 2, calls=20)
            report(name, us, nbytes, fl, route=route)

    # fused QKV (grouped-query shapes) against three separate calls
    for M in (1, 4):
        if not want(f"QKV M={M}"):
            continue
        Ns = (4096, 1024, 1024)
        inps = [synth.make_inputs(M=M, K=K, N=n, bits=4, seed=synth.SEED_BASE + 7 + i, zp_range=(0, 15))
                for i, n in enumerate(Ns)]
        t = {"X": dev(inps[0].X)}
        for i, inp in enumerate(inps):
            t.update({f"Wq{i}": dev(inp.Wq), f"S{i}": dev(inp.scales), f"Z{i}": dev(inp.zp)})
        Ys = [torch.empty((1, M, n), dtype=torch.float16, device="cuda") for n in Ns]
        nbytes = nb(inps[0].X, *[a for inp in inps for a in (inp.Wq, inp.scales, inp.zp)]) + M * sum(Ns) * 2
        hf = mnb.mnb_create(sum(Ns), K, 4, 32, 0, mnb.MODE_AUTO, 0, mnb.FLAG_EARLY_WEIGHTS)
        hs = [mnb.mnb_create(n, K, 4, 32, 0, mnb.MODE_AUTO, 0, mnb.FLAG_EARLY_WEIGHTS) for n in Ns]
        try:
            def fused(c, i):
                mnb.mnb_run_multi(hf, c["X"], [(n, c[f"Wq{j}"], c[f"S{j}"], c[f"Z{j}"], None, Ys[j])
                                               for j, n in enumerate(Ns)], 1, M)

            def separate(c, i):
                for j in range(3):
                    mnb.mnb_run(hs[j], c["X"], c[f"Wq{j}"], c[f"S{j}"], c[f"Z{j}"], None, None, 0, Ys[j], None, 1, M)
            us_f = timed(t, nbytes, fused, [hf], 200)
            us_s = timed(t, nbytes, separate, hs, 200)
        finally:
            mnb.mnb_destroy(hf)
            for h in hs:
                mnb.mnb_destroy(h)
        report(f"QKV M={M} K=4096 N=4096+1024+1024 INT4 zp, one mnb_run_multi", us_f, nbytes, launches=1)
        report(f"QKV M={M} K=4096 N=4096+1024+1024 INT4 zp, three mnb_run", us_s, nbytes, launches=3)
    print(json.dumps({"sweep": "rows beyond the core path", "peaks": {"hbm_GBps": hbm_peak, "tensor_TFps": bf16_peak,
                                                                     "source": peak_src}, "rows": len(rows)}),
          flush=True)
    return 0


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_decode_sample(target_s):
    import oracle
    from block_quantized_matmul_matmulnbits_gb300 import synth
    cfg = DECODE
    inp = synth.decode_4096(rank=cfg["rank"])
    step_bytes = decode_bytes(cfg["M"], cfg["K"], cfg["N"], cfg["bits"], cfg["rank"])
    oracle.run(inp.X2d, inp.Wq[:64], inp.scales[:64], inp.zp[:64], inp.A, inp.B[:64], 64, cfg["K"], 4)  # warm
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.run(inp.X2d, inp.Wq, inp.scales, inp.zp, inp.A, inp.B, cfg["N"], cfg["K"], cfg["bits"])
        n += 1
        dt = time.perf_counter() - t0
        if dt >= target_s:
            break
    return {"value": round(step_bytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"{n} full decode calls (M=1, K=N=4096, INT4, rank 32) in {dt:.1f} s"}, n, dt, step_bytes


def run_reference_arm(args):
    """The oracle as the reference arm: `warmup` then `steps` timed steps, each
    a bounded sample of the decode workload -- one oracle call on R of the
    4096 output rows (a decode call with N = R: the same X, adapter and K), R
    chosen so that the whole run takes about a minute of host time.  GB/s
    counts the sampled call's own bytes (R weight rows with their scales, zero
    points and B rows, plus X, A and the R outputs)."""
    import oracle
    from block_quantized_matmul_matmulnbits_gb300 import synth
    cfg = DECODE
    K, N = cfg["K"], cfg["N"]
    inp = synth.decode_4096(rank=cfg["rank"])
    row_bytes = inp.Wq[0].nbytes + inp.scales[0].nbytes + inp.zp[0].nbytes + inp.B[0].nbytes + 2
    fixed_bytes = inp.X.nbytes + inp.A.nbytes

    def call(r0, R):
        sl = slice(r0, r0 + R)
        oracle.run(inp.X2d, inp.Wq[sl], inp.scales[sl], inp.zp[sl], inp.A, inp.B[sl], R, K, cfg["bits"])

    call(0, 64)
    t0 = time.perf_counter()
    call(0, 256)
    per_row = max(1e-7, (time.perf_counter() - t0) / 256)
    per_step = min(2.0, 60.0 / max(1, args.steps + args.warmup))
    R = int(max(1, min(N, per_step / per_row)))
    starts = list(range(0, N - R + 1, R)) or [0]
    for i in range(args.warmup):
        call(starts[i % len(starts)], R)
    t0 = time.perf_counter()
    for i in range(args.steps):
        call(starts[i % len(starts)], R)
    dt = time.perf_counter() - t0
    step_bytes = R * row_bytes + fixed_bytes
    value = round(step_bytes * args.steps / dt / 1e9, 4)
    sample = (f"{args.steps} timed steps after {args.warmup} warm-up steps; each step one oracle call on {R} of "
              f"the {N} output rows (M=1, K={K}, INT4, zp, rank 32)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / max(1, args.steps) * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "decode GEMV M=1 K=4096 N=4096 INT4 block-32, explicit uint8 zero points, "
                               "rank-32 FP16 LoRA (A,B ~ N(0,0.02))", "M": 1, "K": K, "N": N, "bits": 4,
                   "rank": 32, "bytes_per_step": step_bytes, "rows_per_step": R},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- distribution

def job_rate(units_per_step, steps, t_max, world):
    """Whole-job throughput: every rank processes `steps` steps of its own
    replica (weak scaling), and the job takes the slowest rank's time."""
    return units_per_step * steps * world / t_max


def make_dist_ctx():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, None, (lambda x: x)
    import torch
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dist.init_process_group(backend=backend)
    dev = torch.device("cuda") if backend == "nccl" else torch.device("cpu")

    def barrier():
        dist.barrier()

    def reduce_max(x):
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return dist.get_rank(), world, barrier, reduce_max


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["mnb", "reference"], default="mnb")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["all", "decode", "decode_base", "prefill"], default="all",
                    help="run one leg only (for profiling); the printed line then lacks the other legs")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: the lm_head shapes and the M sweep at K=4096, N=14336 "
                         "(both routes), one JSON line per point")
    ap.add_argument("--sweep-filter", default=None,
                    help="with --sweep: only the workloads whose name contains this text")
    ap.add_argument("--sweep-m", default=None, help="with --sweep: only these M of the N=14336 sweep (comma list)")
    ap.add_argument("--sweep-rank", type=int, choices=[0, 32], default=None,
                    help="with --sweep: only this adapter rank of the N=14336 sweep")
    ap.add_argument("--sweep-mode", choices=["gemv", "gemm"], default=None,
                    help="with --sweep: only this route of the N=14336 sweep")
    ap.add_argument("--sweep-next", action="store_true",
                    help="instead of the bench line: the rows beyond the core path (adapter formats, int8 "
                         "activations, 2-bit weights, bias, fused QKV), one JSON line per point")
    ap.add_argument("--next-filter", default=None,
                    help="with --sweep-next: only the workloads whose name contains this text")
    args = ap.parse_args(argv)
    if args.sweep:
        return run_sweep(args)
    if args.sweep_next:
        return run_next_rows(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference_arm(args)), flush=True)
        return 0

    ctx = make_dist_ctx()
    line = run_gpu_arm(args, ctx)
    if ctx[0] == 0:
        if not args.no_cpu_baseline and ctx[1] == 1 and args.only == "all":
            line["cpu_baseline"] = oracle_decode_sample(args.cpu_seconds)[0]
        print(json.dumps(line), flush=True)
    if ctx[1] > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
