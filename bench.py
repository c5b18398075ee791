#!/usr/bin/env python3
"""Benchmark of the Q4_0 skinny MUL_MAT on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]

Workload (a "step"): the 7B-shaped single-token decode matvecs, M = 1, with Q4_0
weights of shapes [4096, 4096], [11008, 4096] and [4096, 11008] (N x K) and F32
activations: three gq_mul_mat_q4_0_f32 calls, each quantizing its activation row
to Q8_0 in-kernel and streaming the repacked weights once.  Weights ~ N(0, 0.02),
activations ~ N(0, 1), seeded, generated on the device (synthetic stand-ins for a
7B model; no checkpoint is read).  Each step uses the next of C weight copies, C
chosen so that the copies together exceed 4x the L2 cache: every timed step reads
its weights from HBM.

value  = weight-stream GB/s: algorithmic bytes (Q4_0 weights + f32 activations
         + f32 outputs) of all timed steps / device time of the timed steps.
e2e    = the same through the host-pointer entry point with pinned host
         buffers: each product copies its activations host->device, runs and
         copies its outputs back; the step synchronizes at its end.
extras = F16 weights on the same shapes, the M = 1..32 sweep, the prefill sizes
         (TFLOP/s) and the 32-layer 7B-shaped stack (tokens/s), each timed the
         same way (CUDA graph of back-to-back launches, rotating weight copies).

--impl reference times the CPU oracle (test infrastructure; plain C) on a
bounded sample of the same workload on the host cores.  Several GPUs run
independent replicas (the product has no data-path collective).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SHAPES = ((4096, 4096), (11008, 4096), (4096, 11008))
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0     # GB300 HBM3e, nominal
FALLBACK_BF16_TFLOPS = 1900.0


def q4_bytes(N, K):
    return N * K // 32 * 18


def step_bytes_q4(M, N, K):
    """Algorithmic bytes of one Q4_0 product: weights once, src1 once, dst once."""
    return q4_bytes(N, K) + 4 * M * K + 4 * M * N


def step_bytes_q8(M, N, K):
    return N * K * 34 // 32 + 4 * M * K + 4 * M * N


def step_bytes_q41(M, N, K):
    return N * K * 20 // 32 + 4 * M * K + 4 * M * N


def step_bytes_q5(M, N, K):
    return N * K * 22 // 32 + 4 * M * K + 4 * M * N


def step_bytes_f16(M, N, K):
    return 2 * N * K + 4 * M * K + 4 * M * N


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(t: float, dist) -> float:
    """The slowest rank's time: the whole job ends with it."""
    if not dist:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, t: float) -> float:
    """Replicas: every rank runs the full step, so the job moves world x the bytes in time t."""
    return bytes_per_step * steps * world / t / 1e9


# ----------------------------------------------------------------------------- env
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,utilization.gpu,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[2] > 0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded)}


# ----------------------------------------------------------------------------- GPU workload
class GpuBench:
    def __init__(self, device_index: int):
        import torch
        import quantized_skinny_matmul_gb300 as gq
        self.torch, self.gq = torch, gq
        self.dev = torch.device("cuda", device_index)
        torch.cuda.set_device(self.dev)
        self.props = torch.cuda.get_device_properties(self.dev)
        self.l2 = int(getattr(self.props, "L2_cache_size", 126 * 2 ** 20))
        self.stream = torch.cuda.Stream(self.dev)
        # size the stream's workspace for every shape before any graph capture
        gq.gq_reserve_workspace(512, 11008, 11008, stream=self.stream)
        # a decode loop never writes its weights after loading them
        gq.gq_set_static_weights(True)

    def smi_id(self):
        p = self.props
        try:
            return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except AttributeError:
            return str(self.dev.index)

    def gen(self, seed):
        g = self.torch.Generator(device=self.dev)
        g.manual_seed(seed)
        return g

    def q4_weights(self, N, K, seed):
        torch, gq = self.torch, self.gq
        w = torch.randn((N, K), generator=self.gen(seed), device=self.dev, dtype=torch.float32).mul_(0.02)
        q4 = gq.quantize_q4_0(w)
        del w
        rep = gq.repack_q4_0(q4, N, K)
        del q4
        return rep

    def q8_weights(self, N, K, seed):
        torch = self.torch
        gq = self.gq
        w = torch.randn((N, K), generator=self.gen(seed), device=self.dev, dtype=torch.float32).mul_(0.02)
        q8 = gq.quantize_rows_q8_0(w)
        del w
        return gq.repack_q8_0(q8, N, K)

    def q41_weights(self, N, K, seed):
        torch = self.torch
        gq = self.gq
        w = torch.randn((N, K), generator=self.gen(seed), device=self.dev, dtype=torch.float32).mul_(0.02)
        q41 = gq.quantize_q4_1(w)
        del w
        return gq.repack_q4_1(q41, N, K)

    def q5_weights(self, N, K, seed):
        torch = self.torch
        gq = self.gq
        w = torch.randn((N, K), generator=self.gen(seed), device=self.dev, dtype=torch.float32).mul_(0.02)
        q5 = gq.quantize_q5_0(w)
        del w
        return gq.repack_q5_0(q5, N, K)

    def f16_weights(self, N, K, seed):
        torch = self.torch
        w = torch.randn((N, K), generator=self.gen(seed), device=self.dev, dtype=torch.float32).mul_(0.02)
        return w.to(torch.float16)

    def acts(self, M, K, seed, outliers=False):
        torch = self.torch
        x = torch.randn((M, K), generator=self.gen(seed), device=self.dev, dtype=torch.float32)
        if outliers:
            n_out = int(round(0.01 * K))
            g = self.gen(seed + 1)
            for m in range(M):
                idx = torch.randperm(K, generator=g, device=self.dev)[:n_out]
                x[m, idx] *= 20.0
        return x

    def copies_for(self, bytes_per_set):
        return max(2, -(-4 * self.l2 // max(1, bytes_per_set)))

    def capture(self, launches):
        """A CUDA graph of the given launch closures, captured on self.stream."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            for fn in launches[: min(len(launches), 4)]:   # first calls outside capture (caches)
                fn()
        self.stream.synchronize()
        with torch.cuda.graph(g, stream=self.stream):
            for fn in launches:
                fn()
        return g

    def time_graph(self, g, reps=1):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(self.stream)
            for _ in range(reps):
                g.replay()
            end.record(self.stream)
        end.synchronize()
        return start.elapsed_time(end) / 1e3     # seconds

    def time_launches(self, launches, min_seconds=0.05, max_graph=3000):
        """Seconds per launch-list pass, from graphs of back-to-back passes."""
        per_graph = max(1, min(max_graph // max(1, len(launches)), 200))
        g = self.capture(launches * per_graph)
        self.time_graph(g, 2)                          # warm-up
        t1 = self.time_graph(g, 1)
        reps = max(1, min(200, int(min_seconds / max(t1, 1e-6))))
        t = self.time_graph(g, reps)
        del g
        return t / (reps * per_graph)


def run_ours(args, rank, world, local):
    import torch
    import quantized_skinny_matmul_gb300 as gq

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    b = GpuBench(local)
    hbm_peak, bf16_peak, bf16_sustained, peak_kind = measured_peaks()

    # ---- the step: three Q4_0 matvecs (M = 1) over C rotating weight copies
    M = 1
    set_bytes = sum(q4_bytes(N, K) for N, K in SHAPES)
    C = b.copies_for(set_bytes)
    weights = [[b.q4_weights(N, K, 1000 * c + i) for i, (N, K) in enumerate(SHAPES)] for c in range(C)]
    xs = [b.acts(M, K, 77 + i) for i, (N, K) in enumerate(SHAPES)]
    outs = [torch.empty((M, N), device=b.dev) for N, K in SHAPES]
    bytes_per_step = sum(step_bytes_q4(M, N, K) for N, K in SHAPES)
    launches_per_step = len(SHAPES)

    def step_launches(c):
        return [lambda i=i, N=N, K=K, c=c: gq.gq_mul_mat_q4_0_f32(weights[c][i], xs[i], outs[i], M, N, K)
                for i, (N, K) in enumerate(SHAPES)]

    graphs = {}

    def graph_of(n):              # a graph of n consecutive steps over the rotating copies
        if n not in graphs:
            ls = []
            for s in range(n):
                ls += step_launches(s % C)
            graphs[n] = b.capture(ls)
        return graphs[n]

    CHUNK = 1000

    def plan(n):                  # graphs that together run exactly n steps
        out = [graph_of(CHUNK)] * (n // CHUNK)
        if n % CHUNK:
            out.append(graph_of(n % CHUNK))
        return out

    warm_plan, timed_plan = plan(args.warmup), plan(args.steps)
    sampler = ClockSampler(b.smi_id()).start()
    for g in {id(g): g for g in timed_plan}.values():   # untimed: each timed graph's first replay
        b.time_graph(g, 1)
    soak_until = time.time() + 0.5          # untimed: let the clocks settle under load
    while time.time() < soak_until:
        for g in warm_plan:
            b.time_graph(g, 1)
    for g in warm_plan:                     # W untimed warm-up steps
        b.time_graph(g, 1)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(b.stream):
        # untimed pre-roll: the start event then waits behind W warm-up steps, long enough for
        # the host to submit the timed graphs, so the host latency of the first graph launch is
        # not inside the timed region (it would be ~3 % of a 20-step region)
        warm_plan[0].replay()
        start.record(b.stream)
        for g in timed_plan:              # exactly K timed steps
            g.replay()
        end.record(b.stream)
    end.synchronize()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    t = max_over_ranks(start.elapsed_time(end) / 1e3, dist)
    value = whole_job_gbs(bytes_per_step, args.steps, world, t)
    ms_per_step = t / args.steps * 1e3
    achieved = bytes_per_step * args.steps / t / 1e9          # per GPU, all launches of the one kernel family

    # ---- e2e: the same step through the host-pointer entry point with pinned host buffers:
    # each product copies its activations host->device, runs, and copies its outputs back
    hx = [xs[i].cpu().pin_memory() for i in range(len(SHAPES))]
    ho = [torch.empty((M, N), dtype=torch.float32).pin_memory() for N, K in SHAPES]
    e2e_steps = max(1, min(args.steps, 2000))
    wp = [[w.data_ptr() for w in ws] for ws in weights]
    hxp, hop = [h.data_ptr() for h in hx], [h.data_ptr() for h in ho]
    sp = b.stream.cuda_stream
    for s in range(3):
        for i, (N, K) in enumerate(SHAPES):
            gq.gq_mul_mat_q4_0_f32_host(wp[s % C][i], hxp[i], hop[i], M, N, K, sp)
        b.stream.synchronize()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    for h in ho:                       # the check below then sees what the timed steps wrote
        h.zero_()
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        for i, (N, K) in enumerate(SHAPES):
            gq.gq_mul_mat_q4_0_f32_host(wp[s % C][i], hxp[i], hop[i], M, N, K, sp)
        b.stream.synchronize()
    t_e2e = time.perf_counter() - t0
    last = (e2e_steps - 1) % C
    for i, (N, K) in enumerate(SHAPES):            # the host results are the device path's
        with torch.cuda.stream(b.stream):
            gq.gq_mul_mat_q4_0_f32(weights[last][i], xs[i], outs[i], M, N, K)
        b.stream.synchronize()
        if not torch.equal(ho[i], outs[i].cpu()):
            raise RuntimeError(f"e2e: host-buffer product {N}x{K} differs from the device product")
    t_e2e = max_over_ranks(t_e2e, dist)
    e2e = {"value": round(whole_job_gbs(bytes_per_step, e2e_steps, world, t_e2e), 3), "unit": "GB/s",
           "h2d_bytes_per_step": sum(4 * M * K for N, K in SHAPES),
           "d2h_bytes_per_step": sum(4 * M * N for N, K in SHAPES), "steps": e2e_steps}

    out = {
        "metric": "Q4_0 mul_mat weight-stream GB/s at M=1 (7B decode shapes)",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4xi8->f32", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
        "config": {"workload": "7B-shaped single-token decode matvecs, Q4_0 [4096,4096]+[11008,4096]+[4096,11008], M=1",
                   "M": M, "shapes_NxK": [list(s) for s in SHAPES], "weight_copies": C,
                   "l2_defeat": f"{C} rotating weight copies, {C * set_bytes / 2**20:.0f} MiB > 4x L2",
                   "timing": "CUDA events around CUDA-graph replays of exactly K steps; the start event "
                             "follows an untimed replay of warm-up steps on the same stream",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    traffic = profile_traffic()
    out["roofline"] = {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                       "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                       "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
                       "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                       "kernel": "gemv_m1_q4_0_kernel<16>", "launches": launches_per_step * args.steps,
                       "algorithmic_bytes_per_launch": round(bytes_per_step / launches_per_step)}

    # the integer-ALU ceiling of the same kernel: a dp4a throughput probe on this GPU, and the
    # dp4a rate the timed step needed (8 dp4a per 32-weight block: one block dot)
    out["roofline"]["alu"] = dp4a_roofline(b, sum(N * K // 32 * 8 for N, K in SHAPES) * args.steps / t)

    if rank == 0 and world == 1:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)

    if not args.no_extras:
        out["extras"] = extras(b, weights, C, hbm_peak, bf16_peak, bf16_sustained, args)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def dp4a_roofline(b, needed_per_s):
    """dp4a/s of a throughput probe (8 independent chains per thread, 8 CTAs of 256 per SM),
    and the fraction of it that `needed_per_s` dp4a/s is."""
    torch, gq = b.torch, b.gq
    blocks = 8 * b.props.multi_processor_count
    sink = torch.empty(blocks * 256, dtype=torch.int32, device=b.dev)
    iters = 20000
    with torch.cuda.stream(b.stream):
        for _ in range(2):
            gq.gq_debug_dp4a_probe(iters, sink, blocks, stream=b.stream)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(b.stream)
        for _ in range(5):
            gq.gq_debug_dp4a_probe(iters, sink, blocks, stream=b.stream)
        end.record(b.stream)
    end.synchronize()
    t = start.elapsed_time(end) / 1e3 / 5
    peak = blocks * 256 * 8 * iters / t
    return {"bound": "alu", "unit": "dp4a/s", "peak": float(f"{peak:.4g}"), "needed": float(f"{needed_per_s:.4g}"),
            "frac": round(needed_per_s / peak, 4),
            "peak_source": "measured: dp4a probe, 8 independent chains per thread, 8 x 256 threads per SM"}


def attn_bytes(lens, Hq, Hkv, D):
    """Algorithmic bytes of one decode attention over the INT8 cache: the K and V codes and
    scales of the valid tokens, the queries, the outputs and the lengths."""
    tokens = int(sum(int(t) for t in lens))
    B = len(lens)
    return tokens * Hkv * (2 * D + 8) + B * Hq * D * 8 + 4 * B


def attn_case(b, B, Hq, Hkv, Tcap, D, lens_mode, seed):
    import numpy as np
    from quantized_skinny_matmul_gb300 import synth
    torch = b.torch
    k, ks, v, vs = synth.kv_codes_device(seed, B, Hkv, Tcap, D, b.dev)
    q = torch.randn((B, Hq, D), generator=b.gen(seed + 1), device=b.dev, dtype=torch.float32)
    lens_h = synth.kv_lengths(seed + 2, B, Tcap, lens_mode)
    lens = torch.from_numpy(np.ascontiguousarray(lens_h)).to(b.dev)
    out = torch.empty((B, Hq, D), device=b.dev)
    return (q, k, ks, v, vs, lens, out), lens_h


def attn_extras(b, hbm_peak):
    """The INT8 KV-cache decode attention on the Llama2-7B layer of the KV-cache page (batch
    256, 32 heads of 128, 1024 + 1024 tokens): 4.4 GB per launch, far above L2."""
    from quantized_skinny_matmul_gb300 import synth
    gq = b.gq
    cfg = synth.KV_LLAMA2_7B
    B, Hq, Hkv, Tcap, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["Tcap"], cfg["D"]
    res = {}
    for mode in ("full", "mix"):
        (q, k, ks, v, vs, lens, out), lens_h = attn_case(b, B, Hq, Hkv, Tcap, D, mode, 90)
        fn = lambda: gq.gq_attn_decode_i8(q, k, ks, v, vs, lens, out, B, Hq, Hkv, Tcap, D, D ** -0.5,
                                          stream=b.stream)
        t = b.time_launches([fn], min_seconds=0.2, max_graph=20)
        nbytes = attn_bytes(lens_h, Hq, Hkv, D)
        gbs = nbytes / t / 1e9
        res[f"llama2_7b_b{B}_t{Tcap}_{mode}"] = {
            "us": round(t * 1e6, 1), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4),
            "algorithmic_bytes": nbytes, "tokens": int(lens_h.sum())}
        del q, k, ks, v, vs, lens, out
    # grouped queries (G = Hq / Hkv = 4 and 8) and one long sequence, full lengths
    for name, (B2, Hq2, Hkv2, T2) in (("g4_b64_t4096", (64, 32, 8, 4096)), ("g8_b128_t2048", (128, 32, 4, 2048)),
                                      ("g4_b1_t32768", (1, 32, 8, 32768))):
        (q, k, ks, v, vs, lens, out), lens_h = attn_case(b, B2, Hq2, Hkv2, T2, D, "full", 91)
        fn = lambda: gq.gq_attn_decode_i8(q, k, ks, v, vs, lens, out, B2, Hq2, Hkv2, T2, D, D ** -0.5,
                                          stream=b.stream)
        t = b.time_launches([fn], min_seconds=0.2, max_graph=50)
        nbytes = attn_bytes(lens_h, Hq2, Hkv2, D)
        res[name] = {"us": round(t * 1e6, 1), "GB/s": round(nbytes / t / 1e9, 1),
                     "frac_of_hbm": round(nbytes / t / 1e9 / hbm_peak, 4), "B": B2, "Hq": Hq2, "Hkv": Hkv2, "Tcap": T2}
        del q, k, ks, v, vs, lens, out
    b.torch.cuda.empty_cache()
    res["workload"] = (f"decode attention over an INT8 KV cache, B={B} Hq={Hq} Hkv={Hkv} D={D}, "
                       f"Tcap={Tcap}; lens full or uniform in [1, {Tcap}]; then grouped-query and long-context cases")
    return res


def extras(b, weights, C, hbm_peak, bf16_peak, bf16_sustained, args):
    import torch
    gq = b.gq
    res = {}
    res["attn_decode_i8"] = attn_extras(b, hbm_peak)
    # F16 weights, same shapes, M = 1
    f16_set = sum(2 * N * K for N, K in SHAPES)
    C16 = b.copies_for(f16_set)
    w16 = [[b.f16_weights(N, K, 5000 + 10 * c + i) for i, (N, K) in enumerate(SHAPES)] for c in range(C16)]
    xs = [b.acts(1, K, 300 + i) for i, (N, K) in enumerate(SHAPES)]
    os_ = [torch.empty((1, N), device=b.dev) for N, K in SHAPES]
    ls = []
    for c in range(C16):
        for i, (N, K) in enumerate(SHAPES):
            ls.append(lambda c=c, i=i, N=N, K=K: gq.gq_mul_mat_f16_f32(w16[c][i], xs[i], os_[i], 1, N, K))
    t = b.time_launches(ls)
    res["f16_m1"] = {"GB/s": round(sum(step_bytes_f16(1, N, K) for N, K in SHAPES) * C16 / t / 1e9, 1),
                     "frac_of_hbm": round(sum(step_bytes_f16(1, N, K) for N, K in SHAPES) * C16 / t / 1e9 / hbm_peak, 4)}
    # the same weights in the 16 x 32 tile layout (gq_repack_f16), M = 1 and M = 8
    r16 = [[gq.repack_f16(w) for w in ws] for ws in w16]
    del w16
    for M in (1, 8):
        xm = [b.acts(M, K, 320 + i) for i, (N, K) in enumerate(SHAPES)]
        om = [torch.empty((M, N), device=b.dev) for N, K in SHAPES]
        ls = [lambda c=c, i=i, N=N, K=K, M=M: gq.gq_mul_mat_f16r_f32(r16[c][i], xm[i], om[i], M, N, K)
              for c in range(C16) for i, (N, K) in enumerate(SHAPES)]
        t = b.time_launches(ls)
        gbs = sum(step_bytes_f16(M, N, K) for N, K in SHAPES) * C16 / t / 1e9
        res[f"f16r_m{M}"] = {"GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4),
                             "us_per_step": round(t / C16 * 1e6, 2)}
    del r16
    # Q8_0 weights (repacked tiles), same shapes, M = 1 and M = 8
    q8_set = sum(N * K * 34 // 32 for N, K in SHAPES)
    C8 = b.copies_for(q8_set)
    w8 = [[b.q8_weights(N, K, 7000 + 10 * c + i) for i, (N, K) in enumerate(SHAPES)] for c in range(C8)]
    for M in (1, 8):
        xm = [b.acts(M, K, 340 + i) for i, (N, K) in enumerate(SHAPES)]
        om = [torch.empty((M, N), device=b.dev) for N, K in SHAPES]
        ls = [lambda c=c, i=i, N=N, K=K, M=M: gq.gq_mul_mat_q8_0_f32(w8[c][i], xm[i], om[i], M, N, K)
              for c in range(C8) for i, (N, K) in enumerate(SHAPES)]
        t = b.time_launches(ls)
        gbs = sum(step_bytes_q8(M, N, K) for N, K in SHAPES) * C8 / t / 1e9
        res[f"q8_0_m{M}"] = {"GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4),
                             "us_per_step": round(t / C8 * 1e6, 2)}
    del w8
    # Q5_0 weights (repacked tiles), same shapes, M = 1
    C5 = b.copies_for(sum(N * K * 22 // 32 for N, K in SHAPES))
    w5 = [[b.q5_weights(N, K, 7500 + 10 * c + i) for i, (N, K) in enumerate(SHAPES)] for c in range(C5)]
    x1 = [b.acts(1, K, 360 + i) for i, (N, K) in enumerate(SHAPES)]
    o1 = [torch.empty((1, N), device=b.dev) for N, K in SHAPES]
    ls = [lambda c=c, i=i, N=N, K=K: gq.gq_mul_mat_q5_0_f32(w5[c][i], x1[i], o1[i], 1, N, K)
          for c in range(C5) for i, (N, K) in enumerate(SHAPES)]
    t = b.time_launches(ls)
    gbs = sum(step_bytes_q5(1, N, K) for N, K in SHAPES) * C5 / t / 1e9
    res["q5_0_m1"] = {"GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4), "us_per_step": round(t / C5 * 1e6, 2)}
    del w5
    # Q4_1 weights (repacked tiles), same shapes, M = 1
    C41 = b.copies_for(sum(N * K * 20 // 32 for N, K in SHAPES))
    w41 = [[b.q41_weights(N, K, 7700 + 10 * c + i) for i, (N, K) in enumerate(SHAPES)] for c in range(C41)]
    ls = [lambda c=c, i=i, N=N, K=K: gq.gq_mul_mat_q4_1_f32(w41[c][i], x1[i], o1[i], 1, N, K)
          for c in range(C41) for i, (N, K) in enumerate(SHAPES)]
    t = b.time_launches(ls)
    gbs = sum(step_bytes_q41(1, N, K) for N, K in SHAPES) * C41 / t / 1e9
    res["q4_1_m1"] = {"GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4), "us_per_step": round(t / C41 * 1e6, 2)}
    del w41
    # per-shape dispatch profiles (Q4_0): both families benched at M = 16..256; the smallest
    # benched M at which the tile family is faster, per shape
    disp = {}
    for i, (N, K) in enumerate(SHAPES):
        prof = gq.tune_dispatch(weights[0][i], N, K, Ms=(16, 32, 64, 128, 256), reps=10, install=False)
        cross = [M for M, tg, tt in zip(prof["M"], prof["gemv_us"], prof["tc_us"]) if tt < tg]
        disp[f"{N}x{K}"] = {"tile_faster_from_M": cross[0] if cross else None,
                            "gemv_us": [round(t, 2) for t in prof["gemv_us"]],
                            "tc_us": [round(t, 2) for t in prof["tc_us"]], "M": prof["M"]}
    res["dispatch_q4_0"] = disp

    # M sweep on the two FFN shapes (Q4_0)
    sweep = {}
    for i, (N, K) in ((1, SHAPES[1]), (2, SHAPES[2])):
        for M in (1, 2, 4, 8, 16, 32):
            x = b.acts(M, K, 400 + M)
            o = torch.empty((M, N), device=b.dev)
            ls = [lambda c=c, M=M, N=N, K=K, x=x, o=o, i=i: gq.gq_mul_mat_q4_0_f32(weights[c][i], x, o, M, N, K)
                  for c in range(C)]
            t = b.time_launches(ls) / C
            gbs = step_bytes_q4(M, N, K) / t / 1e9
            sweep[f"{N}x{K}_M{M}"] = {"us": round(t * 1e6, 3), "GB/s": round(gbs, 1),
                                      "frac_of_hbm": round(gbs / hbm_peak, 4),
                                      "TFLOP/s": round(2 * M * N * K / t / 1e12, 2)}
    res["sweep_q4_0"] = sweep

    # prefill-sized products (TFLOP/s)
    pre = {}
    for i, (N, K) in ((1, SHAPES[1]), (0, SHAPES[0])):
        for M in (64, 128, 512):
            x = b.acts(M, K, 500 + M, outliers=True)
            o = torch.empty((M, N), device=b.dev)
            ls = [lambda c=c, M=M, N=N, K=K, x=x, o=o, i=i: gq.gq_mul_mat_q4_0_f32(weights[c][i], x, o, M, N, K)
                  for c in range(C)]
            t = b.time_launches(ls, max_graph=200) / C
            tf = 2 * M * N * K / t / 1e12
            pre[f"{N}x{K}_M{M}"] = {"us": round(t * 1e6, 2), "TFLOP/s": round(tf, 2),
                                    "frac_of_bf16_burst": round(tf / bf16_peak, 4)}
    res["prefill_q4_0"] = pre

    # 32-layer 7B-shaped stack, one token pass = 224 products
    if not args.no_stack:
        from quantized_skinny_matmul_gb300 import synth
        layers = []
        for l in range(synth.N_LAYERS):
            layers.append([b.q4_weights(N, K, synth.stack_seed(l, p)) for p, (_, N, K) in enumerate(synth.LAYER_SHAPES)])
        stack_bytes = sum(q4_bytes(N, K) for _, N, K in synth.LAYER_SHAPES) * synth.N_LAYERS
        st = {"weight_bytes": stack_bytes}
        for M in (1, 8):
            # every product of every layer has its own activations (seeded per layer and product),
            # generated on the device before the timed graphs
            xs = [[b.acts(M, K, 100000 + synth.stack_seed(l, p)) for p, (_, N, K) in enumerate(synth.LAYER_SHAPES)]
                  for l in range(synth.N_LAYERS)]
            outs = {N: torch.empty((M, N), device=b.dev) for N in (4096, 11008)}
            ls = []
            for l in range(synth.N_LAYERS):
                for p, (_, N, K) in enumerate(synth.LAYER_SHAPES):
                    ls.append(lambda l=l, p=p, N=N, K=K, M=M, xs=xs, outs=outs:
                              gq.gq_mul_mat_q4_0_f32(layers[l][p], xs[l][p], outs[N], M, N, K))
            t = b.time_launches(ls, max_graph=len(ls))
            del xs
            st[f"M{M}"] = {"ms_per_token_pass": round(t * 1e3, 4), "tokens_per_s": round(M / t, 1),
                           "GB/s": round(stack_bytes / t / 1e9, 1), "frac_of_hbm": round(stack_bytes / t / 1e9 / hbm_peak, 4)}
        res["stack_32_layers"] = st

        # the same stack with the products that share an input fused by row concatenation:
        # Q|K|V (12288 x 4096) and gate|up (22016 x 4096): 4 products per layer instead of 7
        names = [n for n, _, _ in synth.LAYER_SHAPES]
        groups = [("attn_q", "attn_k", "attn_v"), ("attn_o",), ("ffn_gate", "ffn_up"), ("ffn_down",)]
        fused = []
        for l in range(synth.N_LAYERS):
            fl = []
            for grp in groups:
                idx = [names.index(g) for g in grp]
                Ns = [synth.LAYER_SHAPES[i][1] for i in idx]
                K = synth.LAYER_SHAPES[idx[0]][2]
                w = gq.concat_rows_q4_0([layers[l][i] for i in idx], Ns, K) if len(idx) > 1 else layers[l][idx[0]]
                fl.append((w, sum(Ns), K))
            fused.append(fl)
        del layers
        sf = {"weight_bytes": stack_bytes, "products_per_layer": len(groups)}
        for M in (1, 8):
            # one activation per fused product and layer (the products of a group share it)
            xs = [[b.acts(M, K, 200000 + synth.stack_seed(l, gi)) for gi, (w, N, K) in enumerate(fused[l])]
                  for l in range(synth.N_LAYERS)]
            outs = {N: torch.empty((M, N), device=b.dev) for _, N, _ in fused[0]}
            ls = []
            for l in range(synth.N_LAYERS):
                for gi, (w, N, K) in enumerate(fused[l]):
                    ls.append(lambda w=w, N=N, K=K, M=M, xs=xs, outs=outs, l=l, gi=gi:
                              gq.gq_mul_mat_q4_0_f32(w, xs[l][gi], outs[N], M, N, K))
            t = b.time_launches(ls, max_graph=len(ls))
            del xs
            sf[f"M{M}"] = {"ms_per_token_pass": round(t * 1e3, 4), "tokens_per_s": round(M / t, 1),
                           "GB/s": round(stack_bytes / t / 1e9, 1), "frac_of_hbm": round(stack_bytes / t / 1e9 / hbm_peak, 4)}
        res["stack_32_layers_fused_qkv_gate_up"] = sf
        del fused
    return res


def profile_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "gemv_m1_q4_0_decode.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    want = kernel_source_hash()
    traffic, src = None, None
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
        if line.startswith("kernel_source_sha256:"):
            src = line.split(":", 1)[1].strip()
    return traffic if (traffic is not None and src == want) else None


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemv_m1.cu", "gq_common.cuh"):
        with open(os.path.join(ROOT, "quantized_skinny_matmul_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- CPU oracle
def cpu_baseline(seconds: float):
    """The oracle as it stands, all host cores (rows of N split over threads), on a bounded sample."""
    import numpy as np
    import oracle
    o = oracle.get()
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    prepared = []
    for N, K in SHAPES:
        w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
        prepared.append((o.quantize_q4_0(w), rng.standard_normal((1, K), dtype=np.float32), N, K))

    with cf.ThreadPoolExecutor(cores) as ex:          # one pool for the whole sample
        def one_step():
            futs = []
            for q4, x, N, K in prepared:
                bounds = [(N * i // cores, N * (i + 1) // cores) for i in range(cores)]
                futs += [ex.submit(o.mul_mat_q4_0_f32, q4, x, b) for b in bounds]
            for f in futs:
                f.result()

        steps = 0
        t0 = time.perf_counter()
        while True:
            one_step()
            steps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    bytes_per_step = sum(step_bytes_q4(1, N, K) for N, K in SHAPES)
    return {"value": round(bytes_per_step * steps / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{steps} steps of the 3 decode matvecs (M=1), {el:.1f} s, rows of N split over {cores} threads"}


def run_profile(spec: str):
    """A few plain launches of one product, for ncu: KIND:M:N:K with KIND q4_0 | q4_1 | q5_0 | q8_0 | f16 | f16r |
    q4_0_tc | f16_tc; or attn_i8:B:Hq:Hkv:Tcap:D for the INT8 KV-cache decode attention (all lengths Tcap)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import quantized_skinny_matmul_gb300 as gq
    if spec.startswith("attn_i8:"):
        B, Hq, Hkv, Tcap, D = (int(v) for v in spec.split(":")[1:])
        b = GpuBench(0)
        (q, k, ks, v, vs, lens, out), _ = attn_case(b, B, Hq, Hkv, Tcap, D, "full", 90)
        for _ in range(5):
            gq.gq_attn_decode_i8(q, k, ks, v, vs, lens, out, B, Hq, Hkv, Tcap, D, D ** -0.5)
        torch.cuda.synchronize()
        print(f"profile {spec}: 5 launches done")
        return
    kind, M, N, K = spec.split(":")
    M, N, K = int(M), int(N), int(K)
    b = GpuBench(0)
    path = gq.GQ_PATH_TC if kind.endswith("_tc") else gq.GQ_PATH_AUTO
    x = b.acts(M, K, 1)
    o = torch.empty((M, N), device=b.dev)
    if kind.startswith("q4_0"):
        w = b.q4_weights(N, K, 2)
        fn = lambda: gq.gq_mul_mat_q4_0_f32_path(w, x, o, M, N, K, path)
    elif kind == "q4_1":
        w = b.q41_weights(N, K, 2)
        fn = lambda: gq.gq_mul_mat_q4_1_f32(w, x, o, M, N, K)
    elif kind == "q5_0":
        w = b.q5_weights(N, K, 2)
        fn = lambda: gq.gq_mul_mat_q5_0_f32(w, x, o, M, N, K)
    elif kind == "q8_0":
        w = b.q8_weights(N, K, 2)
        fn = lambda: gq.gq_mul_mat_q8_0_f32(w, x, o, M, N, K)
    elif kind == "f16r":
        w = gq.repack_f16(b.f16_weights(N, K, 2))
        fn = lambda: gq.gq_mul_mat_f16r_f32(w, x, o, M, N, K)
    else:
        w = b.f16_weights(N, K, 2)
        fn = lambda: gq.gq_mul_mat_f16_f32_path(w, x, o, M, N, K, path)
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    print(f"profile {spec}: 5 launches done")


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm (rank 0 only; other ranks exit without work).

    Runs exactly W untimed and K timed steps.  A step is the three decode products on a
    bounded, rotating sample of each product's rows, sized from one timed full step so
    that the whole run takes about a minute on the host cores.  The value is the
    algorithmic bytes of the sampled rows (their weights, the activation row, their
    outputs) per second.
    """
    if rank != 0:
        return
    import numpy as np
    import oracle
    oracle.build()
    o = oracle.get()
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    prepared = []
    for N, K in SHAPES:
        w = (rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02))
        prepared.append((o.quantize_q4_0(w), rng.standard_normal((1, K), dtype=np.float32), N, K))

    with cf.ThreadPoolExecutor(cores) as ex:
        def step(frac, k):
            """The three products on rows [r0, r0 + rows) of each (rotating with k); their bytes."""
            done, futs = 0, []
            for q4, x, N, K in prepared:
                rows = max(1, min(N, int(round(frac * N))))
                r0 = (k * rows) % N
                r1 = min(N, r0 + rows)
                bounds = [(r0 + (r1 - r0) * i // cores, r0 + (r1 - r0) * (i + 1) // cores) for i in range(cores)]
                futs += [ex.submit(o.mul_mat_q4_0_f32, q4, x, b) for b in bounds if b[1] > b[0]]
                done += (r1 - r0) * K * 18 // 32 + 4 * K + 4 * (r1 - r0)
            for f in futs:
                f.result()
            return done

        # calibration: a full step and a small one give the per-step overhead and the cost per
        # row fraction; the sample is sized so that W + K steps take about `budget` seconds
        def timed(frac):
            t = time.perf_counter()
            step(frac, 0)
            return time.perf_counter() - t
        f_small = min(1.0, 16.0 * cores / min(N for N, K in SHAPES))
        t_full, t_small = timed(1.0), min(timed(f_small) for _ in range(3))
        budget = 60.0
        per_step = budget / max(1, args.warmup + args.steps)
        slope = max(t_full - t_small, 1e-9) / max(1.0 - f_small, 1e-9)
        # at least 16 rows per thread and product: below that a step is thread-pool dispatch only
        frac = min(1.0, max(f_small, f_small + (per_step - t_small) / slope))
        for k in range(args.warmup):
            step(frac, k)
        total = 0
        t0 = time.perf_counter()
        for k in range(args.steps):
            total += step(frac, args.warmup + k)
        el = time.perf_counter() - t0
    v = round(total / el / 1e9, 4)
    sample = (f"{args.steps} timed steps after {args.warmup} warm-up steps; each step the 3 decode matvecs "
              f"(M=1) on {frac:.4f} of their rows (rotating), rows split over {cores} threads; {el:.1f} s")
    out = {"metric": "Q4_0 mul_mat weight-stream GB/s at M=1 (7B decode shapes)", "value": v, "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(el / args.steps * 1e3, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u4xi8->f64",
           "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
           "config": {"workload": "7B-shaped single-token decode matvecs, Q4_0 [4096,4096]+[11008,4096]+[4096,11008], M=1",
                      "M": 1, "shapes_NxK": [list(s) for s in SHAPES], "parallelism": "host threads"},
           "impl": "reference",
           "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
           "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--profile", metavar="KIND:M:N:K", help="only run 5 launches of one product (for ncu)")
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
