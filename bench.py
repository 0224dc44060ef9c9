#!/usr/bin/env python
"""Benchmark of the quantized linear layer hot path on GB300.

One step = one pass of every hot-path step over one batch of synthetic input:
  1. W4A16 decode (T = 1) through a Llama-2-7B-shaped linear stack: 32 blocks
     x {q, k, v, o: 4096x4096; gate, up: 11008x4096; down: 4096x11008},
     224 fused dequant GEMVs over 3.4 GB of int4 weights (larger than L2, so
     every step streams the weights from HBM), launched with the block's
     dependency structure: q, k, v grouped in one launch on the block input,
     o on v's output, gate and up grouped on o's output, down on up's output
     (4 launches per block).
  2. W8A8 symmetric + bias (T=2048, K=4096, N=4096): per-token int8
     quantization of X, then the int8-exact GEMM with the fused epilogue.
  3. NVFP4 + ARCQuant (T=2048, K=4096, N=4096, S=128): NVFP4 quantization of X
     with residual channels, then the block-scaled fp4 GEMM over K_aug=4224.
Weights are quantized once at set-up (offline step, not timed); the NVFP4
per-tensor scale and channel order are calibrated once on X at set-up.

`value` is the W4A16 decode throughput in GB/s (algorithmic bytes of the 224
GEMVs / time of that phase); W8A8 and NVFP4 report TOPS (2 T N K / GEMM
time) in `paths`.  Each phase is a captured CUDA graph, timed with CUDA
events on its stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-linear HBM GB/s (W4A16 T=1) & TOPS (W8A8/NVFP4 T=2048) vs roofline"
LLAMA_BLOCK = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]
W8A8 = dict(T=2048, K=4096, N=4096)
NVFP4 = dict(T=2048, K=4096, N=4096, S=128)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "w4a16_decode_stack_traffic.txt")
W4A16_SOURCES = [os.path.join(ROOT, "quantized_linear_layer_gb300", "csrc", f)
                 for f in ("w4a16_gemv.cu", "w4a16_gemv_common.cuh")]


def w4a16_bytes(N, K, T):
    """Algorithmic HBM bytes of one W4A16 GEMV: packed codes, fp16 scales,
    packed zero-points, fp16 activations in and fp16 outputs out."""
    G = K // 128
    return N * K // 2 + N * G * 2 + N * ((G + 1) // 2) + 2 * T * K + 2 * T * N


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# our implementation
# --------------------------------------------------------------------------

class Workload:
    """Device-resident inputs, weights and outputs of one step, and the three
    captured phases."""

    def __init__(self, q, torch, layers, w4_path="launches"):
        from quantized_linear_layer_gb300 import inputs
        self.q, self.torch = q, torch
        dev = torch.device("cuda")
        self.stream = torch.cuda.Stream()
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        # 1. W4A16 stack (weights quantized on the device by the a0 kernel)
        protos = {}
        for (N, K) in sorted(set(LLAMA_BLOCK)):
            d = inputs.w4a16_decode(seed=1, T=1, N=N, K=K)
            protos[(N, K)] = (t(d["w"]), t(d["x"]))
        self.w4 = []
        for _ in range(layers):
            for (N, K) in LLAMA_BLOCK:
                wq = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
                sc = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
                zp = torch.empty((N, (K // 128 + 1) // 2), dtype=torch.uint8, device=dev)
                q.qlin_quant_w4_g128(protos[(N, K)][0], wq, sc, zp)
                self.w4.append((N, K, wq, sc, zp))
        # Activations, following a decoder block's dependencies: q, k and v
        # read the block input; o reads v's output (in place of the attention
        # output); gate and up read o's output; down reads up's output (in
        # place of act(gate) * up).  Every block starts again from the step's
        # input (the path has no normalisation between blocks).
        self.w4_in = protos[(4096, 4096)][1]
        self.w4_qkv = [torch.empty((1, 4096), dtype=torch.float16, device=dev) for _ in range(3)]
        self.w4_o = torch.empty((1, 4096), dtype=torch.float16, device=dev)
        self.w4_gate = torch.empty((1, 11008), dtype=torch.float16, device=dev)
        self.w4_up = torch.empty((1, 11008), dtype=torch.float16, device=dev)
        self.w4_out = torch.empty((1, 4096), dtype=torch.float16, device=dev)
        del protos
        self.w4_bytes = sum(w4a16_bytes(N, K, 1) for (N, K, *_r) in self.w4)
        # 2. W8A8 symmetric + bias
        d = inputs.w8a8_sym_bias(seed=2, **W8A8)
        T, K, N = W8A8["T"], W8A8["K"], W8A8["N"]
        self.w8_x = t(d["x"])
        w = t(d["w"])
        self.w8_b = torch.empty((N, K), dtype=torch.int8, device=dev)
        self.w8_sb = torch.empty(N, dtype=torch.float32, device=dev)
        q.qlin_quant_act_int8(w, self.w8_b, self.w8_sb)
        del w
        self.w8_bias = t(d["bias"])
        self.w8_a = torch.empty((T, K), dtype=torch.int8, device=dev)
        self.w8_sa = torch.empty(T, dtype=torch.float32, device=dev)
        self.w8_out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        # 3. NVFP4 + ARCQuant
        d = inputs.nvfp4_arc(seed=4, **{k: NVFP4[k] for k in ("T", "K", "N", "S")})
        T, K, N, S = NVFP4["T"], NVFP4["K"], NVFP4["N"], NVFP4["S"]
        self.nv_x = t(d["x"])
        w = t(d["w"])
        self.nv_gx = torch.empty(1, dtype=torch.float32, device=dev)
        self.nv_gw = torch.empty(1, dtype=torch.float32, device=dev)
        self.nv_perm = torch.empty(K, dtype=torch.int32, device=dev)
        q.qlin_nvfp4_global_scale(self.nv_x, self.nv_gx)     # calibration on X (set-up)
        q.qlin_arc_perm(self.nv_x, self.nv_perm)
        q.qlin_nvfp4_global_scale(w, self.nv_gw)
        self.nv_qw = torch.empty((N, (K + S) // 2), dtype=torch.uint8, device=dev)
        self.nv_sfw = torch.empty(q.qlin_nvfp4_sf_bytes(N, K + S, q.QLIN_SF_MMA), dtype=torch.uint8, device=dev)
        q.qlin_quant_nvfp4(w, self.nv_gw, self.nv_qw, self.nv_sfw, perm=self.nv_perm, S=S,
                           mode=q.QLIN_NVFP4_DUPLICATE, sf_layout=q.QLIN_SF_MMA)
        del w
        self.nv_qx = torch.empty((T, (K + S) // 2), dtype=torch.uint8, device=dev)
        self.nv_sfx = torch.empty(q.qlin_nvfp4_sf_bytes(T, K + S, q.QLIN_SF_MMA), dtype=torch.uint8, device=dev)
        self.nv_out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        self.w4_path = w4_path
        self.w4_seq_steps = self.w4a16_steps()
        self.w4_ws = torch.zeros(q.qlin_w4a16_sequence_workspace_bytes(len(self.w4_seq_steps)), dtype=torch.uint8,
                                 device=dev)
        # kernel launches per phase (the sequence: a workspace memset and one launch per 128 steps)
        n_seq = (len(self.w4_seq_steps) + 127) // 128
        self.launches = {"w4a16": n_seq if w4_path == "sequence" else 4 * layers, "w8a8": 2, "nvfp4": 2}

    # the three phases, as plain launch sequences on the current stream
    def w4a16_steps(self):
        """The decode stack as steps with the block's dependencies."""
        steps = []
        per_block = len(LLAMA_BLOCK)
        for b0 in range(0, len(self.w4), per_block):
            q, k, v, o, gate, up, down = self.w4[b0:b0 + per_block]
            steps.append((self.w4_in, [q[2], k[2], v[2]], [q[3], k[3], v[3]], [q[4], k[4], v[4]], self.w4_qkv))
            steps.append((self.w4_qkv[2], [o[2]], [o[3]], [o[4]], [self.w4_o]))
            steps.append((self.w4_o, [gate[2], up[2]], [gate[3], up[3]], [gate[4], up[4]], [self.w4_gate, self.w4_up]))
            steps.append((self.w4_up, [down[2]], [down[3]], [down[4]], [self.w4_out]))
        return steps

    def phase_w4a16(self):
        if self.w4_path == "sequence":
            # one persistent launch for the whole stack
            self.q.qlin_w4a16_gemv_sequence(self.w4_seq_steps, self.w4_ws)
            return
        for (x, wqs, scs, zps, ys) in self.w4_seq_steps:
            if len(wqs) == 1:
                self.q.qlin_w4a16_gemm(x, wqs[0], scs[0], zps[0], ys[0])
            else:
                self.q.qlin_w4a16_gemm_grouped(x, wqs, scs, zps, ys)

    def phase_w8a8(self):
        self.q.qlin_quant_act_int8(self.w8_x, self.w8_a, self.w8_sa)
        self.q.qlin_w8a8_gemm(self.w8_a, self.w8_b, self.w8_sa, self.w8_sb, self.w8_out, bias=self.w8_bias)

    def phase_nvfp4(self):
        self.q.qlin_quant_nvfp4(self.nv_x, self.nv_gx, self.nv_qx, self.nv_sfx, perm=self.nv_perm, S=NVFP4["S"],
                                sf_layout=self.q.QLIN_SF_MMA)
        self.q.qlin_nvfp4_gemm(self.nv_qx, self.nv_sfx, self.nv_qw, self.nv_sfw, self.nv_gx, self.nv_gw, self.nv_out)

    def capture(self):
        torch = self.torch
        self.graphs = {}
        with torch.cuda.stream(self.stream):
            for name, fn in (("w4a16", self.phase_w4a16), ("w8a8", self.phase_w8a8), ("nvfp4", self.phase_nvfp4)):
                fn()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    fn()
                self.graphs[name] = g
        torch.cuda.synchronize()


def max_over_ranks(dist, values, device=None):
    """Element-wise maximum of a list of floats over all ranks of the process
    group (the values themselves without one)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank, seconds, world):
    """Weak scaling: every rank processes the same units; the job's rate is
    all ranks' units over the slowest rank's time."""
    return units_per_rank * world / seconds


def kernel_timed_run(wl, torch, steps, warmup, dist):
    """Device-resident timing: per phase, the average over `steps` of the
    event-measured duration on the phase's stream."""
    names = ["w4a16", "w8a8", "nvfp4"]
    for _ in range(warmup):
        for n in names:
            wl.graphs[n].replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(wl.stream):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for s in range(steps):
            ev[s][0].record()
            for i, n in enumerate(names):
                wl.graphs[n].replay()
                ev[s][i + 1].record()
        t1.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total = t0.elapsed_time(t1) * 1e-3
    phase = {n: sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(steps)) * 1e-3 / steps
             for i, n in enumerate(names)}
    return total, phase


def e2e_run(wl, torch, steps, warmup):
    """End to end through the same calls with host buffers: every step copies
    its inputs from pinned host memory to the device and reads its results
    back; timed with events around the whole step on the same stream."""
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())  # noqa: E731
    h_in = {"w4a16": [pin(wl.w4_in)], "w8a8": [pin(wl.w8_x)], "nvfp4": [pin(wl.nv_x)]}
    d_in = {"w4a16": [wl.w4_in], "w8a8": [wl.w8_x], "nvfp4": [wl.nv_x]}
    d_out = {"w4a16": [wl.w4_out], "w8a8": [wl.w8_out], "nvfp4": [wl.nv_out]}
    h_out = {k: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in v] for k, v in d_out.items()}
    names = ["w4a16", "w8a8", "nvfp4"]
    h2d = sum(t.numel() * t.element_size() for v in h_in.values() for t in v)
    d2h = sum(t.numel() * t.element_size() for v in h_out.values() for t in v)

    def step(ev=None):
        for i, n in enumerate(names):
            for h, dv in zip(h_in[n], d_in[n]):
                dv.copy_(h, non_blocking=True)
            wl.graphs[n].replay()
            for dv, h in zip(d_out[n], h_out[n]):
                h.copy_(dv, non_blocking=True)
            if ev is not None:
                ev[i + 1].record()

    with torch.cuda.stream(wl.stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
        for s in range(steps):
            evs[s][0].record()
            step(evs[s])
    torch.cuda.synchronize()
    phase = {n: sum(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps)) * 1e-3 / steps
             for i, n in enumerate(names)}
    return phase, h2d, d2h


def w4a16_source_sha():
    """sha256 of the per-launch decode GEMV's source (kernel file + shared device code)."""
    h = hashlib.sha256()
    for f in W4A16_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def recorded_traffic():
    """Per-launch DRAM traffic of the W4A16 GEMV from the committed ncu
    summary, if it was taken on the current kernel source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    txt = open(PROFILE_TRAFFIC).read()
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", txt)
    b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not b:
        return None
    cur = w4a16_source_sha()
    return float(b.group(1)) if m.group(1) == cur else None


def cpu_baseline_sample(seconds=10.0):
    """The oracle, as it stands, on the host cores: W4A16 T=1 on the
    4096x4096 layer (dequantize to float64, one matrix-vector product),
    repeated for about `seconds`."""
    import oracle
    from quantized_linear_layer_gb300 import inputs
    d = inputs.w4a16_decode(seed=1, T=1, N=4096, K=4096)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    nbytes = w4a16_bytes(4096, 4096, 1)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.w4a16_reference(d["x"], codes, s16, z)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": nbytes * n / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "W4A16 T=1 on the 4096x4096 layer (float64 dequantize + matmul), %d calls in %.1f s; "
                      "numpy/BLAS threads on %d host cores" % (n, dt, cores)}


def run_ours(args):
    import torch
    import quantized_linear_layer_gb300 as q
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    q.build()
    q.lib()
    peaks = load_peaks()
    wl = Workload(q, torch, args.layers, args.w4a16_path)
    wl.capture()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    total, phase = kernel_timed_run(wl, torch, args.steps, args.warmup, dist)
    clocks = sampler.stop() if sampler else None
    err = q.qlin_get_device_error()
    # max over ranks of the timed region and of each phase
    total, tw4, tw8, tnv = max_over_ranks(dist, [total] + [phase[n] for n in ("w4a16", "w8a8", "nvfp4")],
                                          device="cuda")
    e2e_phase, h2d, d2h = e2e_run(wl, torch, max(3, args.steps // 5), 2)
    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return
    ms_per_step = total / args.steps * 1e3
    w4_gbs = whole_job_rate(wl.w4_bytes, tw4, world) / 1e9
    w8_ops = 2 * W8A8["T"] * W8A8["N"] * W8A8["K"]
    nv_ops = 2 * NVFP4["T"] * NVFP4["N"] * (NVFP4["K"] + NVFP4["S"])
    peak16 = peaks["bf16_tflops_sustained"]
    per_launch_bytes = wl.w4_bytes / wl.launches["w4a16"]
    per_launch_s = tw4 / wl.launches["w4a16"]
    traffic = recorded_traffic()
    line = {
        "metric": METRIC,
        "value": round(w4_gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u4xf16->f32 | s8(f16-exact)->s32 | e2m1xe4m3->f32",
        "data": "synthetic",
        "config": {
            "workload": "W4A16 T=1 decode over a Llama-2-7B-shaped linear stack (%d blocks x 7 layers with the "
                        "block's dependencies: q,k,v grouped on the block input, o on v, gate,up grouped on o, "
                        "down on up; 4 steps per block, %s) + "
                        "W8A8 sym+bias T=2048 K=4096 N=4096 + NVFP4 ARCQuant T=2048 K=4096 N=4096 S=128" %
                        (args.layers, "one persistent launch per 128 steps" if args.w4a16_path == "sequence"
                         else "one launch per step"),
            "w4a16_path": args.w4a16_path,
            "w4a16_launches_per_step": wl.launches["w4a16"],
            "w4a16_layers_per_step": len(wl.w4),
            "w4a16_weight_bytes_per_step": wl.w4_bytes,
            "l2": "inputs larger than L2: each step streams %.2f GB of W4A16 weights, which also evicts the "
                  "W8A8/NVFP4 operands between steps" % (wl.w4_bytes / 1e9),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "paths": {
            "w4a16": {"ms": round(tw4 * 1e3, 4), "GB/s": round(wl.w4_bytes / tw4 / 1e9, 1),
                      "frac_of_hbm": round(wl.w4_bytes / tw4 / 1e9 / peaks["hbm_gbs"], 4)},
            "w8a8": {"ms": round(tw8 * 1e3, 4), "TOPS_incl_quant": round(w8_ops / tw8 / 1e12, 1),
                     "frac_of_16bit_tensor_peak": round(w8_ops / tw8 / 1e12 / peak16, 4)},
            "nvfp4": {"ms": round(tnv * 1e3, 4), "TOPS_incl_quant": round(nv_ops / tnv / 1e12, 1),
                      "frac_of_fp4_tensor_peak": round(nv_ops / tnv / 1e12 / (peak16 * 6.0), 4)},
        },
        "roofline": {
            "kernel": ("w4a16_seq_kernel (persistent fused dequant GEMV sequence, T=1)" if args.w4a16_path == "sequence"
                       else "w4a16_gemv_kernel (fused dequant GEMV, T=1)"),
            "bound": "hbm",
            "achieved": round(per_launch_bytes / per_launch_s / 1e9, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(per_launch_bytes / per_launch_s / 1e9 / peaks["hbm_gbs"], 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": round(per_launch_bytes),
            "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured" else "fallback",
        },
        "e2e": {
            "value": round(wl.w4_bytes / e2e_phase["w4a16"] / 1e9 * world, 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(sum(e2e_phase.values()) * 1e3, 4),
        },
        "gpu_launches": sum(wl.launches.values()) * args.steps,
        "clocks": clocks,
        "device_error_word": err,
    }
    if world == 1:
        line["cpu_baseline"] = cpu_baseline_sample(args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# reference arm: the CPU oracle, as it stands
# --------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return  # the reference arm runs on rank 0 only
    import oracle
    from quantized_linear_layer_gb300 import inputs
    d = inputs.w4a16_decode(seed=1, T=1, N=4096, K=4096)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    nbytes = w4a16_bytes(4096, 4096, 1)
    for _ in range(args.warmup):
        oracle.w4a16_reference(d["x"], codes, s16, z)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.w4a16_reference(d["x"], codes, s16, z)
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": "W4A16 T=1 decode, bounded sample: one 4096x4096 layer per step of the "
                               "Llama-2-7B-shaped stack", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "one 4096x4096 W4A16 layer per step (float64 dequantize + matmul)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=32, help="transformer blocks in the W4A16 decode stack")
    ap.add_argument("--w4a16-path", choices=["sequence", "launches"], default="launches",
                    help="decode stack as one launch per step (grouped where layers share an input), or as one "
                         "persistent launch")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="length of the bounded oracle sample")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
