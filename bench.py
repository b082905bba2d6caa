"""Benchmark of the GGUF weight-only quantized linear layer on GB300.

One step = one decode pass over the linear layers of an 8B-class dense transformer layer:
Q4_K weights, M = 1 token, (K, N) in (4096, 4096), (4096, 1024), (4096, 12288), (12288, 4096)
-- four qlinear() calls. `value` is the whole job's algorithmic HBM throughput (quantized weight
bytes + fp16 activations + fp32 outputs) in GB/s, with inputs resident in HBM. The step
rotates over several copies of the weights (more than 2x the L2 size in total) so that no
step finds its weights in L2. The prefill figure (TFLOP/s of the Q4_K K=4096, N=12288, M=512
GEMM) and the dominant kernels' roofline fractions ride along in the same JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --case TYPE,K,N,M [--steps K] [--warmup W]   # one layer shape, for profilers
  python bench.py --table                                        # every layer shape, timed alone

--impl reference times the fp64 CPU oracle on this machine's cores (a deliberately slow
baseline) on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs an independent replica of the workload (the layer has
no exchange step); value sums the ranks' work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gguf_weight_only_gb300 import synth  # noqa: E402

DECODE_TYPE = 12
DECODE_M = 1
DECODE_SHAPES = synth.DECODE_8B_SHAPES                 # (K, N)
PREFILL = (12, 4096, 12288, 512)                       # type, K, N, M
METRIC = "qlinear weight GB/s (M=1) & TFLOP/s (M=512), % of HBM / FP16 roofline"
WORKLOAD = "Q4_K decode, 8B-class layer: M=1, (K,N) in (4096,4096),(4096,1024),(4096,12288),(12288,4096)"
Q6_K_A16 = 270   # Q6_K in 224-byte aligned blocks (made on the device by qlinear_repack)
BB = {**synth.BLOCK_BYTES, Q6_K_A16: 224}


def device_weights(t, N, K, seed, dev):
    """Seeded weights of type t on the device; the aligned Q6_K layout is made from Q6_K
    weights by the library's repack."""
    import torch
    if t != Q6_K_A16:
        return torch.from_numpy(synth.weights(t, N, K, seed)).to(dev)
    import gguf_weight_only_gb300 as ql
    W = ql.repack(torch.from_numpy(synth.weights(14, N, K, seed)).to(dev), 14, N, K)
    torch.cuda.synchronize(dev)
    return W


def alg_bytes(t, K, N, M):
    return N * (K // 256) * BB[t] + 2 * M * K + 4 * M * N


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# Translation units of the kernels whose ncu counters are committed: a counter stays valid
# while its own kernel's sources are unchanged.
KERNEL_SOURCES = {"gemv": ("gemv.cu", "decode.cuh", "ptx.cuh", "kernels.h"),
                  "gemm": ("gemm_tc.cu", "ptx.cuh", "kernels.h")}


def kernel_source_hash(kind=None):
    """Hash of a kernel's CUDA sources (all sources when kind is None) with comments and blank
    lines removed (a comment edit does not invalidate counters taken on the same code)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gguf_weight_only_gb300", "csrc")
    names = sorted(KERNEL_SOURCES[kind]) if kind else sorted(os.listdir(csrc))
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines()]
        h.update(name.encode())
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current sources of
    that kernel (key prefix gemv_ or gemm_)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    kind = kernel_key.split("_")[0]
    if d.get("source_hash", {}).get(kind) != kernel_source_hash(kind):
        return None
    v = d.get("kernels", {}).get(kernel_key)
    return None if v is None else float(v)


def max_over_ranks(ms, world, dev=None):
    """The slowest rank's time (all ranks must call it when world > 1)."""
    if world <= 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(step_bytes, ms_step, world):
    """Whole-job GB/s of `world` independent replicas, each moving step_bytes per step, timed
    by the slowest rank's ms per step (weak scaling: per-GPU work is fixed)."""
    return world * step_bytes / (ms_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 6:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[2 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch
    import gguf_weight_only_gb300 as ql
    from gguf_weight_only_gb300 import build

    if rank == 0:
        build.build()   # one build; the other ranks wait for it, then load the same library
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = ql.lib()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    hbm, tf_burst, tf_sust, peak_kind = peaks()

    # ---- inputs resident in HBM: P copies of the layer's weights, > 2x L2 in total
    layer_bytes = sum(N * (K // 256) * BB[DECODE_TYPE] for K, N in DECODE_SHAPES)
    P = max(2, int(np.ceil(2.2 * l2 / layer_bytes)))
    base = [torch.from_numpy(synth.weights(DECODE_TYPE, N, K, synth.workload_seed(1, i))).to(dev)
            for i, (K, N) in enumerate(DECODE_SHAPES)]
    copies = [[b.clone() for b in base] for _ in range(P)]
    xs = [torch.from_numpy(synth.activations(DECODE_M, K, synth.activation_seed(1, i, DECODE_M))).to(dev)
          for i, (K, N) in enumerate(DECODE_SHAPES)]
    ys = [torch.empty((DECODE_M, N), dtype=torch.float32, device=dev) for K, N in DECODE_SHAPES]
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    stream.wait_stream(torch.cuda.current_stream(dev))   # the clones above ran on the default stream

    def step(i):
        Ws = copies[i % P]
        for j, (K, N) in enumerate(DECODE_SHAPES):
            rc = lib.qlinear(DECODE_TYPE, Ws[j].data_ptr(), N, K, xs[j].data_ptr(), DECODE_M, ys[j].data_ptr(), sh)
            if rc != 0:
                raise RuntimeError(f"qlinear failed: {ql.strerror(rc)}")

    launches_per_step = sum(lib.qlinear_launch_count(DECODE_TYPE, N, K, DECODE_M) for K, N in DECODE_SHAPES)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    torch.cuda.synchronize(dev)

    # The timed steps run as replays of one CUDA graph holding `chunk` steps (a decode GEMV
    # is a few microseconds: launched one by one from Python the GPU would idle), chunk
    # dividing K so that exactly K steps are timed; one untimed replay first.
    chunk = next(d for d in range(min(args.steps, 200), 0, -1) if args.steps % d == 0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(chunk):
            step(i)
    # untimed replays for at least 50 ms, so that the timed region starts on warm clocks
    t_warm = time.perf_counter()
    while True:
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize(dev)
        if time.perf_counter() - t_warm >= 0.05:
            break
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        time.sleep(0.05)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps // chunk):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    step_bytes = sum(alg_bytes(DECODE_TYPE, K, N, DECODE_M) for K, N in DECODE_SHAPES)
    value = replica_throughput(step_bytes, ms_step, world)
    if ys[2].isnan().any():
        raise RuntimeError("NaN in output")
    del g

    # ---- dominant decode kernel alone: largest shape, CUDA-event time per launch
    def time_kernel(t, K, N, M, path_fn, reps):
        return time_shape(t, K, N, M, path_fn, reps, dev, stream, l2)

    Kd, Nd = DECODE_SHAPES[2]
    ms_dec = time_kernel(DECODE_TYPE, Kd, Nd, DECODE_M, lib.qlinear, 200)
    dec_bytes = alg_bytes(DECODE_TYPE, Kd, Nd, DECODE_M)
    dec_gbs = dec_bytes / (ms_dec * 1e-3) / 1e9
    t, Kp, Np, Mp = PREFILL
    ms_pre = time_kernel(t, Kp, Np, Mp, lib.qlinear, 40)
    pre_tf = 2.0 * Mp * Np * Kp / (ms_pre * 1e-3) / 1e12

    # ---- end to end through the public Python API with host buffers. As an engine would, a
    # step moves its four activation rows in one host->device copy (one pinned buffer, one
    # device buffer whose slices are the layer inputs) and its four outputs back in one
    # device->host copy, both by the library's copy call (a kernel reading and writing the
    # pinned buffers, chained to the layer calls by programmatic dependent launch); copies and
    # calls are captured once per weight copy as a CUDA graph, and every timed step replays one
    # on the engine's stream and waits for its result on the host.
    import gguf_weight_only_gb300 as qlp
    x_sizes = [DECODE_M * K for K, N in DECODE_SHAPES]
    y_sizes = [DECODE_M * N for K, N in DECODE_SHAPES]
    x_host = torch.cat([torch.from_numpy(synth.activations(DECODE_M, K, [9, i])).reshape(-1)
                        for i, (K, N) in enumerate(DECODE_SHAPES)]).pin_memory()
    y_host = torch.empty(sum(y_sizes), dtype=torch.float32).pin_memory()
    x_all = torch.empty(sum(x_sizes), dtype=torch.float16, device=dev)
    y_all = torch.empty(sum(y_sizes), dtype=torch.float32, device=dev)
    x_dev = [v.view(DECODE_M, K) for v, (K, N) in zip(torch.split(x_all, x_sizes), DECODE_SHAPES)]
    y_dev = [v.view(DECODE_M, N) for v, (K, N) in zip(torch.split(y_all, y_sizes), DECODE_SHAPES)]
    h2d = x_host.numel() * 2
    d2h = y_host.numel() * 4

    def e2e_body(i):
        Ws = copies[i % P]
        qlp.copy(x_all, x_host)
        for j, (K, N) in enumerate(DECODE_SHAPES):
            qlp.qlinear(Ws[j], DECODE_TYPE, N, K, x_dev[j], out=y_dev[j])
        qlp.copy(y_host, y_all)

    with torch.cuda.stream(stream):
        e2e_body(0)   # eager once: the library is loaded and every call checked
    torch.cuda.synchronize(dev)
    graphs = []
    for i in range(P):
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=stream):
            e2e_body(i)
        graphs.append(ge)

    def e2e_steps(first, n):
        for i in range(first, first + n):
            graphs[i % P].replay()
            stream.synchronize()

    with torch.cuda.stream(stream):   # the engine's stream, current for the whole run
        e2e_steps(0, 3)
        t0 = time.perf_counter()
        e2e_steps(3, args.steps)
        e2e_s = (time.perf_counter() - t0) / args.steps
    if not torch.isfinite(y_host).all():
        raise RuntimeError("non-finite end-to-end output")
    del graphs
    e2e_val = world * step_bytes / e2e_s / 1e9

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "accumulate": "f32",
        "data": "synthetic (seeded blocks and N(0,1) activations of the stated shapes)",
        "config": {"workload": WORKLOAD,
                   "weight_copies_rotated": P, "l2_bytes": l2,
                   "l2_policy": f"inputs larger than L2: {P} rotated weight copies, {P * layer_bytes / 1e6:.0f} MB",
                   "parallelism": f"replicas x{world}"},
        "prefill": {"workload": "Q4_K GEMM K=4096 N=12288 M=512", "ms": round(ms_pre, 4),
                    "tflops": round(pre_tf, 1), "peak_tflops": tf_burst, "frac": round(pre_tf / tf_burst, 4),
                    "bound": "tensor"},
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel<12> K=4096 N=12288 M=1",
                     "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(dec_gbs / hbm, 4), "peak_kind": peak_kind,
                     "traffic": ncu_traffic("gemv_q4k_k4096_n12288_m1")},
        "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    return result



def time_shape(t, K, N, M, path_fn, reps, dev, stream, l2, replays=3):
    """CUDA-event time (ms) of one launch of a layer shape: a CUDA graph of `reps` back-to-back
    calls over rotated weight copies (more than 2.2x L2 in total, so weights come from HBM),
    replayed `replays` times after one untimed replay; the median per-launch time."""
    import torch
    wb = N * (K // 256) * BB[t]
    Pk = max(2, int(np.ceil(2.2 * l2 / wb)))
    W0 = device_weights(t, N, K, [7, t, K, N], dev)
    Wk = [W0.clone() for _ in range(Pk)]
    x = torch.from_numpy(synth.activations(M, K, [8, t, M])).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    stream.wait_stream(torch.cuda.current_stream(dev))   # weight copies and inputs made on the default stream
    with torch.cuda.stream(stream):
        for i in range(3):
            path_fn(t, Wk[i % Pk].data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), sh)
    torch.cuda.synchronize(dev)
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=stream):
        for i in range(reps):
            path_fn(t, Wk[i % Pk].data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), sh)
    with torch.cuda.stream(stream):
        gk.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(replays):
        with torch.cuda.stream(stream):
            e0.record(stream)
            gk.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1) / reps)
    if y.isnan().any():
        raise RuntimeError("NaN in output")
    del gk, Wk
    torch.cuda.empty_cache()
    return float(np.median(times))


def time_multi(t, K, Ns, M, reps, dev, stream, l2, lib, fused=True, replays=5):
    """As time_shape, for projections sharing x: one qlinear_multi call per repetition (fused)
    or one qlinear call per projection (separate). Returns ms per repetition."""
    import ctypes
    import torch
    wb = sum(N * (K // 256) * BB[t] for N in Ns)
    Pk = max(2, int(np.ceil(2.2 * l2 / wb)))
    W0 = [torch.from_numpy(synth.weights(t, N, K, [7, t, K, N, j])).to(dev) for j, N in enumerate(Ns)]
    Wk = [[w.clone() for w in W0] for _ in range(Pk)]
    x = torch.from_numpy(synth.activations(M, K, [8, t, M])).to(dev)
    ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for N in Ns]
    sh = stream.cuda_stream
    stream.wait_stream(torch.cuda.current_stream(dev))   # weight copies and inputs made on the default stream
    n = len(Ns)
    n_arr = (ctypes.c_int64 * n)(*Ns)
    y_arr = (ctypes.c_void_p * n)(*[y.data_ptr() for y in ys])
    w_arrs = [(ctypes.c_void_p * n)(*[w.data_ptr() for w in Ws]) for Ws in Wk]

    def call(i):
        if fused:
            rc = lib.qlinear_multi(t, n, w_arrs[i % Pk], n_arr, K, x.data_ptr(), M, y_arr, sh)
            if rc != 0:
                raise RuntimeError(f"qlinear_multi failed: {rc}")
        else:
            for j, N in enumerate(Ns):
                rc = lib.qlinear(t, Wk[i % Pk][j].data_ptr(), N, K, x.data_ptr(), M, ys[j].data_ptr(), sh)
                if rc != 0:
                    raise RuntimeError(f"qlinear failed: {rc}")

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    torch.cuda.synchronize(dev)
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=stream):
        for i in range(reps):
            call(i)
    with torch.cuda.stream(stream):
        gk.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(replays):
        with torch.cuda.stream(stream):
            e0.record(stream)
            gk.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1) / reps)
    if any(y.isnan().any() for y in ys):
        raise RuntimeError("NaN in output")
    del gk, Wk
    torch.cuda.empty_cache()
    return float(np.median(times))


def time_fused(kind, t, K, N, M, reps, dev, stream, l2, lib, replays=5):
    """As time_shape, for a decode call with a fused prologue ("silu": x = silu(gate) * up;
    "rmsnorm": x = rmsnorm(h) * w) and a residual added in place. Returns ms per call."""
    import torch
    wb = N * (K // 256) * BB[t]
    Pk = max(2, int(np.ceil(2.2 * l2 / wb)))
    W0 = device_weights(t, N, K, [7, t, K, N], dev)
    Wk = [W0.clone() for _ in range(Pk)]
    rng = np.random.default_rng([9, t, K, N, M])
    a = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float16 if kind == "silu" else np.float32)).to(dev)
    b = torch.from_numpy(rng.standard_normal((M, K) if kind == "silu" else (K,)).astype(np.float32)).to(dev)
    y = torch.zeros((M, N), dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    stream.wait_stream(torch.cuda.current_stream(dev))   # weight copies and inputs made on the default stream

    def call(i):
        if kind == "silu":
            rc = lib.qlinear_silu_mul(t, Wk[i % Pk].data_ptr(), N, K, a.data_ptr(), b.data_ptr(), M, y.data_ptr(),
                                      y.data_ptr(), sh)
        else:
            rc = lib.qlinear_rmsnorm(t, Wk[i % Pk].data_ptr(), N, K, a.data_ptr(), b.data_ptr(), 1e-6, M, y.data_ptr(),
                                     y.data_ptr(), None, sh)
        if rc != 0:
            raise RuntimeError(f"fused {kind} failed: {rc}")

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    torch.cuda.synchronize(dev)
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=stream):
        for i in range(reps):
            call(i)
    with torch.cuda.stream(stream):
        gk.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(replays):
        with torch.cuda.stream(stream):
            e0.record(stream)
            gk.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1) / reps)
    del gk, Wk
    torch.cuda.empty_cache()
    return float(np.median(times))


def time_argmax(t, K, N, M, reps, dev, stream, l2, lib, replays=5):
    """As time_shape, for the greedy head (qlinear_argmax: a memset and two kernels per call).
    Returns ms per call."""
    import torch
    wb = N * (K // 256) * BB[t]
    Pk = max(2, int(np.ceil(2.2 * l2 / wb)))
    W0 = device_weights(t, N, K, [7, t, K, N], dev)
    Wk = [W0.clone() for _ in range(Pk)]
    x = torch.from_numpy(synth.activations(M, K, [8, t, M])).to(dev)
    idx = torch.empty(M, dtype=torch.int64, device=dev)
    val = torch.empty(M, dtype=torch.float32, device=dev)
    sh = stream.cuda_stream
    stream.wait_stream(torch.cuda.current_stream(dev))   # weight copies and inputs made on the default stream

    def call(i):
        rc = lib.qlinear_argmax(t, Wk[i % Pk].data_ptr(), N, K, x.data_ptr(), M, idx.data_ptr(), val.data_ptr(), sh)
        if rc != 0:
            raise RuntimeError(f"qlinear_argmax failed: {rc}")

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    torch.cuda.synchronize(dev)
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=stream):
        for i in range(reps):
            call(i)
    with torch.cuda.stream(stream):
        gk.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(replays):
        with torch.cuda.stream(stream):
            e0.record(stream)
            gk.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1) / reps)
    del gk, Wk
    torch.cuda.empty_cache()
    return float(np.median(times))


# Greedy output heads: type, K, N (vocabulary), M
TABLE_HEAD = [(14, 4096, 151936, 1), (14, 4096, 32000, 1)]

# Fused decode calls: kind, type, K, N, M (the 8B down projection fed by the SiLU gate, the
# 8B gate projection fed by RMSNorm)
TABLE_FUSED = [("silu", 12, 12288, 4096, 1), ("rmsnorm", 12, 4096, 12288, 1)]

# Projection sets sharing x (one qlinear_multi call each): name, type, K, (N_j), M
TABLE_MULTI = [
    ("8B Q/K/V", 12, 4096, (4096, 1024, 1024), 1),
    ("8B gate/up", 12, 4096, (12288, 12288), 1),
    ("27B Q/K/V", 23, 5120, (5120, 1024, 1024), 1),
]

# Every layer shape of the scope table: (type, K, N, M)
TABLE_SHAPES = [
    (12, 1024, 1024, 1),
    (12, 4096, 4096, 1), (12, 4096, 1024, 1), (12, 4096, 12288, 1), (12, 12288, 4096, 1),
    (12, 4096, 4096, 4), (12, 4096, 12288, 4), (12, 12288, 4096, 4),
    (23, 5120, 5120, 1), (23, 5120, 17408, 1), (23, 17408, 5120, 1),
    (13, 5120, 17408, 1), (14, 5120, 17408, 1),
    (12, 4096, 12288, 32), (12, 4096, 12288, 64), (12, 4096, 12288, 128), (12, 4096, 12288, 512),
    (23, 4096, 12288, 32), (12, 4096, 4096, 64), (12, 12288, 4096, 32), (12, 12288, 4096, 128),
    (13, 5120, 17408, 256), (14, 5120, 17408, 256),
    (Q6_K_A16, 5120, 17408, 1), (Q6_K_A16, 5120, 17408, 256),
]
TYPE_NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K", 23: "IQ4_XS", Q6_K_A16: "Q6_K_A16"}


def run_table(args):
    """--table: every layer shape of the scope table timed alone (time_shape, median of 5
    replays), one JSON line per shape with GB/s, TFLOP/s and the fraction of the measured
    peak that bounds it (HBM for M <= 64, the tensor pipe above)."""
    import torch
    import gguf_weight_only_gb300 as ql
    from gguf_weight_only_gb300 import build

    build.build()
    lib = ql.lib()
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    hbm, tf_burst, _, peak_kind = peaks()
    stream = torch.cuda.Stream(device=dev)
    for t, K, N, M in TABLE_SHAPES:
        ms = time_shape(t, K, N, M, lib.qlinear, 200 if M <= 8 else 40, dev, stream, l2, replays=5)
        gbs = alg_bytes(t, K, N, M) / (ms * 1e-3) / 1e9
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        bound = "hbm" if M <= 64 else "tensor"
        frac = gbs / hbm if bound == "hbm" else tf / tf_burst
        print(json.dumps({"type": TYPE_NAMES[t], "K": K, "N": N, "M": M,
                          "path": "gemv" if M <= lib.qlinear_gemv_max_m() else "gemm",
                          "us": round(ms * 1e3, 2), "GBs": round(gbs, 1), "TFLOPs": round(tf, 1),
                          "bound": bound, "frac": round(frac, 4), "peak_kind": peak_kind,
                          "status": ql.device_status()}), flush=True)
    for name, t, K, Ns, M in TABLE_MULTI:
        byts = sum(alg_bytes(t, K, N, M) for N in Ns) - 2 * M * K * (len(Ns) - 1)   # x read once
        res = {}
        for fused in (True, False):
            ms = time_multi(t, K, Ns, M, 200, dev, stream, l2, lib, fused=fused)
            res["fused" if fused else "separate"] = {"us": round(ms * 1e3, 2), "GBs": round(byts / (ms * 1e-3) / 1e9, 1),
                                                     "frac": round(byts / (ms * 1e-3) / 1e9 / hbm, 4)}
        print(json.dumps({"projections": name, "type": TYPE_NAMES[t], "K": K, "N": list(Ns), "M": M, **res,
                          "peak_kind": peak_kind, "status": ql.device_status()}), flush=True)
    for t, K, N, M in TABLE_HEAD:
        ms = time_argmax(t, K, N, M, 50, dev, stream, l2, lib)
        plain = time_shape(t, K, N, M, lib.qlinear, 50, dev, stream, l2, replays=5)
        byts = N * (K // 256) * BB[t] + 2 * M * K + 12 * M
        print(json.dumps({"argmax_head": TYPE_NAMES[t], "K": K, "N": N, "M": M, "us": round(ms * 1e3, 2),
                          "GBs": round(byts / (ms * 1e-3) / 1e9, 1), "frac": round(byts / (ms * 1e-3) / 1e9 / hbm, 4),
                          "logits_us": round(plain * 1e3, 2), "peak_kind": peak_kind,
                          "status": ql.device_status()}), flush=True)
    for kind, t, K, N, M in TABLE_FUSED:
        ms = time_fused(kind, t, K, N, M, 200, dev, stream, l2, lib)
        plain = time_shape(t, K, N, M, lib.qlinear, 200, dev, stream, l2, replays=5)
        # weights + the prologue's inputs (gate fp16 and up fp32, or h and w fp32) + residual and y
        byts = N * (K // 256) * BB[t] + (6 * M * K if kind == "silu" else 4 * M * K + 4 * K) + 8 * M * N
        print(json.dumps({"fused": kind, "type": TYPE_NAMES[t], "K": K, "N": N, "M": M, "us": round(ms * 1e3, 2),
                          "GBs": round(byts / (ms * 1e-3) / 1e9, 1), "frac": round(byts / (ms * 1e-3) / 1e9 / hbm, 4),
                          "plain_us": round(plain * 1e3, 2), "peak_kind": peak_kind,
                          "status": ql.device_status()}), flush=True)


# ---------------------------------------------------------------------------- oracle on the CPU

def cpu_baseline(budget_s=12.0):
    """The fp64 oracle (C, one POSIX thread per core) on a bounded sample of the decode
    workload: for each layer shape, its first rows (all of them when they fit), computed
    repeatedly until about budget_s / 4 seconds have been spent; scaled to GB/s."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    total_bytes, total_s, used = 0, 0.0, []
    for i, (K, N) in enumerate(DECODE_SHAPES):
        rows = max(cores, 64)
        W = synth.weights(DECODE_TYPE, rows, K, [11, i])
        x = synth.activations(DECODE_M, K, [12, i])
        t0 = time.perf_counter()
        oracle.qlinear(DECODE_TYPE, W, rows, K, x, n_threads=cores)
        dt = max(time.perf_counter() - t0, 1e-6)
        rows = int(min(N, max(rows, rows * (budget_s / 4) / dt)))
        W = synth.weights(DECODE_TYPE, rows, K, [11, i])
        reps, spent = 0, 0.0
        while spent < budget_s / 4 or reps == 0:
            t0 = time.perf_counter()
            oracle.qlinear(DECODE_TYPE, W, rows, K, x, n_threads=cores)
            spent += time.perf_counter() - t0
            reps += 1
        total_s += spent
        total_bytes += reps * alg_bytes(DECODE_TYPE, K, rows, DECODE_M)
        used.append(f"{rows}x{reps}")
    return {"value": round(total_bytes / total_s / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"rows x passes per (K,N) decode shape: {used}, M=1, fp64, {total_s:.1f} s"}


def run_reference(args):
    """--impl reference: the oracle on the host cores, same metric and workload. Each step
    runs the oracle over the first R rows of every layer shape (R calibrated once so that the
    whole run stays within a few minutes) and the value is that sample's GB/s."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    per_step_s = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    samples = []
    for i, (K, N) in enumerate(DECODE_SHAPES):
        x = synth.activations(DECODE_M, K, [12, i])
        rows = max(cores, 32)
        W = synth.weights(DECODE_TYPE, rows, K, [11, i])
        t0 = time.perf_counter()
        oracle.qlinear(DECODE_TYPE, W, rows, K, x, n_threads=cores)
        dt = max(time.perf_counter() - t0, 1e-6)
        rows = int(max(cores, min(N, rows * (per_step_s / 4) / dt)))
        samples.append((K, rows, synth.weights(DECODE_TYPE, rows, K, [11, i]), x))
    vals, times = [], []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        nbytes = 0
        for K, rows, W, x in samples:
            oracle.qlinear(DECODE_TYPE, W, rows, K, x, n_threads=cores)
            nbytes += alg_bytes(DECODE_TYPE, K, rows, DECODE_M)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            vals.append(nbytes / dt / 1e9)
            times.append(dt)
    v = float(np.median(vals))
    sample = f"first {[r for _, r, _, _ in samples]} rows of the four (K,N) decode shapes per step, M=1, fp64"
    return {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(float(np.median(times)) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_case(args):
    """--case TYPE,K,N,M: W warm-up calls and then K calls of one layer shape through the
    C ABI on fresh weights (no CUDA graph, no timing): the command profilers wrap."""
    import torch
    import gguf_weight_only_gb300 as ql
    from gguf_weight_only_gb300 import build

    t, K, N, M = (int(v) for v in args.case.split(","))
    build.build()
    lib = ql.lib()
    dev = torch.device("cuda", 0)
    W = device_weights(t, N, K, [7, t, K, N], dev)
    x = torch.from_numpy(synth.activations(M, K, [8, t, M])).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    sh = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(args.warmup + args.steps):
        rc = lib.qlinear(t, W.data_ptr(), N, K, x.data_ptr(), M, y.data_ptr(), sh)
        if rc != 0:
            raise RuntimeError(f"qlinear failed: {ql.strerror(rc)}")
    torch.cuda.synchronize(dev)
    st = ql.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}")
    print(json.dumps({"case": [t, K, N, M], "launches": args.warmup + args.steps,
                      "kernel_launches_per_call": lib.qlinear_launch_count(t, N, K, M)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--case", default=None, help="TYPE,K,N,M: run one layer shape (for profilers)")
    ap.add_argument("--table", action="store_true", help="time every layer shape of the scope table")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.case:
        run_case(args)
        return
    if args.table:
        run_table(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
