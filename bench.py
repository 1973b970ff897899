"""Benchmark of the streamed pairwise-score hot path on GB300.

Default workload (one GPU): InfoNCE row logsumexp, fp32, z [8192,64] unit rows, S = z z^T / 0.07,
exclude_self, forward plus the replay backward that gives the gradient in z. One step = the forward
(every pair evaluated once) plus the backward (every pair replayed in a row sweep and a column sweep)
through libtp's C ABI. Metric: Gpairs/s = N*M / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libtp|reference] [--workload 1..5]

--impl reference times the oracle (plain fp64 CPU loops) on the host cores, on a bounded sample of
the same workload, and prints the same JSON line with "impl": "reference".
Under torchrun each rank runs an independent replica of the workload on its own GPU (weak scaling,
no collective in the data path); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
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

METRIC = "Gpairs/s per fused consumer (fwd+bwd) at fp32/fp64; % of FP32/FP64 peak"
SM_COUNT = 152
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per SM (4 sub-partitions x 32)


def peaks():
    p = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
    sm_mhz = float(p.get("sm_max_mhz", 2070.0))
    return {
        "hbm_gbs": float(p.get("hbm_gbs", 6800.0)),
        "sm_max_mhz": sm_mhz,
        "fp32_tflops": SM_COUNT * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12,
        "fp64_tflops": 1.25,  # nominal GB300 FP64 rate (no measured figure)
        # fp16 tensor peak = the measured bf16 burst peak (same rate); tf32 = that x the nominal 1.1 / 2.25
        "f16_tflops": float(p.get("bf16_tflops", 1900.0)),
        "tf32_tflops": float(p.get("bf16_tflops", 1900.0)) * 1.1 / 2.25,
        "source": "MEASURED_PEAKS.json" if p else "fallback",
    }


# ------------------------------------------------------------------------------------------------
# per-kernel timing through libtp's launch hook
# ------------------------------------------------------------------------------------------------


class KernelTimer:
    """Per-launch device durations from the library's own event timer (tp_timer_*): an event pair is
    recorded on the launch stream around every libtp kernel, with no host callback in the launch path."""

    def __init__(self, capacity):
        from lazy_score_matrix_gb300 import _lib
        self._lib = _lib
        self.capacity = capacity
        self.n = 0

    def __enter__(self):
        self._lib.check(self._lib.load().tp_timer_start(self.capacity), "tp_timer_start")
        return self

    def __exit__(self, *a):
        self.n = int(self._lib.load().tp_timer_stop())

    def summary(self):
        import ctypes
        lib = self._lib.load()
        name, ms = ctypes.c_char_p(), ctypes.c_float()
        out = {}
        for i in range(self.n):
            self._lib.check(lib.tp_timer_read(i, ctypes.byref(name), ctypes.byref(ms)), "tp_timer_read")
            d = out.setdefault(name.value.decode(), [0, 0.0])
            d[0] += 1
            d[1] += ms.value
        return {k: {"launches": v[0], "total_ms": v[1], "avg_ms": v[1] / v[0]} for k, v in out.items()}


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def result(self):
        win = [l for t, l in self.lines if self.t0 is not None and self.t0 - 0.06 <= t <= self.t1 + 0.06]
        if not win:
            win = [l for _, l in self.lines]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in win:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# workloads
# ------------------------------------------------------------------------------------------------


class Workload:
    """One hot-path step on device-resident inputs, plus the same step end to end from host buffers."""
    name = ""
    dtype = "f32"
    pairs = 0
    flops_per_pair = {}  # per kernel name: algorithmic flop per pair the launch processes
    bound = "alu"

    def step(self):
        raise NotImplementedError

    def e2e_step(self):
        raise NotImplementedError


class InfoNCE(Workload):
    """Workload 2: InfoNCE row logsumexp fwd + replay bwd, z [8192,64] fp32."""

    def __init__(self, dev, N=8192, D=64):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(2, N=N, D=D)
        self.N, self.D = N, D
        self.pairs = N * N
        self.name = f"infonce_logsumexp_f32_z{N}x{D}_fwd+bwd"
        self.score = ops.Score("linear", scale=w["scale"])
        self.z = w["z"].to(dev)
        self.gl = w["grad_lse"].to(dev)
        self.want = (True, True, False, False, False, False, False)
        # pinned host copies for the end-to-end path
        self.z_h = w["z"].pin_memory()
        self.gl_h = w["grad_lse"].pin_memory()
        self.lse_h = torch.empty(N, dtype=torch.float32).pin_memory()
        self.grad_h = torch.empty(N, D, dtype=torch.float32).pin_memory()
        self.z_d = torch.empty_like(self.z)
        self.gl_d = torch.empty_like(self.gl)
        self.h2d = self.z_h.numel() * 4 + self.gl_h.numel() * 4
        self.d2h = self.lse_h.numel() * 4 + self.grad_h.numel() * 4
        D2 = 2 * D
        # algorithmic flop per pair and launch (FMA = 2): forward 2D+3; backward 387 = (2D+3) + 2D + 2D,
        # the row sweep credited with the recompute and dX, the column sweep with dY only; a kernel
        # that produces the whole backward (X = Y, one symmetric sweep) is credited with all of it.
        # (kernel: (flop per pair, bound)); "tensor-f16" kernels run the contraction on tcgen05 kind::f16
        # (scaled fp16 hi/lo split), credited with the algorithmic flop against the fp16 tensor peak
        self.flops_per_pair = {"fwd_sweep_lse": (D2 + 3, "alu"), "bwd_sweep_lse_row": (D2 + 3 + D2, "alu"),
                               "bwd_sweep_lse_col": (D2, "alu"), "bwd_sweep_lse_sym": (D2 + 3 + D2 + D2, "alu"),
                               "lse_fwd_tc": (D2 + 3, "tensor-f16"), "lse_bwd_sym_tc": (D2 + 3 + D2 + D2, "tensor-f16")}
        self.step_flops_per_pair = (D2 + 3) + (D2 + 3 + D2 + D2)

    def step(self):
        lse = self.ops.pairwise_logsumexp(self.z, self.z, self.score, True)
        g = self.ops.pairwise_logsumexp_backward(self.z, self.z, self.score, lse, self.gl, True, self.want, same=True)
        return lse, g["dX"]

    def e2e_step(self):
        self.z_d.copy_(self.z_h, non_blocking=True)
        self.gl_d.copy_(self.gl_h, non_blocking=True)
        lse = self.ops.pairwise_logsumexp(self.z_d, self.z_d, self.score, True)
        g = self.ops.pairwise_logsumexp_backward(self.z_d, self.z_d, self.score, lse, self.gl_d, True, self.want,
                                                 same=True)
        self.lse_h.copy_(lse, non_blocking=True)
        self.grad_h.copy_(g["dX"], non_blocking=True)


class RbfMatmul(Workload):
    """Workload 1: rbf kernel product K @ [V | 1] fp32, X, Y [1024,3], fwd + grads in X, Y, V."""

    def __init__(self, dev):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(1)
        self.N, self.D = w["X"].shape
        self.M = w["Y"].shape[0]
        self.C = w["V"].shape[1]
        self.pairs = self.N * self.M
        self.name = "rbf_kernel_matmul_f32_X1024x3_Y1024x3_V1024x4_fwd+bwd"
        self.score = ops.Score("rbf", gamma=w["gamma"])
        self.X, self.Y, self.V, self.G = (w[k].to(dev) for k in ("X", "Y", "V", "grad_out"))
        self.host = {k: w[k].pin_memory() for k in ("X", "Y", "V", "grad_out")}
        self.dev_in = {k: torch.empty_like(v) for k, v in ((k, getattr(self, kk)) for k, kk in
                                                         (("X", "X"), ("Y", "Y"), ("V", "V"), ("grad_out", "G")))}
        self.out_h = torch.empty(self.N, self.C).pin_memory()
        self.h2d = sum(v.numel() * 4 for v in self.host.values())
        self.d2h = self.out_h.numel() * 4 + (self.N + self.M) * self.D * 4 + self.M * self.C * 4
        D, C = self.D, self.C
        # fwd 2D+2 (distance) + 1 (scale) + 2C; bwd recompute 2D+3, dS 2C, dV 2C, coef 2, dX 2D+1, dY 2D+1
        self.flops_per_pair = {"fwd_sweep_matmul": (2 * D + 3 + 2 * C, "alu"),
                               "bwd_sweep_matmul_row": (2 * D + 3 + 2 * C + 2 + 2 * D + 1, "alu"),
                               "bwd_sweep_matmul_col": (2 * C + 2 * D + 1, "alu")}
        self.step_flops_per_pair = (2 * D + 3 + 2 * C) + (2 * D + 3 + 4 * C + 2 + 4 * D + 2)
        self.grads_h = [torch.empty(self.N, D).pin_memory(), torch.empty(self.M, D).pin_memory(),
                        torch.empty(self.M, C).pin_memory()]

    def step(self):
        out = self.ops.pairwise_matmul(self.X, self.Y, self.V, self.score)
        g = self.ops.pairwise_matmul_backward(self.X, self.Y, self.V, self.score, self.G,
                                              (True, True, True, False, False, False, False))
        return out, g

    def e2e_step(self):
        for k, v in self.host.items():
            self.dev_in[k].copy_(v, non_blocking=True)
        d = self.dev_in
        out = self.ops.pairwise_matmul(d["X"], d["Y"], d["V"], self.score)
        g = self.ops.pairwise_matmul_backward(d["X"], d["Y"], d["V"], self.score, d["grad_out"],
                                              (True, True, True, False, False, False, False))
        self.out_h.copy_(out, non_blocking=True)
        for h, k in zip(self.grads_h, ("dX", "dY", "dV")):
            h.copy_(g[k], non_blocking=True)


class Knn(Workload):
    """Workload 3: exact k-NN top-16, X [65536,16] vs R [1048576,16] integers in [-8,8], fp32."""

    def __init__(self, dev):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(3)
        self.N, self.D = w["X"].shape
        self.M = w["R"].shape[0]
        self.k = w["k"]
        self.pairs = self.N * self.M
        self.name = "knn_topk16_f32_X65536x16_R1048576x16_fwd"
        self.score = ops.Score("sqeuclidean")
        self.X, self.R = w["X"].to(dev), w["R"].to(dev)
        self.X_h, self.R_h = w["X"].pin_memory(), w["R"].pin_memory()
        self.X_d, self.R_d = torch.empty_like(self.X), torch.empty_like(self.R)
        self.v_h = torch.empty(self.N, self.k).pin_memory()
        self.i_h = torch.empty(self.N, self.k, dtype=torch.int64).pin_memory()
        self.h2d = (self.X_h.numel() + self.R_h.numel()) * 4
        self.d2h = self.N * self.k * 12
        # the SIMT sweep runs the distance on the FP32 pipe; the tensor-core kernel runs the contraction
        # on tcgen05 (tf32) and the selection on the ALUs: it is credited with the same algorithmic flop
        self.flops_per_pair = {"topk_sweep": (2 * self.D + 2, "alu"), "topk_tc": (2 * self.D + 2, "tensor-tf32")}
        self.step_flops_per_pair = 2 * self.D + 2

    def step(self):
        return self.ops.pairwise_topk(self.X, self.R, self.score, self.k, False)

    def e2e_step(self):
        self.X_d.copy_(self.X_h, non_blocking=True)
        self.R_d.copy_(self.R_h, non_blocking=True)
        v, i = self.ops.pairwise_topk(self.X_d, self.R_d, self.score, self.k, False)
        self.v_h.copy_(v, non_blocking=True)
        self.i_h.copy_(i, non_blocking=True)


class Attention(Workload):
    """Workload 4: softmax_matmul attention fp32, Q, K, V [16384,64], scale 1/8, fwd + grads."""

    def __init__(self, dev):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(4)
        self.N, self.D = w["Q"].shape
        self.M = w["K"].shape[0]
        self.C = w["V"].shape[1]
        self.pairs = self.N * self.M
        self.name = "attention_softmax_matmul_f32_QKV16384x64_fwd+bwd"
        self.score = ops.Score("linear", scale=w["scale"])
        self.Q, self.K, self.V, self.G = (w[k].to(dev) for k in ("Q", "K", "V", "grad_out"))
        self.host = {k: w[k].pin_memory() for k in ("Q", "K", "V", "grad_out")}
        self.dev_in = {k: torch.empty_like(v) for k, v in
                       (("Q", self.Q), ("K", self.K), ("V", self.V), ("grad_out", self.G))}
        self.out_h = torch.empty(self.N, self.C).pin_memory()
        self.grads_h = [torch.empty(self.N, self.D).pin_memory(), torch.empty(self.M, self.D).pin_memory(),
                        torch.empty(self.M, self.C).pin_memory()]
        self.h2d = sum(v.numel() * 4 for v in self.host.values())
        self.d2h = (self.N * self.C + (self.N + self.M) * self.D + self.M * self.C) * 4
        D, C = self.D, self.C
        # fwd 2D + 2C + 3; bwd: S 2D, dV 2C, dP 2C, dS 2, dQ 2D, dK 2D (dQ row sweep: S, dP, dS, dQ).
        # Tensor-core path: the forward's S and exp go to the log-sum-exp pass and P V (2C) to the second
        # pass (its replay of S is not credited); the row sweep as above, the column sweep dK + dV (its
        # replay of S and dP not credited), against the fp16 tensor peak.
        self.flops_per_pair = {"fwd_sweep_softmax": (2 * D + 2 * C + 3, "alu"),
                               "bwd_sweep_softmax_row": (2 * D + 2 * C + 2 + 2 * D, "alu"),
                               "bwd_sweep_softmax_col": (2 * D, "alu"),
                               "bwd_sweep_softmax_col_dv": (2 * C, "alu"),
                               "lse_fwd_tc": (2 * D + 3, "tensor-f16"),
                               "attn_fwd_tc": (2 * C, "tensor-f16"),
                               "attn_bwd_row_tc": (2 * D + 2 * C + 2 + 2 * D, "tensor-f16"),
                               "attn_bwd_col_tc": (2 * D + 2 * C, "tensor-f16")}
        self.step_flops_per_pair = (2 * D + 2 * C + 3) + (2 * D + 2 * C + 2 * C + 2 + 2 * D + 2 * D)

    def step(self):
        out, lse = self.ops.pairwise_softmax_matmul(self.Q, self.K, self.V, self.score)
        g = self.ops.pairwise_softmax_matmul_backward(self.Q, self.K, self.V, self.score, out, lse, self.G,
                                                      (True, True, True, False, False, False, False))
        return out, g

    def e2e_step(self):
        for k, v in self.host.items():
            self.dev_in[k].copy_(v, non_blocking=True)
        d = self.dev_in
        out, lse = self.ops.pairwise_softmax_matmul(d["Q"], d["K"], d["V"], self.score)
        g = self.ops.pairwise_softmax_matmul_backward(d["Q"], d["K"], d["V"], self.score, out, lse, d["grad_out"],
                                                      (True, True, True, False, False, False, False))
        self.out_h.copy_(out, non_blocking=True)
        for h, k in zip(self.grads_h, ("dX", "dY", "dV")):
            h.copy_(g[k], non_blocking=True)


class CausalAttention(Attention):
    """Workload 6: workload 4 under the causal mask (key j <= query i), the attention of the Task Map's
    softmax_matmul(V, mask=tp.masks.causal()). Pairs are the kept ones, N (N + 1) / 2."""

    def __init__(self, dev):
        super().__init__(dev)
        self.name = "causal_attention_softmax_matmul_f32_QKV16384x64_fwd+bwd"
        self.score = self.ops.Score("linear", scale=self.score.scale, pair_mask="causal")
        self.pairs = self.N * (self.N + 1) // 2


class Svgd(Workload):
    """Workload 5: SVGD direction fp64, x [131072,8], score = -x, rbf gamma 0.1, one fused sweep."""
    dtype = "f64"

    def __init__(self, dev):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(5)
        self.N, self.D = w["x"].shape
        self.M = self.N
        self.gamma = w["gamma"]
        self.pairs = self.N * self.N
        self.name = "svgd_direction_f64_x131072x8_fwd"
        self.x, self.sc = w["x"].to(dev), w["score"].to(dev)
        self.x_h, self.s_h = w["x"].pin_memory(), w["score"].pin_memory()
        self.x_d, self.s_d = torch.empty_like(self.x), torch.empty_like(self.sc)
        self.phi_h = torch.empty(self.N, self.D, dtype=torch.float64).pin_memory()
        self.h2d = 2 * self.N * self.D * 8
        self.d2h = self.N * self.D * 8
        D = self.D
        # one sweep with V = [score | x | 1]: distance 2D+2, -gamma scale 1, accumulate 2(2D+1)
        self.flops_per_pair = {"fwd_sweep_svgd": (2 * D + 3 + 2 * (2 * D + 1), "alu")}
        self.step_flops_per_pair = 2 * D + 3 + 2 * (2 * D + 1)

    def step(self):
        return self.ops.svgd_direction(self.x, self.sc, self.gamma)

    def e2e_step(self):
        self.x_d.copy_(self.x_h, non_blocking=True)
        self.s_d.copy_(self.s_h, non_blocking=True)
        phi = self.ops.svgd_direction(self.x_d, self.s_d, self.gamma)
        self.phi_h.copy_(phi, non_blocking=True)


WORKLOADS = {1: RbfMatmul, 2: InfoNCE, 3: Knn, 4: Attention, 5: Svgd, 6: CausalAttention}


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time (weak scaling: every rank runs its own replica)."""
    if world <= 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gpairs(world: int, pairs: int, steps: int, seconds: float) -> float:
    """Pairs processed by all ranks per second of the slowest rank, in Gpairs/s."""
    return world * pairs * steps / seconds / 1e9


def time_steps(fn, steps, flush):
    """Per-step CUDA events on the current stream; L2 flushed (untimed) before every step."""
    total = 0.0
    pairs = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        pairs.append((a, b))
    torch.cuda.synchronize()
    for a, b in pairs:
        total += a.elapsed_time(b)
    return total  # ms


def capture_step(wl):
    """The step captured once in a CUDA graph (its launches replayed without the host in between), or None
    if the capture fails (the step then runs eagerly)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            wl.step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            wl.step()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        return g
    except Exception:
        torch.cuda.synchronize()
        return None


def gpu_arm(args, rank, world):
    from lazy_score_matrix_gb300 import _lib

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload](dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 256 MB > 129 MB L2
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # The timed steps: replays of the step captured in a CUDA graph, nothing recorded between its launches.
    graph = capture_step(wl)
    clocks.t0 = time.time()
    ms = time_steps(graph.replay if graph is not None else wl.step, args.steps, flush)
    clocks.t1 = time.time()
    torch.cuda.synchronize()
    # Kernel durations for the roofline: the same steps again, eagerly, with CUDA events around every
    # launch on its stream (events between launches would add gaps to the timed steps above).
    _lib.launch_count(reset=True)
    timer = KernelTimer(capacity=64 * args.steps + 64)
    with timer:
        time_steps(wl.step, args.steps, flush)
    launches = _lib.launch_count()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(ms, world, dev)
    # end to end: host buffers, copies inside the timed region
    for _ in range(2):
        wl.e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        wl.e2e_step()
        torch.cuda.current_stream().synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    clocks.stop()
    if rank != 0:
        return None
    pk = peaks()
    ms_step = ms / args.steps
    value = whole_job_gpairs(world, wl.pairs, args.steps, ms / 1e3)
    ksum = timer.summary()
    dom = max(ksum.items(), key=lambda kv: kv[1]["total_ms"])
    dname, dstat = dom
    credit = wl.flops_per_pair.get(dname)
    roof = None
    if credit is not None:
        fpp, bound = credit
        ach = fpp * wl.pairs / (dstat["avg_ms"] / 1e3) / 1e12
        if bound == "tensor-f16":
            peak = pk["f16_tflops"]
            src = f"fp16 tensor (kind::f16 operands): measured bf16 {pk['f16_tflops']:.0f} TFLOP/s, same rate, of measured"
        elif bound == "tensor-tf32":
            peak = pk["tf32_tflops"]
            src = (f"tf32 tensor: measured bf16 {pk['f16_tflops']:.0f} TFLOP/s x 1.1/2.25 "
                   f"(nominal tf32/bf16), of measured")
        else:
            peak = pk["fp32_tflops"] if wl.dtype == "f32" else pk["fp64_tflops"]
            src = (f"FP32 pipe: {SM_COUNT} SMs x {FP32_LANES_PER_SM} lanes x 2 flop x {pk['sm_max_mhz']:.0f} MHz "
                   f"(derived from unit counts and the measured max clock)")
        roof = {"kernel": dname, "bound": "tensor" if bound.startswith("tensor") else bound,
                "operands": bound[len("tensor-"):] if bound.startswith("tensor") else "fp32",
                "achieved": round(ach, 3), "peak": round(peak, 2),
                "unit": "TFLOP/s", "frac": round(ach / peak, 4), "traffic": traffic_for(dname, wl.name),
                "peak_source": src, "flop_per_pair": fpp}
    step_tflops = wl.step_flops_per_pair * wl.pairs / (ms_step / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "Gpairs/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded, shapes of the workload)",
        "config": {"workload": wl.name, "N": wl.N, "M": getattr(wl, "M", wl.N), "D": wl.D, "pairs_per_step": wl.pairs,
                   "l2": "flushed before every timed step (256 MB write, untimed)",
                   "launch": ("step captured once in a CUDA graph, replayed per timed step" if graph is not None
                              else "eager"),
                   "kernel_times": "CUDA events around every launch, in a second pass of the same steps",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "impl": "libtp",
        "roofline": roof,
        "step_roofline": {"achieved_tflops": round(step_tflops, 3), "flop_per_pair": wl.step_flops_per_pair,
                          "frac_fp32_pipe" if wl.dtype == "f32" else "frac_fp64_pipe":
                              round(step_tflops / (pk["fp32_tflops"] if wl.dtype == "f32" else pk["fp64_tflops"]), 4)},
        "kernels": {k: {"launches": v["launches"], "avg_us": round(v["avg_ms"] * 1e3, 2),
                        "share": round(v["total_ms"] / sum(x["total_ms"] for x in ksum.values()), 4)}
                    for k, v in sorted(ksum.items(), key=lambda kv: -kv[1]["total_ms"])},
        "gpu_launches": launches,
        "e2e": {"value": round(whole_job_gpairs(world, wl.pairs, args.steps, e2e_s), 4), "unit": "Gpairs/s",
                "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h},
        "clocks": clocks.result(),
    }
    return line


def traffic_for(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summary (lines
    `kernel workload bytes src=<hash>`), if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = source_hash()
    for l in open(path):
        parts = l.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[3] == f"src={cur}":
            return float(parts[2])
    return None


# The sources the tensor-core kernels (the only ones with traffic entries) are compiled from: their
# translation units and every header those include.
TC_SOURCES = ("tp_args.h", "tp_device.cuh", "tp_launch.h", "tp_tc.cuh", "tp_tc_attn.cu", "tp_tc_host.h",
              "tp_tc_lse.cu", "tp_tc_topk.cu")


def source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lazy_score_matrix_gb300", "csrc")
    for f in TC_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:12]


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------------------


def oracle_infonce(rows: int, threads: int = 0):
    """Oracle forward + backward of the InfoNCE workload on its first `rows` rows against all columns.
    Returns (seconds, pairs, threads used)."""
    from lazy_score_matrix_gb300 import synth
    from oracle import oracle
    w = synth.workload(2)
    z = w["z"].double().numpy()
    N = z.shape[0]
    oracle.set_threads(threads)
    used = oracle.get_threads()
    # rows 0..rows-1 against every column: column i is row i's own point, so exclude_self drops (i, i)
    pb = oracle.Problem(z[:rows], z, metric="linear", scale=w["scale"])
    t0 = time.perf_counter()
    lse = oracle.logsumexp(pb, exclude_self=True)
    oracle.logsumexp_backward(pb, lse, np.full(rows, -1.0 / N), exclude_self=True)
    dt = time.perf_counter() - t0
    return dt, rows * N, used


def cpu_baseline(sample_rows=8192):
    dt, pairs, used = oracle_infonce(sample_rows)
    return {"value": round(pairs / dt / 1e9, 6), "unit": "Gpairs/s", "cores": used, "kind": "oracle",
            "sample": f"oracle fwd+bwd on all {pairs} pairs of the 8192x8192 InfoNCE workload "
                      f"({sample_rows} rows), {dt:.1f} s"}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    rows = 2048 if args.workload == 2 else 0
    times = []
    for _ in range(args.warmup):
        oracle_infonce(256)
    used = 0
    for _ in range(args.steps):
        dt, pairs, used = oracle_infonce(rows)
        times.append(dt)
    tot = sum(times)
    value = pairs * args.steps / tot / 1e9
    return {"metric": METRIC, "value": round(value, 6), "unit": "Gpairs/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": "infonce_logsumexp_f32_z8192x64_fwd+bwd", "N": 8192, "M": 8192, "D": 64,
                       "sample_rows_per_step": rows},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "Gpairs/s", "cores": used, "kind": "oracle",
                             "sample": f"{rows} of 8192 rows against all 8192 columns per step"},
            "e2e": {"value": round(value, 6), "unit": "Gpairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="libtp", choices=["libtp", "reference"])
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = reference_arm(args, rank, world)
        if line:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = gpu_arm(args, rank, world)
    if line is not None:
        if not args.no_cpu_baseline and args.workload == 2:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
