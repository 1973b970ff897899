"""Benchmark of the streamed pairwise-score hot path on GB300.

One step of a workload is one pass of its consumer over the workload's whole problem through libtp's
C ABI: the forward (every pair evaluated once) and, where the workload has one, the replay backward
(every pair evaluated again). Metric: Gpairs/s = pairs of the problem / step time (kept pairs under a
pair mask). The workloads are those of the torchpairwise guide "Using Torchpairwise in Models" (Task
Map and Stein Variational Gradient Descent sections), with seeded synthetic inputs of their shapes:

  1  rbf kernel product K @ [V | 1], X, Y [1024,3], fp32, forward + gradients in X, Y, V
  2  InfoNCE row log-sum-exp, z [8192,64] unit rows, S = z z^T / 0.07, exclude_self, forward + z.grad
  3  exact k-NN top-16, X [65536,16] vs R [1048576,16], integers in [-8,8], fp32, forward
  4  attention softmax_matmul, Q, K, V [16384,64], scale 1/8, fp32, forward + gradients
  5  SVGD direction, x [131072,8], score = -x, rbf gamma 0.1, fp64, forward
  6  workload 4 under the causal mask (kept pairs N (N + 1) / 2)

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libtp|reference] [--workload 2]
                    [--workloads 1,2,3,4,5,6] [--no-cpu-baseline] [--small] [--no-clock-pass] [--no-peaks]

The top-level JSON line is workload --workload (default 2, timed for exactly K steps); the line's
"workloads" object holds every workload of --workloads, each with its own step count, roofline, e2e and
CPU baseline. --impl reference times the oracle (plain fp64 CPU loops) on the host cores, on a bounded
sample of the top-level workload, and prints the same JSON line with "impl": "reference". Under torchrun
each rank runs an independent replica on its own GPU (weak scaling, no collective in the data path); rank
0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
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
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per SM (4 sub-partitions x 32)
FALLBACK_SMS = 152       # GB300, used only when no device can be queried

# ------------------------------------------------------------------------------------------------
# peaks: the measured copy / bf16 GEMM figures of MEASURED_PEAKS.json, the device's SM count, and our own measured
# fp32 / fp64 FMA and exp2 rates (libtp_peaks)
# ------------------------------------------------------------------------------------------------


def measured_alu_peaks():
    """Rates of the calibration kernels on the current device (TFLOP/s for FMA, Tops/s for exp2), each
    timed with CUDA events over one launch of ~50-100 ms after a warm-up launch; None if unavailable."""
    path = os.path.join(ROOT, "lazy_score_matrix_gb300", "libtp_peaks.so")
    if not os.path.exists(path) or not torch.cuda.is_available():
        return None
    lib = ctypes.CDLL(path)
    lib.tpk_peak.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_float)]
    lib.tpk_peak.restype = ctypes.c_double
    out = {}
    for kind, name, iters in ((0, "fp32_fma_tflops", 1_500_000), (1, "fp64_fma_tflops", 40_000),
                              (2, "ex2_tops", 200_000)):
        ms = ctypes.c_float()
        r = lib.tpk_peak(kind, iters, 4, ctypes.byref(ms))
        out[name] = round(r, 3) if r > 0 else None
        out[name.rsplit("_", 1)[0] + "_ms"] = round(ms.value, 2)
    return out


_PEAKS = None


def peaks(dev=None):
    global _PEAKS
    if _PEAKS is not None:
        return _PEAKS
    p = {}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
    sm_mhz = float(p.get("sm_max_mhz", 2070.0))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count if dev is not None else FALLBACK_SMS
    alu = measured_alu_peaks() if dev is not None else None
    derived32 = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    _PEAKS = {
        "hbm_gbs": float(p.get("hbm_gbs", 6800.0)),
        "sm_max_mhz": sm_mhz,
        "sms": sms,
        "fp32_derived_tflops": derived32,
        "fp32_tflops": (alu or {}).get("fp32_fma_tflops") or derived32,
        "fp64_tflops": (alu or {}).get("fp64_fma_tflops") or 1.25,
        "ex2_tops": (alu or {}).get("ex2_tops"),
        "alu_measured": alu,
        # fp16 tensor peak = the measured bf16 burst peak (same rate); tf32 = that x the nominal 1.1 / 2.25
        "f16_tflops": float(p.get("bf16_tflops", 1900.0)),
        "tf32_tflops": float(p.get("bf16_tflops", 1900.0)) * 1.1 / 2.25,
        "source": "MEASURED_PEAKS.json" if p else "fallback",
    }
    return _PEAKS


def roofline_for(kernel, fpp, bound, pairs, avg_ms, dtype, workload):
    """The roofline object of one kernel: algorithmic flop per pair x pairs per launch / launch time.
    A kernel whose time goes to instruction issue rather than to one pipe ("issue-tf32": the k-NN
    top-k, whose selection runs on the ALUs behind a tf32 contraction) is held against the issue rate
    instead: warp instructions per launch, counted by ncu on the current sources, over the launch time,
    against one warp instruction per clock in each of the SM's four schedulers. Without a count taken
    on the current sources it falls back to its algorithmic tf32 credit."""
    pk = peaks()
    if bound.startswith("issue-"):
        inst = issue_for(kernel, workload)
        tensor = roofline_for(kernel, fpp, "tensor-" + bound[len("issue-"):], pairs, avg_ms, dtype, workload)
        if inst is None:
            tensor["issue"] = None
            return tensor
        ach = inst / (avg_ms / 1e3) / 1e9
        peak = pk["sms"] * 4 * pk["sm_max_mhz"] * 1e6 / 1e9
        return {"kernel": kernel, "bound": "alu", "operands": "warp instructions, every pipe",
                "achieved": round(ach, 2), "peak": round(peak, 2), "unit": "Ginst/s", "frac": round(ach / peak, 4),
                "traffic": traffic_for(kernel, workload),
                "peak_source": (f"issue: {pk['sms']} SMs x 4 schedulers x 1 warp instruction per clock x "
                                f"{pk['sm_max_mhz']:.0f} MHz, derived"),
                "inst_per_launch": inst, "inst_per_pair": round(inst * 32 / pairs, 3),
                "pairs_per_launch": pairs, "avg_launch_us": round(avg_ms * 1e3, 2),
                "tensor_credit": {k: tensor[k] for k in ("achieved", "peak", "unit", "frac", "flop_per_pair")}}
    ach = fpp * pairs / (avg_ms / 1e3) / 1e12
    if bound == "tensor-f16":
        peak = pk["f16_tflops"]
        src = f"fp16 tensor (kind::f16 operands): measured bf16 {peak:.0f} TFLOP/s, same rate, of measured"
    elif bound == "tensor-tf32":
        peak = pk["tf32_tflops"]
        src = f"tf32 tensor: measured bf16 {pk['f16_tflops']:.0f} TFLOP/s x 1.1/2.25 (nominal tf32/bf16), of measured"
    elif dtype == "f64":
        peak = pk["fp64_tflops"]
        m = pk["alu_measured"] and pk["alu_measured"].get("fp64_fma_tflops")
        src = ("FP64 pipe: measured by this run's own fp64 FMA kernel (independent chains on every SM), of measured"
               if m else "FP64 pipe: nominal 1.25 TFLOP/s (no measurement available), of fallback")
    else:
        peak = pk["fp32_tflops"]
        m = pk["alu_measured"] and pk["alu_measured"].get("fp32_fma_tflops")
        src = ("FP32 pipe: measured by this run's own fp32 FMA kernel, of measured" if m else
               f"FP32 pipe: {pk['sms']} SMs x {FP32_LANES_PER_SM} lanes x 2 flop x {pk['sm_max_mhz']:.0f} MHz, derived")
    return {"kernel": kernel, "bound": "tensor" if bound.startswith("tensor") else "alu",
            "operands": bound[len("tensor-"):] if bound.startswith("tensor") else dtype,
            "achieved": round(ach, 3), "peak": round(peak, 2), "unit": "TFLOP/s", "frac": round(ach / peak, 4),
            "traffic": traffic_for(kernel, workload), "peak_source": src, "flop_per_pair": fpp,
            "pairs_per_launch": pairs, "avg_launch_us": round(avg_ms * 1e3, 2)}


# ------------------------------------------------------------------------------------------------
# per-kernel timing through libtp's own event timer
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
# clocks during a timed region
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
        win = [l for t, l in self.lines if self.t0 is not None and self.t0 <= t <= self.t1]
        sm, smax, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in win:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm) if sm else None,
                "power_w_median": statistics.median(power) if power else None}


# ------------------------------------------------------------------------------------------------
# workloads
# ------------------------------------------------------------------------------------------------


class Workload:
    """One hot-path step on device-resident inputs, plus the same step end to end from host buffers."""
    wid = 0
    name = ""
    dtype = "f32"
    pairs = 0
    flops_per_pair = {}  # per kernel name: (algorithmic flop per pair the launch processes, bound)
    steps = 20           # timed steps in the "workloads" object (the top-level line uses --steps)

    def config(self):
        return {"workload": self.name, "N": self.N, "M": getattr(self, "M", self.N), "D": self.D,
                "pairs_per_step": self.pairs}

    def step(self):
        raise NotImplementedError

    def e2e_step(self):
        raise NotImplementedError

    def oracle_sample(self, rows):
        """Time the oracle on `rows` sampled rows of this workload: (seconds, pairs, threads, text)."""
        raise NotImplementedError


def _sample_rows(n, count, seed):
    g = np.random.default_rng(seed)
    return np.sort(g.choice(n, size=min(count, n), replace=False))


class InfoNCE(Workload):
    """Workload 2: InfoNCE row logsumexp fwd + replay bwd, z [8192,64] fp32."""
    wid = 2
    cpu_rows = 1024

    def __init__(self, dev, over=None):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(2, **(over or {}))
        N, D = w["z"].shape
        self.N, self.D = N, D
        self.pairs = N * N
        self.name = f"infonce_logsumexp_f32_z{N}x{D}_fwd+bwd"
        self.score = ops.Score("linear", scale=w["scale"])
        self.z = w["z"].to(dev)
        self.gl = w["grad_lse"].to(dev)
        self.want = (True, True, False, False, False, False, False)
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
        # the row sweep credited with the recompute and dX, the column sweep with dY only; a kernel that
        # produces the whole backward (X = Y, one symmetric sweep) is credited with all of it.
        # "tensor-f16" kernels run the contraction on tcgen05 kind::f16 (scaled fp16 hi/lo split),
        # credited with the algorithmic flop against the fp16 tensor peak
        self.flops_per_pair = {"fwd_sweep_lse": (D2 + 3, "alu"), "bwd_sweep_lse_row": (D2 + 3 + D2, "alu"),
                               "bwd_sweep_lse_col": (D2, "alu"), "bwd_sweep_lse_sym": (D2 + 3 + D2 + D2, "alu"),
                               "lse_fwd_tc": (D2 + 3, "tensor-f16"), "lse_fwd_sym_tc": (D2 + 3, "tensor-f16"),
                               "lse_bwd_lin_tc": (D2 + 3 + D2 + D2, "tensor-f16"),
                               "lse_bwd_sym_tc": (D2 + 3 + D2 + D2, "tensor-f16")}
        # after the triangle sweep (lse_fwd_sym_tc: every ordered pair's term, each tile once for both of its
        # row blocks) lse_fwd_tc only merges the partials: no contraction to credit
        self.merged_by = {"lse_fwd_tc": "lse_fwd_sym_tc"}

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

    @staticmethod
    def oracle_sample(rows):
        return oracle_infonce(rows)


class RbfMatmul(Workload):
    """Workload 1: rbf kernel product K @ [V | 1] fp32, X, Y [1024,3], fwd + grads in X, Y, V."""
    wid = 1
    cpu_rows = 1024

    def __init__(self, dev, over=None):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(1, **(over or {}))
        self.N, self.D = w["X"].shape
        self.M = w["Y"].shape[0]
        self.C = w["V"].shape[1]
        self.pairs = self.N * self.M
        self.name = (f"rbf_kernel_matmul_f32_X{self.N}x{self.D}_Y{self.M}x{self.D}_V{self.M}x{self.C}_fwd+bwd")
        self.score = ops.Score("rbf", gamma=w["gamma"])
        self.X, self.Y, self.V, self.G = (w[k].to(dev) for k in ("X", "Y", "V", "grad_out"))
        self.host = {k: w[k].pin_memory() for k in ("X", "Y", "V", "grad_out")}
        self.dev_in = {k: torch.empty_like(v) for k, v in
                       (("X", self.X), ("Y", self.Y), ("V", self.V), ("grad_out", self.G))}
        self.out_h = torch.empty(self.N, self.C).pin_memory()
        self.h2d = sum(v.numel() * 4 for v in self.host.values())
        self.d2h = self.out_h.numel() * 4 + (self.N + self.M) * self.D * 4 + self.M * self.C * 4
        D, C = self.D, self.C
        # fwd 2D+2 (distance) + 1 (scale) + 2C; bwd recompute 2D+3, dS 2C, dV 2C, coef 2, dX 2D+1, dY 2D+1
        self.flops_per_pair = {"fwd_sweep_matmul": (2 * D + 3 + 2 * C, "alu"),
                               "bwd_sweep_matmul_row": (2 * D + 3 + 2 * C + 2 + 2 * D + 1, "alu"),
                               "bwd_sweep_matmul_col": (2 * C + 2 * D + 1, "alu")}
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

    @staticmethod
    def oracle_sample(rows):
        from lazy_score_matrix_gb300 import synth
        from oracle import oracle
        w = synth.workload(1)
        pb = oracle.Problem(w["X"], w["Y"], metric="rbf", gamma=w["gamma"])
        t0 = time.perf_counter()
        oracle.matmul(pb, w["V"])
        oracle.matmul_backward(pb, w["V"], w["grad_out"])
        return (time.perf_counter() - t0, w["X"].shape[0] * w["Y"].shape[0], oracle.get_threads(),
                "oracle fwd + bwd of the whole 1024 x 1024 problem")


class Knn(Workload):
    """Workload 3: exact k-NN top-16, X [65536,16] vs R [1048576,16] integers in [-8,8], fp32."""
    wid = 3
    steps = 10
    cpu_rows = 64

    def __init__(self, dev, over=None):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(3, **(over or {}))
        self.N, self.D = w["X"].shape
        self.M = w["R"].shape[0]
        self.k = w["k"]
        self.pairs = self.N * self.M
        self.name = f"knn_topk{self.k}_f32_X{self.N}x{self.D}_R{self.M}x{self.D}_fwd"
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
        # (and held against the issue rate, where its selection's instructions are counted)
        self.flops_per_pair = {"topk_sweep": (2 * self.D + 2, "alu"), "topk_tc": (2 * self.D + 2, "issue-tf32")}

    def step(self):
        return self.ops.pairwise_topk(self.X, self.R, self.score, self.k, False)

    def e2e_step(self):
        self.X_d.copy_(self.X_h, non_blocking=True)
        self.R_d.copy_(self.R_h, non_blocking=True)
        v, i = self.ops.pairwise_topk(self.X_d, self.R_d, self.score, self.k, False)
        self.v_h.copy_(v, non_blocking=True)
        self.i_h.copy_(i, non_blocking=True)

    @staticmethod
    def oracle_sample(rows):
        from lazy_score_matrix_gb300 import synth
        from oracle import oracle
        w = synth.workload(3)
        r = _sample_rows(w["X"].shape[0], rows, 33)
        pb = oracle.Problem(w["X"][r], w["R"], metric="sqeuclidean")
        t0 = time.perf_counter()
        oracle.topk(pb, w["k"], False)
        return (time.perf_counter() - t0, len(r) * w["R"].shape[0], oracle.get_threads(),
                f"oracle top-16 of {len(r)} seeded sampled rows against all 1048576 references")


class Attention(Workload):
    """Workload 4: softmax_matmul attention fp32, Q, K, V [16384,64], scale 1/8, fwd + grads."""
    wid = 4
    cpu_rows = 256
    mask = "all"

    def __init__(self, dev, over=None):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(4, **(over or {}))
        self.N, self.D = w["Q"].shape
        self.M = w["K"].shape[0]
        self.C = w["V"].shape[1]
        self.pairs = self.N * self.M
        self.name = f"attention_softmax_matmul_f32_QKV{self.N}x{self.D}_fwd+bwd"
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

    @classmethod
    def oracle_sample(cls, rows):
        """The oracle's forward and backward of `rows` seeded sampled query rows against all keys (the
        sub-problem of those rows). Under the causal mask: the causal problem of the first 32 `rows`
        queries and keys (a prefix of the workload, R (R + 1) / 2 kept pairs)."""
        from lazy_score_matrix_gb300 import synth
        from oracle import oracle
        w = synth.workload(4)
        if cls.mask == "causal":
            R = 32 * rows
            pb = oracle.Problem(w["Q"][:R], w["K"][:R], metric="linear", scale=w["scale"], pair_mask="causal")
            t0 = time.perf_counter()
            o, l = oracle.softmax_matmul(pb, w["V"][:R])
            oracle.softmax_matmul_backward(pb, w["V"][:R], o, l, w["grad_out"][:R])
            return (time.perf_counter() - t0, R * (R + 1) // 2, oracle.get_threads(),
                    f"oracle fwd + bwd of the causal problem of the first {R} queries and keys")
        r = _sample_rows(w["Q"].shape[0], rows, 44)
        pb = oracle.Problem(w["Q"][r], w["K"], metric="linear", scale=w["scale"])
        t0 = time.perf_counter()
        o, l = oracle.softmax_matmul(pb, w["V"])
        oracle.softmax_matmul_backward(pb, w["V"], o, l, w["grad_out"][r])
        return (time.perf_counter() - t0, len(r) * w["K"].shape[0], oracle.get_threads(),
                f"oracle fwd + bwd of {len(r)} seeded sampled query rows against all 16384 keys")


class CausalAttention(Attention):
    """Workload 6: workload 4 under the causal mask (key j <= query i), the attention of the Task Map's
    softmax_matmul(V, mask=tp.masks.causal()). Pairs are the kept ones, N (N + 1) / 2."""
    wid = 6
    mask = "causal"

    def __init__(self, dev, over=None):
        super().__init__(dev, over)
        self.name = f"causal_attention_softmax_matmul_f32_QKV{self.N}x{self.D}_fwd+bwd"
        self.score = self.ops.Score("linear", scale=self.score.scale, pair_mask="causal")
        self.pairs = self.N * (self.N + 1) // 2


class Svgd(Workload):
    """Workload 5: SVGD direction fp64, x [131072,8], score = -x, rbf gamma 0.1, one fused sweep."""
    wid = 5
    dtype = "f64"
    steps = 3
    cpu_rows = 512

    def __init__(self, dev, over=None):
        from lazy_score_matrix_gb300 import ops, synth
        self.ops = ops
        w = synth.workload(5, **(over or {}))
        self.N, self.D = w["x"].shape
        self.M = self.N
        self.gamma = w["gamma"]
        self.pairs = self.N * self.N
        self.name = f"svgd_direction_f64_x{self.N}x{self.D}_fwd"
        self.x, self.sc = w["x"].to(dev), w["score"].to(dev)
        self.x_h, self.s_h = w["x"].pin_memory(), w["score"].pin_memory()
        self.x_d, self.s_d = torch.empty_like(self.x), torch.empty_like(self.sc)
        self.phi_h = torch.empty(self.N, self.D, dtype=torch.float64).pin_memory()
        self.h2d = 2 * self.N * self.D * 8
        self.d2h = self.N * self.D * 8
        D = self.D
        # credited: the per-pair cost of one sweep with V = [score | x | 1] (distance 2D+2, -gamma scale 1,
        # accumulate 2(2D+1)); the kernel accumulates [score - 2 gamma x | 1] instead (2(D+1)), one fp64 exp
        self.flops_per_pair = {"fwd_sweep_svgd": (2 * D + 3 + 2 * (2 * D + 1), "alu")}

    def step(self):
        return self.ops.svgd_direction(self.x, self.sc, self.gamma)

    def e2e_step(self):
        self.x_d.copy_(self.x_h, non_blocking=True)
        self.s_d.copy_(self.s_h, non_blocking=True)
        phi = self.ops.svgd_direction(self.x_d, self.s_d, self.gamma)
        self.phi_h.copy_(phi, non_blocking=True)

    @staticmethod
    def oracle_sample(rows):
        from lazy_score_matrix_gb300 import synth
        from oracle import oracle
        w = synth.workload(5)
        r = _sample_rows(w["x"].shape[0], rows, 55)
        t0 = time.perf_counter()
        oracle.svgd_direction(w["x"][r], w["score"], w["gamma"], y=w["x"])
        return (time.perf_counter() - t0, len(r) * w["x"].shape[0], oracle.get_threads(),
                f"oracle SVGD direction of {len(r)} seeded sampled particles against all 131072")


WORKLOADS = {1: RbfMatmul, 2: InfoNCE, 3: Knn, 4: Attention, 5: Svgd, 6: CausalAttention}
# --small: the same kernels on reduced sizes, for profiler captures (a few hundred MB and launches of
# tens of milliseconds at most); never the benchmark's numbers. The k-NN case keeps the whole reference
# set and the length of a work unit (two column chunks of 524288 columns per row block), so its
# selection sees lists that fill and tighten as on the full workload, with 19/32 of the rows.
SMALL = {1: {}, 2: {}, 3: dict(N=38912, M=1048576), 4: dict(N=4096, M=4096), 5: dict(N=16384, M=16384),
         6: dict(N=4096, M=4096)}


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


def bench_workload(wl, steps, warmup, flush, world, dev):
    """Graph-replayed timed steps (value), a second eager pass with per-launch events (kernel durations
    and the roofline), and the end-to-end pass through the public API with host buffers."""
    from lazy_score_matrix_gb300 import _lib
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    graph = capture_step(wl)
    ms = time_steps(graph.replay if graph is not None else wl.step, steps, flush)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(ms, world, dev)
    # kernel durations: the same steps again, eagerly, with CUDA events around every launch on its stream
    # (events between launches would add gaps to the timed steps above)
    _lib.launch_count(reset=True)
    timer = KernelTimer(capacity=64 * steps + 64)
    with timer:
        time_steps(wl.step, steps, flush)
    launches = _lib.launch_count()
    torch.cuda.synchronize()
    # end to end: host buffers, copies inside the timed region
    for _ in range(2):
        wl.e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        wl.e2e_step()
        torch.cuda.current_stream().synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    ksum = timer.summary()
    dname, dstat = max(ksum.items(), key=lambda kv: kv[1]["total_ms"])
    merged_by = getattr(wl, "merged_by", {})
    credits = {k: v for k, v in wl.flops_per_pair.items() if not (k in merged_by and merged_by[k] in ksum)}
    credit = credits.get(dname)
    roof = None
    if credit is not None:
        roof = roofline_for(dname, credit[0], credit[1], wl.pairs, dstat["avg_ms"], wl.dtype, wl.name)
    total = sum(x["total_ms"] for x in ksum.values())
    return {
        "workload": wl.name, "value": round(whole_job_gpairs(world, wl.pairs, steps, ms / 1e3), 4), "unit": "Gpairs/s",
        "ms_per_step": round(ms / steps, 5), "steps": steps, "warmup": warmup, "dtype": wl.dtype,
        "config": wl.config(),
        "launch": "step captured once in a CUDA graph, replayed per timed step" if graph is not None else "eager",
        "roofline": roof,
        "kernels": {k: {"launches": v["launches"], "avg_us": round(v["avg_ms"] * 1e3, 2),
                        "share": round(v["total_ms"] / total, 4),
                        **({"roofline_frac": roofline_for(k, *credits[k], wl.pairs, v["avg_ms"], wl.dtype,
                                                          wl.name)["frac"]}
                           if k in credits else {})}
                    for k, v in sorted(ksum.items(), key=lambda kv: -kv[1]["total_ms"])},
        "gpu_launches": launches,
        "e2e": {"value": round(whole_job_gpairs(world, wl.pairs, steps, e2e_s), 4), "unit": "Gpairs/s",
                "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h},
        "_graph": graph,
    }


def clock_pass(wl, graph, dev, seconds=1.2):
    """Replays the step for at least `seconds` with nvidia-smi sampling the clocks every 50 ms: the clock
    record under load, and the throughput of that pass (L2 not flushed between replays)."""
    fn = graph.replay if graph is not None else wl.step
    fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    torch.cuda.synchronize()
    per = max(a.elapsed_time(b), 1e-3)
    n = max(int(seconds * 1e3 / per) + 1, 10)
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.4)
    clocks.t0 = time.time()
    a.record()
    for _ in range(n):
        fn()
    b.record()
    torch.cuda.synchronize()
    clocks.t1 = time.time()
    time.sleep(0.1)
    clocks.stop()
    ms = a.elapsed_time(b)
    res = clocks.result()
    res.update({"pass_s": round(ms / 1e3, 3), "pass_steps": n,
                "pass_value": round(wl.pairs * n / (ms / 1e3) / 1e9, 3),
                "how": "nvidia-smi every 50 ms during a >= 1 s pass of graph replays of the step"})
    return res


def gpu_arm(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks(None if args.no_peaks else dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 256 MB > 129 MB L2
    order = [args.workload] + [w for w in args.workloads if w != args.workload]
    results, top, top_wl = {}, None, None
    for wid in order:
        wl = WORKLOADS[wid](dev, SMALL[wid] if args.small else None)
        steps = args.steps if wid == args.workload else min(args.steps, wl.steps)
        r = bench_workload(wl, steps, args.warmup, flush, world, dev)
        graph = r.pop("_graph")
        if wid == args.workload:
            top, top_wl = r, wl
            r["clocks"] = clock_pass(wl, graph, dev) if rank == 0 and not args.no_clock_pass else None
        if rank == 0 and not args.no_cpu_baseline and wid in args.workloads:
            r["cpu_baseline"] = cpu_baseline(wl)
        results[str(wid)] = r
        del graph, wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    if rank != 0:
        return None
    pk = peaks()
    line = {
        "metric": METRIC, "value": top["value"], "unit": "Gpairs/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": top["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": top["dtype"], "data": "synthetic (seeded, shapes of the workload)",
        "config": dict(top["config"], l2="flushed before every timed step (256 MB write, untimed)",
                       parallelism="replicas" if world > 1 else "single GPU"),
        "impl": "libtp",
        "timing": {"launch": top["launch"],
                   "kernel_times": "CUDA events around every launch on its stream, in a second pass of the steps"},
        "roofline": top["roofline"],
        "kernels": top["kernels"],
        "gpu_launches": top["gpu_launches"],
        "e2e": top["e2e"],
        "clocks": top["clocks"],
        "peaks": {k: pk[k] for k in ("sms", "sm_max_mhz", "fp32_tflops", "fp32_derived_tflops", "fp64_tflops",
                                     "ex2_tops", "f16_tflops", "tf32_tflops", "hbm_gbs", "source")},
        "workloads": {k: v for k, v in results.items() if int(k) in args.workloads},
    }
    if "cpu_baseline" in top:
        line["cpu_baseline"] = top["cpu_baseline"]
    return line


def issue_for(kernel, workload):
    """Warp instructions per launch of `kernel` on `workload` (ncu smsp__inst_executed.sum) from the
    committed summary (lines `kernel workload count src=<hash>`), if taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "issue.txt")
    if not os.path.exists(path):
        return None
    cur = source_hash()
    for l in open(path):
        parts = l.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[3] == f"src={cur}":
            return float(parts[2])
    return None


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


# Traffic entries are keyed to a hash of every source the kernels are compiled from: all of csrc/ and the
# public header.
CSRC = os.path.join(ROOT, "lazy_score_matrix_gb300", "csrc")
HEADER = os.path.join(ROOT, "include", "tp.h")


def kernel_sources():
    return sorted([os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))] + [HEADER])


def source_hash():
    import hashlib
    h = hashlib.sha256()
    for path in kernel_sources():
        with open(path, "rb") as fh:
            h.update(os.path.basename(path).encode() + fh.read())
    return h.hexdigest()[:12]


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------------------


def oracle_infonce(rows: int, threads: int = 0):
    """Oracle forward + backward of the InfoNCE workload on its first `rows` rows against all columns.
    Returns (seconds, pairs, threads used, description)."""
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
    return dt, rows * N, used, f"oracle fwd + bwd of rows 0..{rows - 1} of z against all {N} columns"


def cpu_baseline(wl):
    """The oracle as it stands, on all host cores, on a bounded sample of the workload (a few seconds)."""
    from oracle import oracle
    oracle.set_threads(0)
    wl.oracle_sample(max(1, wl.cpu_rows // 8))  # warm-up (page-in, thread start)
    dt, pairs, used, what = wl.oracle_sample(wl.cpu_rows)
    return {"value": round(pairs / dt / 1e9, 6), "unit": "Gpairs/s", "cores": used, "kind": "oracle",
            "sample": f"{what}: {pairs} pairs in {dt:.2f} s"}


def reference_arm(args, rank, world):
    """The oracle timed as the reference implementation: each step a bounded row sample of the top-level
    workload (InfoNCE: 2048 of the 8192 rows against all columns, forward + backward)."""
    if rank != 0 or args.workload != 2:
        if rank == 0:
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the oracle on the "
                              "InfoNCE workload (--workload 2) only"}), flush=True)
        return None
    rows = 2048
    for _ in range(args.warmup):
        oracle_infonce(256)
    times, used, pairs = [], 0, 0
    for _ in range(args.steps):
        dt, pairs, used, _ = oracle_infonce(rows)
        times.append(dt)
    tot = sum(times)
    value = pairs * args.steps / tot / 1e9
    cfg = {"workload": "infonce_logsumexp_f32_z8192x64_fwd+bwd", "N": 8192, "M": 8192, "D": 64,
           "pairs_per_step": 8192 * 8192, "l2": "flushed before every timed step (256 MB write, untimed)",
           "parallelism": "replicas" if world > 1 else "single GPU"}
    return {"metric": METRIC, "value": round(value, 6), "unit": "Gpairs/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, shapes of the workload)",
            "config": cfg, "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "Gpairs/s", "cores": used, "kind": "oracle",
                             "sample": f"rows 0..{rows - 1} of the 8192 against all 8192 columns per step "
                                       f"(forward + backward); value = sampled pairs / time"},
            "e2e": {"value": round(value, 6), "unit": "Gpairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="libtp", choices=["libtp", "reference"])
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS))
    ap.add_argument("--workloads", default="1,2,3,4,5,6",
                    help="workloads of the line's 'workloads' object (comma-separated; empty for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true", help="reduced sizes of the same kernels (profiler captures)")
    ap.add_argument("--no-clock-pass", action="store_true", help="skip the >= 1 s clock-sampling pass")
    ap.add_argument("--no-peaks", action="store_true", help="skip the ALU peak measurement (derived peaks)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.workloads = [int(w) for w in args.workloads.split(",") if w.strip()]
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
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
