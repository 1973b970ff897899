"""The DRAM-traffic figures bench.py reports are keyed to a hash of the sources the kernels are compiled
from (CPU only): that set must hold the whole include closure of every kernel translation unit, so that a
change to any file a kernel is built from voids the recorded figures."""
import os
import re

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "lazy_score_matrix_gb300", "csrc")


def test_traffic_hash_covers_every_source_of_the_kernels():
    inc = os.path.join(os.path.dirname(CSRC), os.pardir, "include")
    units = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu")]
    seen, todo = set(), list(units)
    while todo:
        f = os.path.realpath(todo.pop())
        if f in seen:
            continue
        seen.add(f)
        for name in re.findall(r'#include "([^"]+)"', open(f).read()):
            todo.append(os.path.join(CSRC, name) if os.path.exists(os.path.join(CSRC, name)) else os.path.join(inc, name))
    assert seen <= {os.path.realpath(p) for p in bench.kernel_sources()}


def test_bench_reports_only_traffic_taken_on_the_current_sources():
    # every line of the committed summary carries the hash it was captured on: bench.py reports the lines
    # on the current sources and null for the others
    h = bench.source_hash()
    lines = [l.split() for l in open(os.path.join(bench.ROOT, "profiles", "traffic.txt")) if not l.startswith("#")]
    for kernel, workload, value, src in (l[:4] for l in lines if len(l) >= 4):
        want = float(value) if src == f"src={h}" else None
        if want is not None or not any(m[:2] == [kernel, workload] and m[3] == f"src={h}" for m in lines):
            assert bench.traffic_for(kernel, workload) == want


def test_bench_reports_only_instruction_counts_taken_on_the_current_sources():
    # the warp-instruction counts behind the issue-rate roofline follow the same rule as the traffic
    h = bench.source_hash()
    path = os.path.join(bench.ROOT, "profiles", "issue.txt")
    lines = [l.split() for l in open(path) if not l.startswith("#")] if os.path.exists(path) else []
    for kernel, workload, value, src in (l[:4] for l in lines if len(l) >= 4):
        want = float(value) if src == f"src={h}" else None
        if want is not None or not any(m[:2] == [kernel, workload] and m[3] == f"src={h}" for m in lines):
            assert bench.issue_for(kernel, workload) == want
    assert bench.issue_for("no_such_kernel", "no_such_workload") is None


def test_issue_roofline_falls_back_to_the_tensor_credit_without_counts(monkeypatch):
    monkeypatch.setattr(bench, "issue_for", lambda k, w: None)
    monkeypatch.setattr(bench, "traffic_for", lambda k, w: None)
    monkeypatch.setattr(bench, "_PEAKS", {"sms": 152, "sm_max_mhz": 2070.0, "f16_tflops": 1900.0,
                                           "tf32_tflops": 928.9, "fp32_tflops": 77.0, "fp64_tflops": 1.25,
                                           "alu_measured": None})
    r = bench.roofline_for("topk_tc", 34, "issue-tf32", 10 ** 9, 1.0, "f32", "w")
    assert r["bound"] == "tensor" and r["operands"] == "tf32" and r["issue"] is None
    monkeypatch.setattr(bench, "issue_for", lambda k, w: 2.0e8)
    r = bench.roofline_for("topk_tc", 34, "issue-tf32", 10 ** 9, 1.0, "f32", "w")
    peak = 152 * 4 * 2070e6 / 1e9
    assert r["bound"] == "alu" and r["unit"] == "Ginst/s"
    assert abs(r["achieved"] - 200.0) < 1e-6 and abs(r["peak"] - round(peak, 2)) < 1e-6
    assert abs(r["inst_per_pair"] - 6.4) < 1e-9 and r["tensor_credit"]["unit"] == "TFLOP/s"
