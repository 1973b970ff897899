"""The device-side status path on the GPU (failure detection without a GPU fault): a bounded wait that
runs out records its code in the library's device error word, the kernel returns, tp_device_status
reports TP_ERR_TIMEOUT after a synchronise, a reset clears it, and the context stays usable for the
next call. Host-side fault injection (TP_FAULT_INJECT) fails an entry before it launches anything.
The status convention follows the torchpairwise guide's "What to Check" section (solvers report a
status beside their result)."""
import ctypes

import pytest
import torch

from lazy_score_matrix_gb300 import _lib, ops, synth
from lazy_score_matrix_gb300.ops import Score
from tests._util import TOL_F32_FWD, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def test_bounded_wait_timeout_is_reported_and_cleared(oracle):
    lib = _lib.load()
    torch.cuda.synchronize()
    lib.tp_device_status(1)  # start from a clear word
    assert lib.tp_device_status(0) == _lib.TP_OK
    _lib.check(lib.tp_selftest_bounded_wait(1_000_000, _stream()), "tp_selftest_bounded_wait")  # 1 ms
    torch.cuda.synchronize()
    assert lib.tp_device_status(0) == _lib.TP_ERR_TIMEOUT
    msg = lib.tp_last_error()
    assert b"self-test" in msg and b"site code 1" in msg, msg
    # sticky until reset; the reset call still reports what it found
    assert lib.tp_device_status(1) == _lib.TP_ERR_TIMEOUT
    assert lib.tp_device_status(0) == _lib.TP_OK
    # the context is usable: a tensor-core call right after matches the oracle and leaves the word clear
    w = synth.workload(2, N=600)
    z = w["z"].to(DEV)
    lse = ops.pairwise_logsumexp(z, z, Score("linear", scale=w["scale"]), True)
    torch.cuda.synchronize()
    assert lib.tp_device_status(0) == _lib.TP_OK
    ref = oracle.logsumexp(oracle.Problem(w["z"], w["z"], metric="linear", scale=w["scale"]), True)
    assert_close(lse, ref, TOL_F32_FWD, "lse after the self-test")


def test_first_code_is_kept(oracle):
    lib = _lib.load()
    torch.cuda.synchronize()
    lib.tp_device_status(1)
    for _ in range(2):
        _lib.check(lib.tp_selftest_bounded_wait(100_000, _stream()), "tp_selftest_bounded_wait")
    torch.cuda.synchronize()
    assert lib.tp_device_status(1) == _lib.TP_ERR_TIMEOUT
    assert b"site code 1" in lib.tp_last_error()
    assert lib.tp_device_status(0) == _lib.TP_OK


def test_fault_injection_launches_nothing(monkeypatch):
    lib = _lib.load()
    w = synth.workload(2, N=300)
    z = w["z"].to(DEV)
    sc = Score("linear", scale=w["scale"])
    before = ops.pairwise_logsumexp(z, z, sc, True)
    torch.cuda.synchronize()
    monkeypatch.setenv("TP_FAULT_INJECT", "pairwise_logsumexp")
    _lib.launch_count(reset=True)
    out = torch.full_like(before, 7.0)
    pairs = _lib.tp_pairs(_lib.TP_F32, 300, 300, 64, z.data_ptr(), z.data_ptr())
    score = _lib.tp_score(_lib.METRICS["linear"], 1.0, w["scale"], 0, None, None, None, None)
    need = lib.tp_workspace_size(b"pairwise_logsumexp", ctypes.byref(pairs), 0, 0)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=DEV)
    st = lib.tp_pairwise_logsumexp(ctypes.byref(pairs), ctypes.byref(score), 1, ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(ws.data_ptr()), need, _stream())
    torch.cuda.synchronize()
    assert st == _lib.TP_ERR_CUDA and b"fault injected" in lib.tp_last_error()
    assert _lib.launch_count() == 0
    assert torch.all(out == 7.0)
    # other entries are unaffected, and clearing the variable restores this one
    g = ops.pairwise_logsumexp_backward(z, z, sc, before, w["grad_lse"].to(DEV), True, same=True)
    assert torch.isfinite(g["dX"]).all()
    monkeypatch.delenv("TP_FAULT_INJECT")
    again = ops.pairwise_logsumexp(z, z, sc, True)
    assert torch.equal(again, before)
