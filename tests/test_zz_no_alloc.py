"""tp_pairwise_logsumexp_noalloc, called through the C ABI, against tp_pairwise_logsumexp.

The no-alloc entry point serves callers that cannot allocate device memory when they need the
result (inside another allocator's critical section, in real-time loops that forbid allocation
after start-up, in hosts that cannot own a workspace); it takes no workspace and uses a fixed array
of the library's own device memory instead. Its results must match the workspace entry point's
within the fp32 forward tolerance, on two calls in a row (the second finds the first call's
contents in the shared array). This file is collected last so that a stop at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from lazy_score_matrix_gb300 import _lib, ops, synth
from tests._util import TOL_F32_FWD, TOL_F64, assert_close

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, z, scale, exclude_self):
    N, D = z.shape
    dt = _lib.TP_F64 if z.dtype == torch.float64 else _lib.TP_F32
    pairs = _lib.tp_pairs(dt, N, N, D, z.data_ptr(), z.data_ptr())
    score = _lib.tp_score(_lib.METRICS["linear"], 1.0, scale, 0, None, None, None, None)
    lse = torch.empty(N, dtype=z.dtype, device=z.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream(z.device).cuda_stream)
    st = lib.tp_pairwise_logsumexp_noalloc(ctypes.byref(pairs), ctypes.byref(score), int(exclude_self),
                                           ctypes.c_void_p(lse.data_ptr()), stream)
    assert st == _lib.TP_OK, lib.tp_last_error()
    return lse


@pytest.mark.parametrize("N", [8192, 700])
def test_noalloc_matches_workspace_entry_twice(N):
    lib = _lib.load()
    dev = torch.device("cuda:0")
    w = synth.workload(2, N=N)
    z = w["z"].to(dev)
    ref = ops.pairwise_logsumexp(z, z, ops.Score("linear", scale=w["scale"]), True)
    # the shape does need scratch: the entry point really uses its fixed array
    assert lib.tp_workspace_size(b"pairwise_logsumexp", ctypes.byref(
        _lib.tp_pairs(_lib.TP_F32, N, N, 64, z.data_ptr(), z.data_ptr())), 0, 0) > 0
    first = _call_noalloc(lib, z, w["scale"], True)
    second = _call_noalloc(lib, z, w["scale"], True)
    torch.cuda.synchronize()
    assert_close(first, ref, TOL_F32_FWD, "first call")
    assert_close(second, ref, TOL_F32_FWD, "second call")


@pytest.mark.parametrize("dtype,D", [(torch.float64, 64), (torch.float32, 16)])
def test_noalloc_streamed_path_twice(dtype, D):
    """Shapes the streamed (SIMT) log-sum-exp serves, whose split partial states use the fixed array."""
    lib = _lib.load()
    dev = torch.device("cuda:0")
    N = 5000
    g = torch.Generator().manual_seed(901 + D)
    z = torch.nn.functional.normalize(torch.randn(N, D, generator=g, dtype=dtype), dim=1).to(dev)
    ref = ops.pairwise_logsumexp(z, z, ops.Score("linear", scale=1 / 0.07), True)
    assert lib.tp_workspace_size(b"pairwise_logsumexp", ctypes.byref(
        _lib.tp_pairs(_lib.TP_F64 if dtype == torch.float64 else _lib.TP_F32, N, N, D, z.data_ptr(), z.data_ptr())),
        0, 0) > 0
    tol = TOL_F64 if dtype == torch.float64 else TOL_F32_FWD
    for call in ("first", "second"):
        got = _call_noalloc(lib, z, 1 / 0.07, True)
        torch.cuda.synchronize()
        assert_close(got, ref, tol, f"{call} call")
