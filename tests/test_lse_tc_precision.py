"""GPU parity of the tensor-core InfoNCE log-sum-exp (forward, and the symmetric backward of a linear
score without exp) on inputs whose magnitudes spread across 2^20 inside one matrix (torchpairwise guide
"Using Torchpairwise in Models", Task Map: InfoNCE row, S = lazy(z, z) / t, logsumexp(-1,
exclude_self=True)). The backward gives z ONE power of two and the coefficient matrix kappa one power
of two fixed from max|g|, then splits every element into fp16 hi + lo: rows and upstream gradients far
below the largest keep fewer bits. Held to the fp32 tolerances, or to twice what a plain dense fp32
evaluation reaches on the same inputs where that is larger (tests/_plain.py)."""
import ctypes

import pytest
import torch

from lazy_score_matrix_gb300 import _lib, ops
from lazy_score_matrix_gb300.ops import Score
from tests._plain import TC_SLACK, Plain, achievable
from tests._util import TOL_F32_FWD, TOL_F32_GRAD, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _pow2_rows(seed, n, lo):
    g = torch.Generator().manual_seed(seed)
    return torch.pow(2.0, torch.randint(lo, 1, (n,), generator=g).float())


def _kernels(fn):
    lib = _lib.load()
    torch.cuda.synchronize()
    _lib.check(lib.tp_timer_start(64), "tp_timer_start")
    fn()
    n = lib.tp_timer_stop()
    names = set()
    name, ms = ctypes.c_char_p(), ctypes.c_float()
    for i in range(n):
        _lib.check(lib.tp_timer_read(i, ctypes.byref(name), ctypes.byref(ms)), "tp_timer_read")
        names.add(name.value.decode())
    return names


@pytest.mark.parametrize("spread", ["rows", "grad", "both"])
@pytest.mark.parametrize("N", [700, 2100])
def test_infonce_mixed_magnitudes(oracle, N, spread):
    g0 = torch.Generator().manual_seed(500 + N)
    z = torch.nn.functional.normalize(torch.randn(N, 64, generator=g0), dim=1)
    if spread in ("rows", "both"):
        z = z * _pow2_rows(501 + N, N, -20)[:, None]
    gl = torch.full((N,), -1.0 / N)
    if spread in ("grad", "both"):
        gl = gl * _pow2_rows(502 + N, N, -20)
    scale = 1 / 0.07
    zd = z.to(DEV)
    sc = Score("linear", scale=scale)
    holder = {}

    def run():
        holder["lse"] = ops.pairwise_logsumexp(zd, zd, sc, True)
        holder["g"] = ops.pairwise_logsumexp_backward(zd, zd, sc, holder["lse"], gl.to(DEV), True, same=True)

    names = _kernels(run)
    assert {"lse_fwd_tc", "lse_bwd_lin_tc"} <= names, names
    pb = oracle.Problem(z, z, metric="linear", scale=scale)
    ol = oracle.logsumexp(pb, True)
    og = oracle.logsumexp_backward(pb, ol, gl, True)
    pl = Plain(z, z, metric="linear", scale=scale, same=True)
    p_lse = pl.logsumexp(True)
    want = og["dX"] + og["dY"]
    assert_close(holder["lse"], ol, achievable(p_lse.detach(), ol, TOL_F32_FWD, slack=TC_SLACK), f"lse {spread}")
    assert_close(holder["g"]["dX"], want, achievable(pl.grads(p_lse, gl)["dX"], want, TOL_F32_GRAD, slack=TC_SLACK),
                 f"z.grad {spread}")


@pytest.mark.parametrize("scale", [1 / 0.07, 60.0])
@pytest.mark.parametrize("N", [129, 1000, 4097])
@pytest.mark.parametrize("excl", [True, False])
def test_infonce_forward_triangle_and_fallback(oracle, N, scale, excl):
    """X = Y, linear score without exp: the forward sweeps the upper triangle of tiles against one fixed
    offset M = |scale| log2(e) max|z|^2 when 2 M <= 120 (scale 1/0.07 on unit rows: M = 20.6), and falls
    back to the full sweep with running maxima otherwise (scale 60: M = 86.6). Both are held to the fp32
    forward tolerance against the oracle, on row counts with a ragged last block."""
    g0 = torch.Generator().manual_seed(900 + N)
    z = torch.nn.functional.normalize(torch.randn(N, 64, generator=g0), dim=1)
    zd = z.to(DEV)
    sc = Score("linear", scale=scale)
    holder = {}
    names = _kernels(lambda: holder.setdefault("lse", ops.pairwise_logsumexp(zd, zd, sc, excl)))
    assert {"lse_fwd_sym_tc", "lse_fwd_tc"} <= names, names
    pb = oracle.Problem(z, z, metric="linear", scale=scale)
    want = oracle.logsumexp(pb, excl)
    plain = Plain(z, z, metric="linear", scale=scale, same=True).logsumexp(excl)
    assert_close(holder["lse"], want, achievable(plain.detach(), want, TOL_F32_FWD, slack=TC_SLACK),
                 f"lse N={N} scale={scale} exclude_self={excl}")


@pytest.mark.parametrize("N", [12288, 12289])
def test_infonce_forward_triangle_cap(oracle, N):
    """The triangle forward runs up to 96 row blocks (N = 12288) and the full sweep beyond (N = 12289),
    where the triangle's column partials would outgrow their cap; both against the oracle, unit rows,
    scale 1/0.07, exclude_self."""
    g0 = torch.Generator().manual_seed(1200 + N)
    z = torch.nn.functional.normalize(torch.randn(N, 64, generator=g0), dim=1)
    zd = z.to(DEV)
    sc = Score("linear", scale=1 / 0.07)
    holder = {}
    names = _kernels(lambda: holder.setdefault("lse", ops.pairwise_logsumexp(zd, zd, sc, True)))
    assert ("lse_fwd_sym_tc" in names) == (N <= 96 * 128), names
    want = oracle.logsumexp(oracle.Problem(z, z, metric="linear", scale=1 / 0.07), True)
    plain = Plain(z, z, metric="linear", scale=1 / 0.07, same=True).logsumexp(True)
    assert_close(holder["lse"], want, achievable(plain.detach(), want, TOL_F32_FWD, slack=TC_SLACK),
                 f"lse N={N}")
