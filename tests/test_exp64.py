"""The fp64 exponential of the fp64 kernels (a table-driven method, csrc/tp_device.cuh) on the GPU,
through tp_selftest_exp64, against a correctly rounded reference: numpy's exp on the host, itself
checked here against 50-digit decimal arithmetic on a sample. Bound: 2 ulp on [-707, 709.78]
(the kernels' own bound is about 1.2 ulp); 0 below -707, +inf above 709.78."""
import ctypes
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

from lazy_score_matrix_gb300 import _lib

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _exp_gpu(x):
    lib = _lib.load()
    xd = torch.as_tensor(x, dtype=torch.float64).to(DEV)
    y = torch.empty_like(xd)
    _lib.check(lib.tp_selftest_exp64(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(y.data_ptr()), xd.numel(),
                                     ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)), "tp_selftest_exp64")
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _ulps(got, ref):
    return np.abs(got - ref) / np.array([math.ulp(v) for v in ref])


def test_exp64_within_two_ulp():
    rng = np.random.default_rng(64)
    x = np.concatenate([rng.uniform(-707, 709.78, 400_000), rng.uniform(-1, 1, 200_000),
                        rng.uniform(-40, 0, 200_000),  # the rbf kernel's range
                        np.ldexp(rng.uniform(-1, 1, 1000), -40), [0.0, -0.0, 1.0, -1.0, -706.999, 709.77]])
    ref = np.exp(x)
    # the host reference is correctly rounded on a sample (50-digit decimal)
    getcontext().prec = 50
    for v in x[::4001]:
        exact = Decimal(float(v)).exp()
        assert abs(Decimal(float(np.exp(v))) - exact) <= Decimal(math.ulp(float(exact))) * Decimal("0.51")
    u = _ulps(_exp_gpu(x), ref)
    assert u.max() <= 2.0, (u.max(), x[u.argmax()])


def test_exp64_range_ends():
    y = _exp_gpu(np.array([-707.5, -1e4, -np.inf, 709.9, 1e4, np.inf]))
    assert (y[:3] == 0).all()
    assert np.isposinf(y[3:]).all()
