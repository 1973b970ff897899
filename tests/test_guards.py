"""Memory-safety and determinism checks of every entry point on the GPU, in place of a sanitizer (which is
not available here): every output and the workspace are placed inside larger buffers whose guard bytes
(4 KiB before and after, a fixed pattern) must come back untouched, every output element must have been
written (the interior starts as a canary pattern that no result takes), and a second call on fresh
buffers must give bitwise the same results (no race: the kernels use no floating-point atomics). Shapes
are ragged (several tiles and a partial one), on both the tensor-core and the streamed (SIMT) paths.
"""
import ctypes

import numpy as np
import pytest
import torch

from lazy_score_matrix_gb300 import ops
from lazy_score_matrix_gb300.ops import Score

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = 4096
GUARD_BYTE = 0xA5
CANARY_BYTE = 0x7F  # fp32 3.39e38, fp64 1.4e306, int64 9.2e18: values no consumer returns here


class Guarded:
    """Allocation hooks for ops._Call: outputs and workspaces inside guarded buffers."""

    def __init__(self):
        self.bufs = []  # (buffer, offset, nbytes, is_output, tensor)

    def alloc(self, nbytes, dtype, shape, output):
        raw = torch.full((GUARD + nbytes + GUARD + 256,), GUARD_BYTE, dtype=torch.uint8, device=DEV)
        off = GUARD + (-(raw.data_ptr() + GUARD) % 256)
        raw[off:off + nbytes] = CANARY_BYTE if output else 0
        view = raw[off:off + nbytes].view(dtype).view(*shape)
        assert view.data_ptr() % 256 == 0
        self.bufs.append((raw, off, nbytes, output, view))
        return view

    def check(self, what):
        torch.cuda.synchronize()
        for raw, off, nbytes, output, view in self.bufs:
            host = raw.cpu().numpy()
            assert (host[:off] == GUARD_BYTE).all(), f"{what}: write before a buffer"
            assert (host[off + nbytes:] == GUARD_BYTE).all(), f"{what}: write past a buffer"
            if output:
                body = host[off:off + nbytes].reshape(-1, view.element_size())
                left = (body == CANARY_BYTE).all(axis=1)
                assert not left.any(), f"{what}: {int(left.sum())} output elements never written"


@pytest.fixture
def guarded(monkeypatch):
    g = Guarded()

    def empty(self, *shape, dtype=None):
        dt = dtype or self.dtype
        n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        return g.alloc(n, dt, shape, True)

    def workspace(self, entry, C=0, k=0):
        n = self.lib.tp_workspace_size(entry.encode(), ctypes.byref(self.pairs), int(C), int(k))
        assert n != ctypes.c_size_t(-1).value
        if n == 0:
            return None, 0
        return g.alloc(n, torch.uint8, (n,), False), n

    monkeypatch.setattr(ops._Call, "empty", empty)
    monkeypatch.setattr(ops._Call, "workspace", workspace)
    return g


def _n(seed, shape, dtype=torch.float32):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed), dtype=dtype).to(DEV)


def _twice(guarded, fn, what):
    a = fn()
    guarded.check(what)
    b = fn()
    guarded.check(what + " (second call)")
    fa = a if isinstance(a, (tuple, list)) else [a]
    fb = b if isinstance(b, (tuple, list)) else [b]
    for x, y in zip(fa, fb):
        if isinstance(x, dict):
            for k in x:
                if x[k] is not None:
                    assert torch.equal(x[k], y[k]), f"{what}: {k} differs between two calls"
        else:
            assert torch.equal(x, y), f"{what}: results differ between two calls"


SHAPES = [(300, 517), (257, 129), (1, 77)]


@pytest.mark.parametrize("dt", [torch.float32, torch.float64])
@pytest.mark.parametrize("N,M", SHAPES)
def test_matmul_displacement_guarded(guarded, N, M, dt):
    X, Y, V, G = _n(1, (N, 3), dt), _n(2, (M, 3), dt), _n(3, (M, 5), dt), _n(4, (N, 5), dt)
    sc = Score("rbf", gamma=0.4, row_bias=_n(5, (N,), dt), col_weight=_n(6, (M,), dt).abs() + 0.5)
    _twice(guarded, lambda: ops.pairwise_matmul(X, Y, V, sc), "matmul")
    _twice(guarded, lambda: ops.pairwise_matmul_backward(X, Y, V, sc, G), "matmul backward")
    _twice(guarded, lambda: ops.pairwise_displacement(X, Y, sc), "displacement")
    _twice(guarded, lambda: ops.pairwise_displacement_backward(X, Y, sc, _n(7, (N, 3), dt)), "displacement backward")
    _twice(guarded, lambda: ops.svgd_direction(X, -X, 0.3), "svgd")


@pytest.mark.parametrize("D,metric", [(64, "linear"), (64, "sqeuclidean"), (16, "rbf")])
@pytest.mark.parametrize("N,M", SHAPES)
def test_logsumexp_guarded(guarded, N, M, D, metric):
    X, Y = _n(11, (N, D)), _n(12, (M, D))
    sc = Score(metric, scale=0.1 if metric == "linear" else -0.05, gamma=0.05)
    _twice(guarded, lambda: ops.pairwise_logsumexp(X, Y, sc), "lse")
    lse = ops.pairwise_logsumexp(X, Y, sc)
    _twice(guarded, lambda: ops.pairwise_logsumexp_backward(X, Y, sc, lse, _n(13, (N,))), "lse backward")
    # the same points, exclude_self, one summed gradient (the InfoNCE path)
    Z = torch.nn.functional.normalize(X, dim=1)
    sz = Score("linear", scale=1 / 0.07)
    _twice(guarded, lambda: ops.pairwise_logsumexp(Z, Z, sz, True), "lse same")
    lz = ops.pairwise_logsumexp(Z, Z, sz, True)
    _twice(guarded, lambda: ops.pairwise_logsumexp_backward(Z, Z, sz, lz, _n(14, (N,)), True, same=True),
           "lse backward same")


@pytest.mark.parametrize("mask", ["all", "causal", "band"])
@pytest.mark.parametrize("D,C", [(64, 64), (16, 8)])
@pytest.mark.parametrize("N,M", SHAPES)
def test_softmax_matmul_guarded(guarded, N, M, D, C, mask):
    Q, K, V, G = _n(21, (N, D)), _n(22, (M, D)), _n(23, (M, C)), _n(24, (N, C))
    sc = Score("linear", scale=D ** -0.5, pair_mask=mask, band=9)
    _twice(guarded, lambda: ops.pairwise_softmax_matmul(Q, K, V, sc), "softmax")
    out, lse = ops.pairwise_softmax_matmul(Q, K, V, sc)
    _twice(guarded, lambda: ops.pairwise_softmax_matmul_backward(Q, K, V, sc, out, lse, G), "softmax backward")


@pytest.mark.parametrize("dt,D", [(torch.float32, 16), (torch.float32, 64), (torch.float64, 5)])
@pytest.mark.parametrize("N,M", SHAPES)
def test_topk_guarded(guarded, N, M, D, dt):
    g = torch.Generator().manual_seed(31)
    X = torch.randint(-4, 5, (N, D), generator=g).to(dt).to(DEV)
    Y = torch.randint(-4, 5, (M, D), generator=g).to(dt).to(DEV)
    k = min(16, M)
    sc = Score("sqeuclidean")
    _twice(guarded, lambda: ops.pairwise_topk(X, Y, sc, k, False), "topk")
    v, i = ops.pairwise_topk(X, Y, sc, k, False)
    _twice(guarded, lambda: ops.pairwise_topk_backward(X, Y, sc, k, i, _n(32, (N, k), dt)), "topk backward")
