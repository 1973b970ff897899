"""GPU parity when X is a prefix view of Y: the same device pointer with fewer rows (X = Z[:N], Y = Z,
N < M). The two point sets then share a pointer but are not the same set, so the tensor-core paths
must keep separate copies of their rows (a workspace copy of X holds only N rows). Log-sum-exp
(torchpairwise guide "Using Torchpairwise in Models", Task Map: InfoNCE row) and top-k (k-NN row),
against the oracle."""
import numpy as np
import pytest
import torch

from lazy_score_matrix_gb300 import ops
from lazy_score_matrix_gb300.ops import Score
from tests._util import TOL_F32_FWD, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _z(seed, n, d):
    g = torch.Generator().manual_seed(seed)
    return torch.nn.functional.normalize(torch.randn(n, d, generator=g), dim=1)


@pytest.mark.parametrize("N,M", [(100, 700), (300, 517), (129, 4000)])
@pytest.mark.parametrize("metric", ["linear", "sqeuclidean"])
def test_logsumexp_prefix_view(oracle, N, M, metric):
    Z = _z(7 + N, M, 64)
    Zd = Z.to(DEV)
    X, Y = Zd[:N], Zd
    assert X.data_ptr() == Y.data_ptr()
    scale = 1 / 0.07 if metric == "linear" else -2.0
    lse = ops.pairwise_logsumexp(X, Y, Score(metric, scale=scale), False)
    want = oracle.logsumexp(oracle.Problem(Z[:N], Z, metric=metric, scale=scale), False)
    assert_close(lse, want, TOL_F32_FWD, f"lse prefix {N}x{M}")


@pytest.mark.parametrize("N,M", [(100, 700), (300, 517), (129, 4000)])
@pytest.mark.parametrize("D", [16, 64])
def test_topk_prefix_view(oracle, N, M, D):
    g = torch.Generator().manual_seed(11 + N)
    Z = torch.randint(-8, 9, (M, D), generator=g).float()
    Zd = Z.to(DEV)
    v, i = ops.pairwise_topk(Zd[:N], Zd, Score("sqeuclidean"), 16, False)
    ov, oi = oracle.topk(oracle.Problem(Z[:N], Z, metric="sqeuclidean"), 16, False)
    np.testing.assert_array_equal(i.cpu().numpy(), oi)
    np.testing.assert_array_equal(v.cpu().double().numpy(), ov)
