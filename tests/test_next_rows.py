"""GPU parity of the column-direction reductions, boolean row/column masks, MMD statistics and the
Sinkhorn divergence (compositions of the fused consumers) against the oracle. A reduction over dim -2 of
S(X, Y) is the oracle's row reduction of the transposed problem S(Y, X) (every metric here is symmetric
in its two points). A boolean keep mask is the oracle's same-group pair mask with kept rows and columns
in group 0 and dropped ones in groups of their own, so the pair is removed from the consumer: the
library's lowering (a -inf bias for log-sum-exp, softmax and top-k, a zero weight for sums) is checked
against removal, not against itself. The MMD gradient alone is held against dense fp64 autograd."""
import numpy as np
import pytest
import torch

import lazy_score_matrix_gb300 as tp
from oracle import oracle_losses as OL
from tests._util import TOL_F32_FWD, TOL_F32_GRAD, TOL_F64, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _pts(seed, n, d, dtype=torch.float32, integers=False):
    g = torch.Generator().manual_seed(seed)
    if integers:
        return torch.randint(-8, 9, (n, d), generator=g).to(dtype)
    return torch.randn(n, d, generator=g, dtype=dtype)


@pytest.mark.parametrize("N,M", [(300, 700), (129, 33)])
def test_chamfer_min_both_directions_exact(oracle, N, M):
    X, Y = _pts(1, N, 16, integers=True), _pts(2, M, 16, integers=True)
    D = tp.lazy(X.to(DEV), Y.to(DEV), "sqeuclidean")
    v2, i2 = D.min(-2)
    rv, ri = OL.column_min(X.numpy(), Y.numpy())
    assert np.array_equal(v2.cpu().double().numpy(), rv) and np.array_equal(i2.cpu().numpy(), ri)
    v1, i1 = D.min(-1)
    ov, oi = oracle.topk(oracle.Problem(X, Y, metric="sqeuclidean"), 1)
    assert np.array_equal(v1.cpu().double().numpy(), ov[:, 0]) and np.array_equal(i1.cpu().numpy(), oi[:, 0])


def test_topk_over_columns_matches_oracle(oracle):
    X, Y = _pts(3, 90, 8, integers=True), _pts(4, 200, 8, integers=True)
    v, i = tp.lazy(X.to(DEV), Y.to(DEV), "sqeuclidean").topk(5, dim=-2, largest=False)
    ov, oi = oracle.topk(oracle.Problem(Y, X, metric="sqeuclidean"), 5)  # the transposed problem, rows = y
    assert np.array_equal(v.cpu().double().numpy(), ov.T) and np.array_equal(i.cpu().numpy(), oi.T)


@pytest.mark.parametrize("dtype,tol", [(torch.float32, TOL_F32_FWD), (torch.float64, TOL_F64)])
def test_logsumexp_sum_mean_over_columns(oracle, dtype, tol):
    X, Y = _pts(5, 150, 6, dtype), _pts(6, 260, 6, dtype)
    L = tp.lazy(X.to(DEV), Y.to(DEV), "rbf", gamma=0.4) * 2.0
    rows = oracle.Problem(X, Y, metric="rbf", gamma=0.4, scale=2.0)
    cols = oracle.Problem(Y, X, metric="rbf", gamma=0.4, scale=2.0)
    assert_close(L.logsumexp(dim=-2), oracle.logsumexp(cols), tol, "lse dim -2")
    assert_close(L.sum(-2), oracle.matmul(cols, np.ones((260, 1)))[:, 0], tol, "sum dim -2")
    assert_close(L.mean(-1), oracle.matmul(rows, np.ones((260, 1)))[:, 0] / 260, tol, "mean dim -1")
    assert_close(L.mean(-2), oracle.matmul(cols, np.ones((150, 1)))[:, 0] / 150, tol, "mean dim -2")


def _keep_groups(keep):
    """Group ids under which the oracle's same-group mask keeps exactly the pairs of kept points."""
    return np.where(np.asarray(keep), 0, -1).astype(np.int32)


def test_column_mask_on_every_row_consumer(oracle):
    X, Y, V = _pts(7, 120, 5), _pts(8, 300, 5), _pts(9, 300, 4)
    keep = torch.rand(300, generator=torch.Generator().manual_seed(10)) > 0.3
    L = tp.lazy(X.to(DEV), Y.to(DEV), "linear") * 0.5
    Lm = L.mask_columns(keep.to(DEV))
    pm = oracle.Problem(X, Y, metric="linear", scale=0.5, pair_mask="same_group",
                        row_group=np.zeros(120, np.int32), col_group=_keep_groups(keep))
    assert_close(Lm.logsumexp(-1), oracle.logsumexp(pm), TOL_F32_FWD, "masked lse")
    assert_close(Lm.softmax_matmul(V.to(DEV)), oracle.softmax_matmul(pm, V)[0], TOL_F32_FWD, "masked softmax")
    assert_close(Lm.matmul(V.to(DEV)), oracle.matmul(pm, V), TOL_F32_FWD, "masked K@V")
    assert_close(Lm.mean(-1), oracle.matmul(pm, np.ones((300, 1)))[:, 0] / int(keep.sum()), TOL_F32_FWD,
                 "masked mean")
    v, i = Lm.topk(3, largest=True)
    ov, oi = oracle.topk(pm, 3, largest=True)
    assert_close(v, ov, TOL_F32_FWD, "masked topk values")
    assert bool(keep[i.cpu()].all())
    # a row mask affects the reductions over columns: the transposed problem with the mask on its columns
    rkeep = torch.rand(120, generator=torch.Generator().manual_seed(11)) > 0.5
    pr = oracle.Problem(Y, X, metric="linear", scale=0.5, pair_mask="same_group",
                        row_group=np.zeros(300, np.int32), col_group=_keep_groups(rkeep))
    assert_close(L.mask_rows(rkeep.to(DEV)).logsumexp(dim=-2), oracle.logsumexp(pr), TOL_F32_FWD, "row-masked lse")


def test_column_mask_gradient_is_zero_on_masked_columns():
    X, Y = _pts(12, 64, 4).to(DEV).requires_grad_(), _pts(13, 80, 4).to(DEV).requires_grad_()
    keep = (torch.arange(80) % 3 != 0).to(DEV)
    tp.lazy(X, Y, "sqeuclidean").__mul__(-0.5).mask_columns(keep).logsumexp(-1).sum().backward()
    assert torch.all(Y.grad[~keep] == 0) and torch.all(Y.grad[keep].abs().sum(1) > 0)


@pytest.mark.parametrize("dtype,tol", [(torch.float64, 1e-10), (torch.float32, 2e-5)])
@pytest.mark.parametrize("unbiased", [True, False])
def test_mmd_statistics_matches_oracle(dtype, tol, unbiased):
    X = torch.stack([_pts(20, 500, 8, dtype), _pts(21, 500, 8, dtype) + 0.3])
    Y = torch.stack([_pts(22, 400, 8, dtype), _pts(23, 400, 8, dtype)])
    got = tp.mmd_statistics(X.to(DEV), Y.to(DEV), kernel="rbf", gamma=0.1, unbiased=unbiased).cpu().double()
    ref = torch.from_numpy(OL.mmd(X.double().numpy(), Y.double().numpy(), "rbf", 0.1, unbiased))
    # the statistic is a difference of O(1) means: absolute error against the size of those means
    assert float((got - ref).abs().max()) <= tol, (got, ref)


def test_mmd_gradient_matches_dense_autograd():
    X = _pts(24, 200, 6).to(DEV)[None].requires_grad_()
    Y = _pts(25, 150, 6).to(DEV)[None]
    tp.mmd_statistics(X, Y, kernel="rbf", gamma=0.2).sum().backward()
    Xd = X.detach().double().cpu().requires_grad_()
    Yd = Y.double().cpu()
    K = lambda A, B: torch.exp(-0.2 * ((A[:, None] - B[None]) ** 2).sum(-1))
    kxx, kyy, kxy = K(Xd[0], Xd[0]), K(Yd[0], Yd[0]), K(Xd[0], Yd[0])
    u = ((kxx.sum() - kxx.diagonal().sum()) / (200 * 199) + (kyy.sum() - kyy.diagonal().sum()) / (150 * 149)
         - 2 * kxy.mean())
    u.backward()
    assert_close(X.grad, Xd.grad, TOL_F32_GRAD, "mmd grad")


@pytest.mark.parametrize("dtype,tol", [(torch.float64, 1e-9), (torch.float32, 1e-4)])
def test_sinkhorn_divergence_matches_oracle(dtype, tol):
    X, Y = _pts(30, 200, 3, dtype), _pts(31, 150, 3, dtype) + 0.5
    a = torch.rand(200, generator=torch.Generator().manual_seed(32), dtype=dtype) + 0.5
    a = a / a.sum()
    b = torch.full((150,), 1.0 / 150, dtype=dtype)
    Xd, Yd = X.to(DEV), Y.to(DEV)
    C = lambda P, Q: tp.lazy(P, Q, "sqeuclidean") * 0.5
    got = tp.sinkhorn_divergence(C(Xd, Yd), C(Xd, Xd), C(Yd, Yd), a.to(DEV), b.to(DEV), epsilon=0.1, iters=50)
    Xn, Yn = X.double().numpy(), Y.double().numpy()
    ref = OL.sinkhorn_divergence(0.5 * OL.sqdist(Xn, Yn), 0.5 * OL.sqdist(Xn, Xn), 0.5 * OL.sqdist(Yn, Yn),
                                 a.double().numpy(), b.double().numpy(), 0.1, 50)
    assert abs(float(got) - ref) <= tol * max(1.0, abs(ref)), (float(got), ref)


def test_sinkhorn_gradient_is_the_plan():
    # d OT / d x_i = sum_j P_ij (x_i - y_j) for the cost |x - y|^2 / 2, with P the plan at the potentials
    X = _pts(33, 120, 2, torch.float64).to(DEV).requires_grad_()
    Y = _pts(34, 90, 2, torch.float64).to(DEV)
    a = torch.full((120,), 1 / 120, dtype=torch.float64, device=DEV)
    b = torch.full((90,), 1 / 90, dtype=torch.float64, device=DEV)
    eps = 0.2
    ot = tp.losses._entropic_ot(tp.lazy(X, Y, "sqeuclidean") * 0.5, a, b, eps, 80)
    ot.backward()
    Xn, Yn = X.detach().cpu().numpy(), Y.cpu().numpy()
    C = 0.5 * OL.sqdist(Xn, Yn)
    _, f, g = OL.entropic_ot(C, a.cpu().numpy(), b.cpu().numpy(), eps, 80)
    P = a.cpu().numpy()[:, None] * b.cpu().numpy()[None, :] * np.exp((f[:, None] + g[None, :] - C) / eps)
    ref = P.sum(1)[:, None] * Xn - P @ Yn
    assert_close(X.grad, torch.from_numpy(ref), 1e-8, "sinkhorn grad")


def test_minus_inf_column_bias_over_leading_columns(oracle):
    # a run of -inf scores at the start of a row's stream adds nothing (it once produced NaN)
    X, Y = _pts(40, 70, 5), _pts(41, 130, 5)
    b = torch.zeros(130)
    b[:45] = float("-inf")
    got = tp.lazy(X.to(DEV), Y.to(DEV), "linear").add_columns(b.to(DEV)).logsumexp(-1)
    want = oracle.logsumexp(oracle.Problem(X, Y, metric="linear", col_bias=b))
    assert_close(got, want, TOL_F32_FWD, "lse with -inf column bias")
