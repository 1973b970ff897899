"""Pins of the oracle's column reductions and losses (CPU only): brute force, closed forms, invariants."""
import numpy as np
import pytest
import torch

from oracle import oracle_losses as OL


def _pts(seed, n, d, integers=False):
    g = torch.Generator().manual_seed(seed)
    if integers:
        return torch.randint(-4, 5, (n, d), generator=g).double()
    return torch.randn(n, d, generator=g, dtype=torch.float64)


def test_column_min_matches_dense_argmin_with_ties():
    X, Y = _pts(1, 37, 3, True), _pts(2, 23, 3, True)
    v, i = OL.column_min(X.numpy(), Y.numpy())
    D = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
    rv, ri = D.min(0)  # torch documents the first minimal index
    assert np.array_equal(v, rv.numpy()) and np.array_equal(i, ri.numpy())
    assert len(set(D.min(0).values.tolist())) < 23  # the data has ties


def test_mmd_biased_of_a_cloud_with_itself_is_zero():
    X = _pts(3, 40, 5).numpy()[None]
    assert abs(OL.mmd(X, X, "rbf", 0.3, unbiased=False)[0]) < 1e-13


def test_mmd_linear_closed_forms():
    X, Y = _pts(4, 30, 4).numpy(), _pts(5, 25, 4).numpy()
    mx, my = X.mean(0), Y.mean(0)
    assert abs(OL.mmd(X[None], Y[None], "linear", unbiased=False)[0] - ((mx - my) ** 2).sum()) < 1e-12
    m, n = len(X), len(Y)
    sx, sy = X.sum(0), Y.sum(0)
    u = ((sx @ sx - (X * X).sum()) / (m * (m - 1)) + (sy @ sy - (Y * Y).sum()) / (n * (n - 1)) - 2 * mx @ my)
    assert abs(OL.mmd(X[None], Y[None], "linear", unbiased=True)[0] - u) < 1e-12


def test_mmd_rbf_matches_dense_torch():
    X, Y = _pts(6, 20, 3), _pts(7, 15, 3)
    g = 0.7
    K = lambda A, B: torch.exp(-g * torch.cdist(A, B) ** 2)
    kxx, kyy, kxy = K(X, X), K(Y, Y), K(X, Y)
    u = ((kxx.sum() - kxx.diagonal().sum()) / (20 * 19) + (kyy.sum() - kyy.diagonal().sum()) / (15 * 14)
         - 2 * kxy.mean())
    assert abs(OL.mmd(X.numpy()[None], Y.numpy()[None], "rbf", g)[0] - u.item()) < 1e-12


def test_entropic_ot_one_point_each_is_the_cost():
    C = np.array([[2.5]])
    one = np.array([1.0])
    for eps in (0.01, 1.0):
        assert abs(OL.entropic_ot(C, one, one, eps, 3)[0] - 2.5) < 1e-12
    Cxx, Cyy = np.array([[0.25]]), np.array([[0.5]])
    assert abs(OL.sinkhorn_divergence(C, Cxx, Cyy, one, one, 0.3, 5) - (2.5 - 0.125 - 0.25)) < 1e-12


def test_sinkhorn_divergence_of_a_measure_with_itself_is_zero():
    X = _pts(8, 12, 2).numpy()
    C = 0.5 * OL.sqdist(X, X)
    a = np.full(12, 1 / 12)
    assert abs(OL.sinkhorn_divergence(C, C, C, a, a, 0.2, 60)) < 1e-12


def test_sinkhorn_plan_marginals_and_symmetry():
    X, Y = _pts(9, 15, 2).numpy(), _pts(10, 11, 2).numpy()
    a = np.random.default_rng(0).random(15) + 0.5
    a /= a.sum()
    b = np.full(11, 1 / 11)
    C = 0.5 * OL.sqdist(X, Y)
    eps = 0.5
    val, f, g = OL.entropic_ot(C, a, b, eps, 300)
    P = a[:, None] * b[None, :] * np.exp((f[:, None] + g[None, :] - C) / eps)
    assert np.allclose(P.sum(1), a, atol=1e-12)  # the last f update fits the rows exactly
    assert np.allclose(P.sum(0), b, atol=1e-9)   # converged columns
    val_t = OL.entropic_ot(C.T, b, a, eps, 300)[0]
    assert abs(val - val_t) < 1e-9
    # the dual value equals the primal <P, C> + eps KL(P | a b^T) at the fixed point
    kl = (P * np.log(P / (a[:, None] * b[None, :]))).sum()
    assert abs(val - ((P * C).sum() + eps * kl)) < 1e-9


def test_mask_on_exp_logsumexp_is_rejected():
    import lazy_score_matrix_gb300 as tp
    X = torch.zeros(4, 2)
    L = tp.lazy(X, X, "linear").exp().mask_columns(torch.tensor([True, False, True, True]))
    with pytest.raises(NotImplementedError):
        L.logsumexp(-1)
