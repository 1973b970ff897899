"""Losses built on the fused consumers: MMD two-sample statistics and the Sinkhorn divergence.

torchpairwise guide "Using Torchpairwise in Models", Task Map: "MMD loss, two-sample test"
(``mmd_statistics(X[None], Y[None], kernel="rbf", gamma=g)``, unbiased by default, one point cloud per
batch entry) and "Optimal transport loss" (``sinkhorn_divergence(C_xy, C_xx, C_yy, a, b, epsilon=e)``
on any lazy cost). Each is a short composition of lazy score matrices and their fused consumers
(K @ ones, row and column log-sum-exp); no [n, n] matrix is formed.
"""
from __future__ import annotations

import torch

from .lazy import LazyScores, lazy


def _kernel(X: torch.Tensor, Y: torch.Tensor, kernel: str, gamma: float) -> LazyScores:
    if kernel == "rbf":
        return lazy(X, Y, "rbf", gamma=gamma)
    if kernel == "linear":
        return lazy(X, Y, "linear")
    raise ValueError(f"mmd_statistics: unknown kernel {kernel!r} (rbf or linear)")


def _self_kernel_sum(X: torch.Tensor, kernel: str) -> torch.Tensor:
    """sum_i k(x_i, x_i): m for rbf (k(x, x) = 1), sum_i |x_i|^2 for linear."""
    if kernel == "rbf":
        return torch.tensor(float(X.shape[0]), dtype=X.dtype, device=X.device)
    return (X * X).sum()


def mmd_statistics(X: torch.Tensor, Y: torch.Tensor, kernel: str = "rbf", gamma: float = 1.0,
                   unbiased: bool = True) -> torch.Tensor:
    """Squared maximum mean discrepancy between the point clouds X[b] [m, D] and Y[b] [n, D], per batch
    entry b: X [B, m, D], Y [B, n, D] -> [B].

    unbiased (default): the U-statistic, whose within-cloud sums leave out the pairs i = i':
        sum_{i != i'} k(x_i, x_i') / (m (m - 1)) + sum_{j != j'} k(y_j, y_j') / (n (n - 1))
        - 2 sum_{i, j} k(x_i, y_j) / (m n)          (m, n >= 2)
    biased: the V-statistic, every sum over all pairs and divided by m^2, n^2 and m n.
    Each sum is one fused K @ ones sweep; gradients flow to X and Y through it."""
    if X.dim() != 3 or Y.dim() != 3:
        raise ValueError("mmd_statistics: X and Y are batches of point clouds [B, m, D] and [B, n, D]")
    out = []
    for b in range(X.shape[0]):
        x, y = X[b], Y[b]
        m, n = x.shape[0], y.shape[0]
        kxx = _kernel(x, x, kernel, gamma).sum(-1).sum()
        kyy = _kernel(y, y, kernel, gamma).sum(-1).sum()
        kxy = _kernel(x, y, kernel, gamma).sum(-1).sum()
        if unbiased:
            if m < 2 or n < 2:
                raise ValueError("mmd_statistics: the unbiased statistic needs at least two points per cloud")
            v = ((kxx - _self_kernel_sum(x, kernel)) / (m * (m - 1)) + (kyy - _self_kernel_sum(y, kernel)) / (n * (n - 1))
                 - 2.0 * kxy / (m * n))
        else:
            v = kxx / (m * m) + kyy / (n * n) - 2.0 * kxy / (m * n)
        out.append(v)
    return torch.stack(out)


def _entropic_ot(C: LazyScores, a: torch.Tensor, b: torch.Tensor, epsilon: float, iters: int) -> torch.Tensor:
    """Entropic transport value between weights a [N] and b [M] for the lazy cost C [N, M]: the dual value
    <a, f> + <b, g> at the fixed point of the log-domain Sinkhorn updates
        f_i = -eps log sum_j b_j exp((g_j - C_ij) / eps),   g_j = -eps log sum_i a_i exp((f_i - C_ij) / eps),
    starting from g = 0. The iterations run without gradient; a last f update is differentiable, so the
    gradient with respect to the cost is the transport plan (envelope theorem)."""
    if C.row_bias is not None or C.col_bias is not None or C._meta.apply_exp:
        raise ValueError("sinkhorn_divergence: a cost must be a lazy matrix without biases or exp")
    la, lb = a.log(), b.log()
    K = C * (-1.0 / epsilon)
    g = torch.zeros_like(b)
    with torch.no_grad():
        for _ in range(iters):
            f = -epsilon * K.add_columns(lb + g / epsilon).logsumexp(-1)
            g = -epsilon * K.T.add_columns(la + f / epsilon).logsumexp(-1)
    g = g.detach()
    f = -epsilon * K.add_columns(lb + g / epsilon).logsumexp(-1)
    return (a * f).sum() + (b * g).sum()


def sinkhorn_divergence(C_xy: LazyScores, C_xx: LazyScores, C_yy: LazyScores, a: torch.Tensor, b: torch.Tensor,
                        epsilon: float, iters: int = 100) -> torch.Tensor:
    """Debiased entropic transport: OT_eps(a, b) - OT_eps(a, a) / 2 - OT_eps(b, b) / 2, with C_xy the cost
    between the two point sets and C_xx, C_yy the costs within each. a, b: positive weights that sum to
    one. Each OT_eps is `iters` rounds of two fused log-sum-exp sweeps (rows, then columns through the
    transposed matrix) with the potentials as column biases."""
    return (_entropic_ot(C_xy, a, b, epsilon, iters) - 0.5 * _entropic_ot(C_xx, a, a, epsilon, iters)
            - 0.5 * _entropic_ot(C_yy, b, b, epsilon, iters))
