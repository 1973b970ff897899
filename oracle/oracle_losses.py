"""Oracle for the losses built on the consumers: TEST INFRASTRUCTURE ONLY.

Plain fp64 numpy from the definitions, dense and slow (test sizes only). Only ``tests/`` may import
this module; the product package never imports it.

Passages (torchpairwise guide "Using Torchpairwise in Models", Task Map): "Chamfer-style losses:
D.min(-1) and D.min(-2) on D = lazy(X, Y, "sqeuclidean"), min returns values and indices";
"MMD loss, two-sample test: mmd_statistics(X[None], Y[None], kernel="rbf", gamma=g), unbiased by
default" (X[None]: one point cloud per batch entry); "Optimal transport loss:
sinkhorn_divergence(C_xy, C_xx, C_yy, a, b, epsilon=e), any lazy cost".
"""
from __future__ import annotations

import numpy as np


def sqdist(X, Y):
    """|x_i - y_j|^2 by the direct difference, fp64 [N, M]."""
    X = np.asarray(X, np.float64)
    Y = np.asarray(Y, np.float64)
    out = np.empty((X.shape[0], Y.shape[0]))
    for i in range(X.shape[0]):
        d = Y - X[i]
        out[i] = (d * d).sum(1)
    return out


def kernel_matrix(X, Y, kernel, gamma):
    if kernel == "rbf":
        return np.exp(-gamma * sqdist(X, Y))
    if kernel == "linear":
        return np.asarray(X, np.float64) @ np.asarray(Y, np.float64).T
    raise ValueError(kernel)


def column_min(X, Y):
    """Chamfer's D.min(-2) on D = sqeuclidean: per column j, the smallest D_ij and the smallest i
    attaining it."""
    D = sqdist(X, Y)
    idx = np.argmin(D, axis=0)  # first occurrence: the lowest row index among equal values
    return D[idx, np.arange(D.shape[1])], idx


def mmd(X, Y, kernel="rbf", gamma=1.0, unbiased=True):
    """Squared MMD per batch entry, X [B, m, D], Y [B, n, D]. Unbiased: U-statistic (the pairs i = i'
    left out of the within-cloud means); biased: V-statistic."""
    out = []
    for b in range(X.shape[0]):
        kxx = kernel_matrix(X[b], X[b], kernel, gamma)
        kyy = kernel_matrix(Y[b], Y[b], kernel, gamma)
        kxy = kernel_matrix(X[b], Y[b], kernel, gamma)
        m, n = kxx.shape[0], kyy.shape[0]
        if unbiased:
            v = ((kxx.sum() - np.trace(kxx)) / (m * (m - 1)) + (kyy.sum() - np.trace(kyy)) / (n * (n - 1))
                 - 2.0 * kxy.sum() / (m * n))
        else:
            v = kxx.sum() / (m * m) + kyy.sum() / (n * n) - 2.0 * kxy.sum() / (m * n)
        out.append(v)
    return np.array(out)


def _lse_rows(A):
    """log sum_j exp(A_ij) per row, two passes (max, then sum)."""
    m = A.max(1, keepdims=True)
    return m[:, 0] + np.log(np.exp(A - m).sum(1))


def entropic_ot(C, a, b, eps, iters):
    """Dual value <a, f> + <b, g> after `iters` rounds of the log-domain Sinkhorn updates
    f_i = -eps log sum_j b_j exp((g_j - C_ij)/eps), g_j = -eps log sum_i a_i exp((f_i - C_ij)/eps), g = 0
    at the start, and one more f update (the value the library returns)."""
    C = np.asarray(C, np.float64)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    g = np.zeros(C.shape[1])
    for _ in range(iters):
        f = -eps * _lse_rows(np.log(b)[None, :] + (g[None, :] - C) / eps)
        g = -eps * _lse_rows(np.log(a)[None, :] + (f[None, :] - C.T) / eps)
    f = -eps * _lse_rows(np.log(b)[None, :] + (g[None, :] - C) / eps)
    return float(a @ f + b @ g), f, g


def sinkhorn_divergence(Cxy, Cxx, Cyy, a, b, eps, iters):
    """OT_eps(a, b) - OT_eps(a, a) / 2 - OT_eps(b, b) / 2."""
    return (entropic_ot(Cxy, a, b, eps, iters)[0] - 0.5 * entropic_ot(Cxx, a, a, eps, iters)[0]
            - 0.5 * entropic_ot(Cyy, b, b, eps, iters)[0])
