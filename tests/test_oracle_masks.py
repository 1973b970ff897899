"""Pins of the oracle's pair masks (CPU only) against dense fp64 torch: the masked pairs leave every
consumer, forward and backward (torchpairwise guide "Using Torchpairwise in Models", Score Expressions
and Task Map: tp.masks causal, band, same_group)."""
import numpy as np
import pytest
import torch

from oracle import oracle

N, M, D, C = 23, 31, 5, 3


def _data(seed):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(N, D, generator=g, dtype=torch.float64)
    Y = torch.randn(M, D, generator=g, dtype=torch.float64)
    V = torch.randn(M, C, generator=g, dtype=torch.float64)
    rg = torch.randint(0, 4, (N,), generator=g, dtype=torch.int32)
    cg = torch.randint(0, 4, (M,), generator=g, dtype=torch.int32)
    rg[0] = 7  # a row whose group no column has: every pair masked
    return X, Y, V, rg, cg


def _keep(kind, rg, cg, band=3):
    i = torch.arange(N)[:, None]
    j = torch.arange(M)[None, :]
    if kind == "causal":
        return j <= i
    if kind == "band":
        return (i - j).abs() <= band
    return rg[:, None] == cg[None, :]


MASKS = ["causal", "band", "same_group"]


def _problem(X, Y, kind, rg, cg, **kw):
    return oracle.Problem(X, Y, pair_mask=kind, band=3, row_group=rg.numpy(), col_group=cg.numpy(), **kw)


def _dense(X, Y, scale):
    return scale * (X @ Y.T)


@pytest.mark.parametrize("kind", MASKS)
def test_masked_matmul_and_displacement_are_dense_masked_sums(kind):
    X, Y, V, rg, cg = _data(1)
    keep = _keep(kind, rg, cg)
    pb = _problem(X, Y, kind, rg, cg, metric="rbf", gamma=0.3)
    K = torch.exp(-0.3 * torch.cdist(X, Y) ** 2) * keep
    assert np.allclose(oracle.matmul(pb, V), (K @ V).numpy(), rtol=1e-12, atol=1e-13)
    disp = K @ Y - K.sum(1, keepdim=True) * X
    assert np.allclose(oracle.displacement(pb), disp.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind", MASKS)
def test_masked_lse_and_softmax_are_dense_masked(kind):
    X, Y, V, rg, cg = _data(2)
    keep = _keep(kind, rg, cg)
    pb = _problem(X, Y, kind, rg, cg, scale=0.7)
    S = _dense(X, Y, 0.7).masked_fill(~keep, float("-inf"))
    ref = torch.logsumexp(S, 1)
    got = oracle.logsumexp(pb)
    assert np.array_equal(np.isfinite(got), torch.isfinite(ref).numpy())
    fin = torch.isfinite(ref).numpy()
    assert np.allclose(got[fin], ref.numpy()[fin], rtol=1e-13, atol=1e-13)
    out, lse = oracle.softmax_matmul(pb, V)
    P = torch.softmax(S, 1).nan_to_num(0.0)  # an empty row returns 0
    assert np.allclose(out, (P @ V).numpy(), rtol=1e-12, atol=1e-13)
    if kind == "same_group":
        assert not fin[0] and np.all(out[0] == 0)  # row 0 has no kept pair


@pytest.mark.parametrize("kind", MASKS)
def test_masked_topk_pads_rows_with_fewer_kept_pairs(kind):
    X, Y, _, rg, cg = _data(3)
    X, Y = torch.round(3 * X), torch.round(3 * Y)  # integer distances: ties
    keep = _keep(kind, rg, cg)
    pb = _problem(X, Y, kind, rg, cg, metric="sqeuclidean")
    k = 6
    vals, idx = oracle.topk(pb, k, largest=False)
    Dm = (torch.cdist(X, Y) ** 2).round()  # exact: integer inputs
    for i in range(N):
        js = [j for j in range(M) if keep[i, j]]
        order = sorted(js, key=lambda j: (Dm[i, j].item(), j))[:k]
        assert list(idx[i, :len(order)]) == order
        assert np.allclose(vals[i, :len(order)], Dm[i, order].numpy())
        assert np.all(idx[i, len(order):] == -1) and np.all(np.isinf(vals[i, len(order):]))


@pytest.mark.parametrize("kind", MASKS)
def test_masked_backward_matches_dense_autograd(kind):
    X0, Y0, V, rg, cg = _data(4)
    keep = _keep(kind, rg, cg)
    rows = keep.any(1)  # rows with a kept pair (the others carry no gradient)
    X, Y, Vg = X0.clone().requires_grad_(), Y0.clone().requires_grad_(), V.clone().requires_grad_()
    S = _dense(X, Y, 0.5).masked_fill(~keep, float("-inf"))
    G = torch.randn(N, C, generator=torch.Generator().manual_seed(5), dtype=torch.float64)
    gl = torch.randn(N, generator=torch.Generator().manual_seed(6), dtype=torch.float64)
    out = torch.softmax(S[rows], 1) @ Vg
    (out * G[rows]).sum().backward()
    pb = _problem(X0, Y0, kind, rg, cg, scale=0.5)
    o, l = oracle.softmax_matmul(pb, V)
    g = oracle.softmax_matmul_backward(pb, V, o, l, G.numpy())
    for got, want in ((g["dX"], X.grad), (g["dY"], Y.grad), (g["dV"], Vg.grad)):
        assert np.allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)
    X.grad = Y.grad = None
    S = _dense(X, Y, 0.5).masked_fill(~keep, float("-inf"))
    (torch.logsumexp(S[rows], 1) * gl[rows]).sum().backward()
    lse = oracle.logsumexp(pb)
    g2 = oracle.logsumexp_backward(pb, lse, gl.numpy())
    assert np.allclose(g2["dX"], X.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(g2["dY"], Y.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_masks_that_keep_one_pair_per_row_are_closed_forms():
    # band width 0 on N = M, and a same-group mask whose groups pair each row with one column: the
    # softmax of a row over a single kept pair is 1, so lse_i = S_i,pi(i), out_i = V_pi(i), dS = 0 (no score
    # gradient) and dV_pi(i) = dO_i; with causal, row 0 keeps column 0 alone
    g = torch.Generator().manual_seed(5)
    n = 17
    X = torch.randn(n, D, generator=g, dtype=torch.float64)
    Y = torch.randn(n, D, generator=g, dtype=torch.float64)
    V = torch.randn(n, C, generator=g, dtype=torch.float64)
    G = torch.randn(n, C, generator=g, dtype=torch.float64)
    perm = torch.randperm(n, generator=g)
    S = 0.3 * (X @ Y.T)
    cases = [("band", dict(band=0), torch.arange(n)),
             ("same_group", dict(row_group=torch.arange(n, dtype=torch.int32).numpy(),
                                 col_group=torch.argsort(perm).to(torch.int32).numpy()), perm)]
    for kind, kw, pick in cases:
        pb = oracle.Problem(X, Y, metric="linear", scale=0.3, pair_mask=kind, **kw)
        out, lse = oracle.softmax_matmul(pb, V)
        np.testing.assert_allclose(lse, S[torch.arange(n), pick].numpy(), rtol=0, atol=1e-14)
        np.testing.assert_allclose(out, V[pick].numpy(), rtol=0, atol=1e-14)
        gr = oracle.softmax_matmul_backward(pb, V, out, lse, G)
        assert np.abs(gr["dX"]).max() < 1e-13 and np.abs(gr["dY"]).max() < 1e-13
        dV = np.zeros((n, C))
        dV[pick.numpy()] = G.numpy()
        np.testing.assert_allclose(gr["dV"], dV, rtol=0, atol=1e-14)
    pb = oracle.Problem(X, Y, metric="linear", scale=0.3, pair_mask="causal")
    out, lse = oracle.softmax_matmul(pb, V)
    assert abs(lse[0] - float(S[0, 0])) < 1e-14 and np.abs(out[0] - V[0].numpy()).max() < 1e-14
    # row 1 keeps columns 0 and 1: a two-term log-sum-exp
    assert abs(lse[1] - float(torch.logsumexp(S[1, :2], 0))) < 1e-13
