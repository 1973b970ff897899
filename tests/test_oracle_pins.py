"""Pins for the oracle, checked on the CPU without any GPU code involved.

The oracle is pinned to things other than itself:
  * a hand-derived worked example (tests/golden/tiny_1d_closed_forms.txt);
  * dense fp64 brute force built from torch library primitives (torch.logsumexp, torch.softmax,
    matrix products, a stable sort) and, for gradients, torch.autograd on that dense expression;
  * central finite differences of the oracle's own forward (pins each backward to its forward);
  * closed forms and invariants that the guide "Using Torchpairwise in Models" fixes: rbf(x,x)=1,
    the row-mass column of K @ [V | ones] (Task Map), softmax rows summing to one, logsumexp of a
    constant row with exclude_self, the SVGD direction formula and its n=1 and n=2 special cases
    (Stein Variational Gradient Descent), translation invariance of distance-based scores.
Shapes are asymmetric (N != M, D != C) with random biases and weights so that a dropped term, a
wrong sign or index, or a transposed operand fails at least one test.
"""
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(12345)

# --------------------------------------------------------------------------------------------
# independent dense brute force (torch fp64, CPU)
# --------------------------------------------------------------------------------------------


def dense_scores(X, Y, metric, gamma=1.0, scale=1.0, rb=None, cb=None, rw=None, cw=None,
                 apply_exp=False):
    if metric == "linear":
        base = X @ Y.T
    else:
        d2 = (X[:, None, :] - Y[None, :, :]).pow(2).sum(-1)
        base = torch.exp(-gamma * d2) if metric == "rbf" else d2
    t = scale * base
    if rw is not None:
        t = t * rw[:, None]
    if cw is not None:
        t = t * cw[None, :]
    if rb is not None:
        t = t + rb[:, None]
    if cb is not None:
        t = t + cb[None, :]
    return torch.exp(t) if apply_exp else t


def t64(a, grad=False):
    if a is None:
        return None
    t = torch.tensor(np.asarray(a), dtype=torch.float64)
    return t.requires_grad_(grad)


def make_case(N, M, D, metric, bias=False, weight=False, apply_exp=False, scale=None, gamma=None):
    X = RNG.standard_normal((N, D))
    Y = RNG.standard_normal((M, D))
    kw = dict(metric=metric,
              gamma=gamma if gamma is not None else float(RNG.uniform(0.2, 0.8)),
              scale=scale if scale is not None else float(RNG.uniform(-0.7, 0.7)),
              apply_exp=apply_exp)
    if bias:
        kw["row_bias"] = RNG.standard_normal(N) * 0.3
        kw["col_bias"] = RNG.standard_normal(M) * 0.3
    if weight:
        kw["row_weight"] = RNG.uniform(0.5, 1.5, N)
        kw["col_weight"] = RNG.uniform(0.5, 1.5, M)
    return X, Y, kw


def dense_from(X, Y, kw, grad=False):
    Xt, Yt = t64(X, grad), t64(Y, grad)
    extra = {k: t64(kw.get(k), grad) for k in ("row_bias", "col_bias", "row_weight", "col_weight")}
    S = dense_scores(Xt, Yt, kw["metric"], kw["gamma"], kw["scale"], extra["row_bias"],
                     extra["col_bias"], extra["row_weight"], extra["col_weight"], kw["apply_exp"])
    return S, Xt, Yt, extra


CASES = [
    ("sqeuclidean", False, False, False),
    ("linear", True, False, False),
    ("rbf", True, True, False),
    ("sqeuclidean", True, True, True),
    ("linear", False, True, True),
    ("rbf", False, False, True),
]


def _close(a, b, tol=1e-11):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.abs(b).max()) if b.size else 1.0)
    np.testing.assert_allclose(a, b, rtol=tol, atol=tol * scale)


def _grad_list(kw):
    return [k for k in ("row_bias", "col_bias", "row_weight", "col_weight") if kw.get(k) is not None]


def _check_grads(g, Xt, Yt, extra, kw, tol=1e-10):
    _close(g["dX"], Xt.grad.numpy(), tol)
    _close(g["dY"], Yt.grad.numpy(), tol)
    names = {"row_bias": "d_row_bias", "col_bias": "d_col_bias", "row_weight": "d_row_weight",
             "col_weight": "d_col_weight"}
    for k in _grad_list(kw):
        _close(g[names[k]], extra[k].grad.numpy(), tol)


# --------------------------------------------------------------------------------------------
# hand-derived worked example
# --------------------------------------------------------------------------------------------


def _golden_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "tiny_1d_closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("=", 1)
            case, consumer, row = lhs.split()
            vals = [eval(e, {"__builtins__": {}}, {"log": math.log, "exp": math.exp})
                    for e in rhs.split(";")]
            rows.append((case, consumer, int(row), vals))
    return rows


def test_golden_tiny_1d(oracle):
    X = np.array([[0.0], [1.0]])
    Y = np.array([[0.0], [2.0], [3.0]])
    rows = _golden_rows()
    assert len(rows) >= 16
    for case, consumer, r, vals in rows:
        gamma = 0.5 if case == "rbf" else 1.0
        pb = oracle.Problem(X, Y, metric=case, gamma=gamma)
        if consumer == "logsumexp":
            got = [oracle.logsumexp(pb)[r]]
        elif consumer.startswith("topk"):
            largest = "largest" in consumer
            v, i = oracle.topk(pb, 2, largest=largest)
            got = list(v[r]) if consumer.endswith("values") else list(i[r])
        elif consumer == "softmax_matmul_V123":
            got = [oracle.softmax_matmul(pb, np.array([[1.0], [2.0], [3.0]]))[0][r, 0]]
        elif consumer == "matmul_rowmass":
            V = np.concatenate([RNG.standard_normal((3, 2)), np.ones((3, 1))], 1)
            got = [oracle.matmul(pb, V)[r, -1]]
        elif consumer == "displacement":
            got = [oracle.displacement(pb)[r, 0]]
        else:
            raise AssertionError(consumer)
        _close(got, vals, 1e-13)


def test_golden_shapes_from_the_guide(oracle):
    """Encoded-features page, "Prepare Once, Use Several Consumers": N=3 samples against M=5
    references give a logical [3,5] score; topk(2, largest=False) -> [3,2]; matmul(V [5,4]) -> [3,4].
    """
    X = RNG.standard_normal((3, 16))
    Y = RNG.standard_normal((5, 16))
    pb = oracle.Problem(X, Y, metric="sqeuclidean")
    v, i = oracle.topk(pb, 2)
    assert v.shape == (3, 2) and i.shape == (3, 2)
    assert oracle.matmul(pb, RNG.standard_normal((5, 4))).shape == (3, 4)


# --------------------------------------------------------------------------------------------
# dense brute force: forward
# --------------------------------------------------------------------------------------------


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_scores_match_dense(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(7, 5, 3, metric, bias, weight, apply_exp)
    pb = oracle.Problem(X, Y, **kw)
    S = dense_from(X, Y, kw)[0].numpy()
    got = np.array([[oracle.pair_score(pb, i, j) for j in range(5)] for i in range(7)])
    _close(got, S, 1e-13)


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_matmul_dense(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(9, 6, 4, metric, bias, weight, apply_exp)
    V = RNG.standard_normal((6, 3))
    S = dense_from(X, Y, kw)[0]
    _close(oracle.matmul(oracle.Problem(X, Y, **kw), V), (S @ t64(V)).numpy())


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
@pytest.mark.parametrize("exclude_self", [False, True])
def test_logsumexp_dense(oracle, metric, bias, weight, apply_exp, exclude_self):
    n = 8
    X, Y, kw = make_case(n, n, 3, metric, bias, weight, apply_exp)
    S = dense_from(X, Y, kw)[0]
    if exclude_self:
        S = S.masked_fill(torch.eye(n, dtype=torch.bool), -math.inf)
    _close(oracle.logsumexp(oracle.Problem(X, Y, **kw), exclude_self), torch.logsumexp(S, -1).numpy())


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_softmax_matmul_dense(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(7, 10, 5, metric, bias, weight, apply_exp)
    V = RNG.standard_normal((10, 4))
    S = dense_from(X, Y, kw)[0]
    out, lse = oracle.softmax_matmul(oracle.Problem(X, Y, **kw), V)
    _close(out, (torch.softmax(S, -1) @ t64(V)).numpy())
    _close(lse, torch.logsumexp(S, -1).numpy())


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_displacement_dense(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(6, 9, 3, metric, bias, weight, apply_exp)
    S = dense_from(X, Y, kw)[0]
    want = S @ t64(Y) - S.sum(1, keepdim=True) * t64(X)
    _close(oracle.displacement(oracle.Problem(X, Y, **kw)), want.numpy())


@pytest.mark.parametrize("largest", [False, True])
@pytest.mark.parametrize("metric", ["sqeuclidean", "linear"])
def test_topk_integer_ties_dense(oracle, metric, largest):
    """Integer coordinates: every score is exact in fp64 and ties are frequent; the result must
    equal a stable sort of each row (equal values keep ascending index order)."""
    X = RNG.integers(-2, 3, (11, 3)).astype(np.float64)
    Y = RNG.integers(-2, 3, (40, 3)).astype(np.float64)
    S = dense_scores(t64(X), t64(Y), metric)
    key = -S if largest else S
    order = torch.sort(key, dim=-1, stable=True).indices[:, :7]
    v, i = oracle.topk(oracle.Problem(X, Y, metric=metric), 7, largest=largest)
    np.testing.assert_array_equal(i, order.numpy())
    np.testing.assert_array_equal(v, torch.gather(S, 1, order).numpy())
    # invariants: sorted values, ascending indices within equal values
    d = np.diff(v, axis=1) if not largest else -np.diff(v, axis=1)
    assert (d >= 0).all()
    ties = np.diff(v, axis=1) == 0
    assert (np.diff(i, axis=1)[ties] > 0).all()
    assert ties.any()


def test_topk_full_row(oracle):
    X = RNG.standard_normal((4, 2))
    Y = RNG.standard_normal((6, 2))
    v, i = oracle.topk(oracle.Problem(X, Y, metric="sqeuclidean"), 6)
    for r in range(4):
        assert sorted(i[r].tolist()) == list(range(6))


# --------------------------------------------------------------------------------------------
# dense brute force: gradients via torch.autograd
# --------------------------------------------------------------------------------------------


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_matmul_backward_autograd(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(7, 5, 3, metric, bias, weight, apply_exp)
    V = RNG.standard_normal((5, 4))
    G = RNG.standard_normal((7, 4))
    S, Xt, Yt, extra = dense_from(X, Y, kw, grad=True)
    Vt = t64(V, True)
    (S @ Vt).backward(t64(G))
    g = oracle.matmul_backward(oracle.Problem(X, Y, **kw), V, G)
    _check_grads(g, Xt, Yt, extra, kw)
    _close(g["dV"], Vt.grad.numpy())


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
@pytest.mark.parametrize("exclude_self", [False, True])
def test_logsumexp_backward_autograd(oracle, metric, bias, weight, apply_exp, exclude_self):
    n = 7
    X, Y, kw = make_case(n, n, 3, metric, bias, weight, apply_exp)
    gl = RNG.standard_normal(n)
    S, Xt, Yt, extra = dense_from(X, Y, kw, grad=True)
    if exclude_self:
        S = S.masked_fill(torch.eye(n, dtype=torch.bool), -math.inf)
    lse = torch.logsumexp(S, -1)
    lse.backward(t64(gl))
    pb = oracle.Problem(X, Y, **kw)
    g = oracle.logsumexp_backward(pb, lse.detach().numpy(), gl, exclude_self)
    _check_grads(g, Xt, Yt, extra, kw)


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_softmax_matmul_backward_autograd(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(6, 8, 3, metric, bias, weight, apply_exp)
    V = RNG.standard_normal((8, 5))
    G = RNG.standard_normal((6, 5))
    S, Xt, Yt, extra = dense_from(X, Y, kw, grad=True)
    Vt = t64(V, True)
    out = torch.softmax(S, -1) @ Vt
    out.backward(t64(G))
    pb = oracle.Problem(X, Y, **kw)
    o, lse = oracle.softmax_matmul(pb, V)
    g = oracle.softmax_matmul_backward(pb, V, o, lse, G)
    _check_grads(g, Xt, Yt, extra, kw)
    _close(g["dV"], Vt.grad.numpy())


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_displacement_backward_autograd(oracle, metric, bias, weight, apply_exp):
    X, Y, kw = make_case(5, 7, 4, metric, bias, weight, apply_exp)
    G = RNG.standard_normal((5, 4))
    S, Xt, Yt, extra = dense_from(X, Y, kw, grad=True)
    out = S @ Yt - S.sum(1, keepdim=True) * Xt
    out.backward(t64(G))
    g = oracle.displacement_backward(oracle.Problem(X, Y, **kw), G)
    _check_grads(g, Xt, Yt, extra, kw)


@pytest.mark.parametrize("metric,bias,weight,apply_exp", CASES)
def test_topk_backward_autograd(oracle, metric, bias, weight, apply_exp):
    """Gradients flow through the selected pairs only ("What to Check", selections)."""
    X, Y, kw = make_case(6, 9, 3, metric, bias, weight, apply_exp)
    k = 4
    pb = oracle.Problem(X, Y, **kw)
    v, idx = oracle.topk(pb, k)
    gv = RNG.standard_normal((6, k))
    S, Xt, Yt, extra = dense_from(X, Y, kw, grad=True)
    sel = torch.gather(S, 1, torch.tensor(idx))
    _close(sel.detach().numpy(), v)
    sel.backward(t64(gv))
    g = oracle.topk_backward(pb, k, idx, gv)
    _check_grads(g, Xt, Yt, extra, kw)


# --------------------------------------------------------------------------------------------
# finite differences (backward against the oracle's own forward)
# --------------------------------------------------------------------------------------------


def _fd(f, A, h=1e-6):
    g = np.zeros_like(A)
    for idx in np.ndindex(A.shape):
        Ap = A.copy(); Ap[idx] += h
        Am = A.copy(); Am[idx] -= h
        g[idx] = (f(Ap) - f(Am)) / (2 * h)
    return g


@pytest.mark.parametrize("metric", ["sqeuclidean", "linear", "rbf"])
def test_finite_differences_all_consumers(oracle, metric):
    N, M, D, C = 4, 5, 2, 3
    X, Y, kw = make_case(N, M, D, metric, bias=True, weight=True)
    V = RNG.standard_normal((M, C))
    GO = RNG.standard_normal((N, C))
    GD = RNG.standard_normal((N, D))

    def loss_mm(Xa, Ya, Va=V):
        return float((oracle.matmul(oracle.Problem(Xa, Ya, **kw), Va) * GO).sum())

    def loss_sm(Xa, Ya, Va=V):
        return float((oracle.softmax_matmul(oracle.Problem(Xa, Ya, **kw), Va)[0] * GO).sum())

    def loss_disp(Xa, Ya):
        return float((oracle.displacement(oracle.Problem(Xa, Ya, **kw)) * GD).sum())

    pb = oracle.Problem(X, Y, **kw)
    g = oracle.matmul_backward(pb, V, GO)
    _close(g["dX"], _fd(lambda A: loss_mm(A, Y), X), 1e-6)
    _close(g["dY"], _fd(lambda A: loss_mm(X, A), Y), 1e-6)
    _close(g["dV"], _fd(lambda A: loss_mm(X, Y, A), V), 1e-6)

    o, lse = oracle.softmax_matmul(pb, V)
    g = oracle.softmax_matmul_backward(pb, V, o, lse, GO)
    _close(g["dX"], _fd(lambda A: loss_sm(A, Y), X), 1e-6)
    _close(g["dY"], _fd(lambda A: loss_sm(X, A), Y), 1e-6)
    _close(g["dV"], _fd(lambda A: loss_sm(X, Y, A), V), 1e-6)

    g = oracle.displacement_backward(pb, GD)
    _close(g["dX"], _fd(lambda A: loss_disp(A, Y), X), 1e-6)
    _close(g["dY"], _fd(lambda A: loss_disp(X, A), Y), 1e-6)

    # row/column bias and weight gradients of logsumexp
    Xs, _, kws = make_case(5, 5, 2, metric, bias=True, weight=True)
    gl = RNG.standard_normal(5)

    def loss_lse(**over):
        k2 = dict(kws); k2.update(over)
        return float((oracle.logsumexp(oracle.Problem(Xs, Xs, **k2), True) * gl).sum())

    pbs = oracle.Problem(Xs, Xs, **kws)
    g = oracle.logsumexp_backward(pbs, oracle.logsumexp(pbs, True), gl, True)
    for name, key in (("row_bias", "d_row_bias"), ("col_bias", "d_col_bias"),
                      ("row_weight", "d_row_weight"), ("col_weight", "d_col_weight")):
        base = kws[name]
        _close(g[key], _fd(lambda A: loss_lse(**{name: A}), base), 1e-6)
    # X and Y are the same points here: their gradients add up to the gradient in the points
    tot = g["dX"] + g["dY"]

    def loss_same(A):
        return float((oracle.logsumexp(oracle.Problem(A, A, **kws), True) * gl).sum())

    _close(tot, _fd(loss_same, Xs), 1e-6)


# --------------------------------------------------------------------------------------------
# closed forms and invariants
# --------------------------------------------------------------------------------------------


def test_rbf_self_is_one_and_sqeuclidean_self_is_zero(oracle):
    X = RNG.standard_normal((6, 5))
    pr = oracle.Problem(X, X, metric="rbf", gamma=0.37)
    ps = oracle.Problem(X, X, metric="sqeuclidean")
    for i in range(6):
        assert oracle.pair_score(pr, i, i) == 1.0
        assert oracle.pair_score(ps, i, i) == 0.0


def test_rbf_gamma_zero_gives_column_sums(oracle):
    X = RNG.standard_normal((5, 3))
    Y = RNG.standard_normal((8, 3))
    V = RNG.standard_normal((8, 4))
    out = oracle.matmul(oracle.Problem(X, Y, metric="rbf", gamma=0.0), V)
    _close(out, np.broadcast_to(V.sum(0), (5, 4)), 1e-13)


def test_row_mass_column(oracle):
    """Task Map, kernel attention: the last column of K @ [V | ones] is the row mass."""
    X = RNG.standard_normal((7, 3))
    Y = RNG.standard_normal((9, 3))
    V = np.concatenate([RNG.standard_normal((9, 3)), np.ones((9, 1))], 1)
    out = oracle.matmul(oracle.Problem(X, Y, metric="rbf", gamma=0.5), V)
    mass = np.exp(-0.5 * ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)).sum(1)
    _close(out[:, -1], mass, 1e-13)


def test_lse_constant_row_exclude_self(oracle):
    """All rows equal and unit norm: S = 1/0.07 everywhere, so lse = 1/0.07 + log(M-1)."""
    n = 33
    z = np.tile(RNG.standard_normal(16), (n, 1))
    z /= np.linalg.norm(z, axis=1, keepdims=True)
    lse = oracle.logsumexp(oracle.Problem(z, z, metric="linear", scale=1 / 0.07), True)
    _close(lse, np.full(n, 1 / 0.07 + math.log(n - 1)), 1e-12)


def test_lse_orthonormal_and_bias_shift(oracle):
    n = 12
    z = np.eye(n)
    lse = oracle.logsumexp(oracle.Problem(z, z, metric="linear"), True)
    _close(lse, np.full(n, math.log(n - 1)), 1e-13)
    b = RNG.standard_normal(n)
    lse_b = oracle.logsumexp(oracle.Problem(z, z, metric="linear", row_bias=b), True)
    _close(lse_b, lse + b, 1e-13)
    # empty rows: N = M = 1 with exclude_self -> -inf and zero gradient
    one = np.ones((1, 2))
    pb = oracle.Problem(one, one, metric="linear")
    l1 = oracle.logsumexp(pb, True)
    assert l1[0] == -math.inf
    g = oracle.logsumexp_backward(pb, l1, np.ones(1), True)
    assert (g["dX"] == 0).all() and (g["dY"] == 0).all()


def test_lse_row_bias_gradient_is_upstream(oracle):
    """d lse_i / d br_i = sum_j P_ij = 1, so the row-bias gradient equals the upstream gradient."""
    X, _, kw = make_case(9, 9, 3, "linear", bias=True)
    gl = RNG.standard_normal(9)
    pb = oracle.Problem(X, X, **kw)
    g = oracle.logsumexp_backward(pb, oracle.logsumexp(pb, True), gl, True)
    _close(g["d_row_bias"], gl, 1e-12)


def test_softmax_rows_sum_to_one(oracle):
    X, Y, kw = make_case(8, 11, 3, "sqeuclidean", bias=True, weight=True)
    pb = oracle.Problem(X, Y, **kw)
    out, _ = oracle.softmax_matmul(pb, np.ones((11, 1)))
    _close(out, np.ones((8, 1)), 1e-13)
    # a row bias shifts every score of a row equally: the output and d(row bias) do not move
    kw2 = dict(kw); kw2["row_bias"] = kw["row_bias"] + 3.0
    V = RNG.standard_normal((11, 2))
    _close(oracle.softmax_matmul(oracle.Problem(X, Y, **kw2), V)[0],
           oracle.softmax_matmul(pb, V)[0], 1e-12)
    o, lse = oracle.softmax_matmul(pb, V)
    g = oracle.softmax_matmul_backward(pb, V, o, lse, RNG.standard_normal((8, 2)))
    _close(g["d_row_bias"], np.zeros(8), 1e-12)


@pytest.mark.parametrize("metric", ["sqeuclidean", "rbf"])
def test_translation_invariance_of_gradients(oracle, metric):
    """Scores that depend on x - y only: sum_i dX_i + sum_j dY_j = 0 for every consumer."""
    X, Y, kw = make_case(6, 7, 3, metric, bias=True, weight=True)
    pb = oracle.Problem(X, Y, **kw)
    V = RNG.standard_normal((7, 2))
    G = RNG.standard_normal((6, 2))
    for g in (oracle.matmul_backward(pb, V, G),
              oracle.displacement_backward(pb, RNG.standard_normal((6, 3))),
              oracle.softmax_matmul_backward(pb, V, *oracle.softmax_matmul(pb, V), G)):
        _close(g["dX"].sum(0) + g["dY"].sum(0), np.zeros(3), 1e-11)


def test_svgd_matches_guide_formula_and_autograd(oracle):
    """Stein Variational Gradient Descent: phi = (K @ score - 2 gamma K.displacement()) / n, and
    phi_i = (1/n) sum_j [k(x_j,x_i) score_j + grad_{x_j} k(x_j,x_i)] with the gradient by autograd."""
    n, D, gamma = 9, 3, 0.3
    x = RNG.standard_normal((n, D))
    score = -x
    phi = oracle.svgd_direction(x, score, gamma)
    pb = oracle.Problem(x, x, metric="rbf", gamma=gamma)
    _close(phi, (oracle.matmul(pb, score) - 2 * gamma * oracle.displacement(pb)) / n, 1e-12)
    xt = t64(x)
    want = torch.zeros(n, D, dtype=torch.float64)
    for i in range(n):
        xj = xt.clone().requires_grad_(True)
        k = torch.exp(-gamma * (xj - xt[i]).pow(2).sum(-1))  # k(x_j, x_i) for all j
        (gk,) = torch.autograd.grad(k.sum(), xj)  # row j holds grad_{x_j} k(x_j, x_i)
        want[i] = ((k.detach()[:, None] * t64(score)) + gk).sum(0) / n
    _close(phi, want.numpy(), 1e-12)


def test_svgd_special_cases(oracle):
    gamma = 0.7
    # n = 1: the kernel is 1 and its gradient vanishes, so phi = score
    x = RNG.standard_normal((1, 4))
    s = RNG.standard_normal((1, 4))
    _close(oracle.svgd_direction(x, s, gamma), s, 1e-14)
    # n = 2: phi_1 = (score_1 + k score_2 - 2 gamma k (x_2 - x_1)) / 2, k = exp(-gamma |x_1-x_2|^2)
    x = RNG.standard_normal((2, 3))
    s = RNG.standard_normal((2, 3))
    k = math.exp(-gamma * ((x[0] - x[1]) ** 2).sum())
    want0 = (s[0] + k * s[1] - 2 * gamma * k * (x[1] - x[0])) / 2
    want1 = (s[1] + k * s[0] - 2 * gamma * k * (x[0] - x[1])) / 2
    _close(oracle.svgd_direction(x, s, gamma), np.stack([want0, want1]), 1e-14)


def test_thread_count_does_not_change_results(oracle):
    X, Y, kw = make_case(50, 40, 3, "rbf", bias=True)
    V = RNG.standard_normal((40, 2))
    pb = oracle.Problem(X, Y, **kw)
    oracle.set_threads(1)
    a = oracle.matmul(pb, V)
    oracle.set_threads(5)
    b = oracle.matmul(pb, V)
    oracle.set_threads(0)
    np.testing.assert_array_equal(a, b)
