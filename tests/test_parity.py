"""GPU parity: every libtp entry point against the oracle, element by element, on seeded inputs.

Shapes span several 128-point CTAs and 32-point tiles with ragged tails, with the split (workspace +
merge) path and the single-split path both exercised, every metric, fp32 and fp64, with and without
row/column biases and weights and the exp node. Tolerances: max relative error (tests/_util.rel_err,
floor 1e-3 of the largest magnitude) 1e-4 for fp32 forward, 5e-4 for fp32 gradients, 1e-10 for fp64,
or twice what a plain dense evaluation in the same precision reaches on the same inputs where that is
larger (tests/_plain.py: random biases, weights and exp build outputs that cancel far below their
terms, where fp32 itself misses 1e-4 by up to ~3x). Top-k on integer-valued inputs is bit-exact in
values and indices.
"""
import ctypes
import numpy as np
import pytest
import torch

from lazy_score_matrix_gb300 import _lib, ops
from lazy_score_matrix_gb300.ops import Score
from tests._plain import Plain, achievable, svgd_direction as plain_svgd
from tests._util import TOL_F32_FWD, TOL_F32_GRAD, TOL_F64, assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

SHAPES = {  # N, M, D, C
    "ragged_split": (300, 517, 3, 4),
    "one_split": (130, 40, 16, 5),
    "wide": (257, 300, 64, 64),
    "padded": (200, 333, 33, 17),
}


def gen(seed, shape, dtype, kind="normal"):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(*shape, generator=g, dtype=dtype)
    if kind == "weight":
        return 0.5 + torch.rand(*shape, generator=g, dtype=dtype)
    raise ValueError(kind)


def problem(shape, dtype, metric, affine, apply_exp, seed=0):
    N, M, D, C = SHAPES[shape]
    X = gen(seed + 1, (N, D), dtype)
    Y = gen(seed + 2, (M, D), dtype)
    V = gen(seed + 3, (M, C), dtype)
    scale = (-0.5 if metric == "sqeuclidean" else 0.5) / D ** 0.5
    if apply_exp:  # keep exp(t) moderate: exp of a large exp is not evaluable to 1e-4 in fp32 at all
        scale *= 0.5
    sc = dict(metric=metric, gamma=0.5 / D, scale=scale if metric != "rbf" else 0.8, apply_exp=apply_exp)
    if affine:
        sc.update(row_bias=0.3 * gen(seed + 4, (N,), dtype), col_bias=0.3 * gen(seed + 5, (M,), dtype),
                  row_weight=gen(seed + 6, (N,), dtype, "weight"), col_weight=gen(seed + 7, (M,), dtype, "weight"))
    return X, Y, V, sc


def gpu_score(sc):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in sc.items()}
    return Score(**d)


def oracle_problem(oracle, X, Y, sc):
    return oracle.Problem(X, Y, **sc)


def tols(dtype):
    return (TOL_F64, TOL_F64) if dtype == torch.float64 else (TOL_F32_FWD, TOL_F32_GRAD)


GRAD_KEYS = ["dX", "dY", "dV", "d_row_bias", "d_col_bias", "d_row_weight", "d_col_weight"]


def check(got, want, plain, tol, what, abs_floor=0.0):
    """got against the oracle's want, held to achievable(): the tolerance or twice the plain evaluation's
    error in the working precision (plain: its result on the same inputs, or None)."""
    bound = tol if plain is None else achievable(plain, want, tol, abs_floor=abs_floor)
    return assert_close(got, want, bound, what, abs_floor=abs_floor)


def compare_grads(got, want, tol, what, plain=None, zero_scale=None):
    """plain: gradients of the plain evaluation (Plain.grads). zero_scale: {key: magnitude} for outputs
    that are zero by the mathematics (their floor is that magnitude instead of a fraction of the,
    rounding-level, expected values)."""
    zero_scale = zero_scale or {}
    plain = plain or {}
    for k in GRAD_KEYS:
        if want.get(k) is None or got.get(k) is None:
            assert (want.get(k) is None) == (got.get(k) is None) or k == "dV", (what, k)
            continue
        check(got[k], want[k], plain.get(k), tol, f"{what} {k}", zero_scale.get(k, 0.0))


CASES = [(shape, dt, metric, affine, ex)
         for shape in SHAPES
         for dt in (torch.float32, torch.float64)
         for metric in ("sqeuclidean", "linear", "rbf")
         for affine, ex in ((False, False), (True, False), (True, True))
         if not (dt == torch.float64 and shape == "wide" and affine)]


def _id(c):
    return f"{c[0]}-{str(c[1])[6:]}-{c[2]}-{'aff' if c[3] else 'plain'}{'-exp' if c[4] else ''}"


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_matmul(oracle, case):
    shape, dt, metric, affine, ex = case
    X, Y, V, sc = problem(shape, dt, metric, affine, ex)
    G = gen(11, (X.shape[0], V.shape[1]), dt)
    ftol, gtol = tols(dt)
    out = ops.pairwise_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))
    pb = oracle_problem(oracle, X, Y, sc)
    pl = Plain(X, Y, dtype=dt, V=V, **sc)
    p_out = pl.matmul()
    check(out, oracle.matmul(pb, V), p_out.detach(), ftol, "matmul out")
    g = ops.pairwise_matmul_backward(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc), G.to(DEV))
    compare_grads(g, oracle.matmul_backward(pb, V, G), gtol, "matmul", pl.grads(p_out, G))


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_softmax_matmul(oracle, case):
    shape, dt, metric, affine, ex = case
    X, Y, V, sc = problem(shape, dt, metric, affine, ex)
    G = gen(12, (X.shape[0], V.shape[1]), dt)
    ftol, gtol = tols(dt)
    out, lse = ops.pairwise_softmax_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))
    pb = oracle_problem(oracle, X, Y, sc)
    o_out, o_lse = oracle.softmax_matmul(pb, V)
    pl = Plain(X, Y, dtype=dt, V=V, **sc)
    p_out, p_lse = pl.softmax_matmul()
    check(out, o_out, p_out.detach(), ftol, "softmax out")
    check(lse, o_lse, p_lse.detach(), ftol, "softmax lse")
    g = ops.pairwise_softmax_matmul_backward(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc), out, lse, G.to(DEV))
    # a row bias shifts a whole row of scores: its softmax gradient is zero; measure it against the
    # size of the terms that cancel (|dO| |V|)
    zs = {"d_row_bias": float(G.abs().max() * V.abs().max())}
    compare_grads(g, oracle.softmax_matmul_backward(pb, V, o_out, o_lse, G), gtol, "softmax", pl.grads(p_out, G),
                  zero_scale=zs)


@pytest.mark.parametrize("exclude_self", [False, True])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_logsumexp(oracle, case, exclude_self):
    shape, dt, metric, affine, ex = case
    X, Y, _, sc = problem(shape, dt, metric, affine, ex)
    if exclude_self:  # needs N == M: use Y's rows for both sides
        X = Y.clone()
        if affine:
            sc["row_bias"] = 0.3 * gen(21, (X.shape[0],), dt)
            sc["row_weight"] = gen(22, (X.shape[0],), dt, "weight")
    gl = gen(13, (X.shape[0],), dt)
    ftol, gtol = tols(dt)
    lse = ops.pairwise_logsumexp(X.to(DEV), Y.to(DEV), gpu_score(sc), exclude_self)
    pb = oracle_problem(oracle, X, Y, sc)
    o_lse = oracle.logsumexp(pb, exclude_self)
    pl = Plain(X, Y, dtype=dt, **sc)
    p_lse = pl.logsumexp(exclude_self)
    check(lse, o_lse, p_lse.detach(), ftol, "lse")
    g = ops.pairwise_logsumexp_backward(X.to(DEV), Y.to(DEV), gpu_score(sc), lse, gl.to(DEV), exclude_self)
    compare_grads(g, oracle.logsumexp_backward(pb, o_lse, gl, exclude_self), gtol, "lse", pl.grads(p_lse, gl))


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_displacement(oracle, case):
    shape, dt, metric, affine, ex = case
    X, Y, _, sc = problem(shape, dt, metric, affine, ex)
    G = gen(14, X.shape, dt)
    ftol, gtol = tols(dt)
    out = ops.pairwise_displacement(X.to(DEV), Y.to(DEV), gpu_score(sc))
    pb = oracle_problem(oracle, X, Y, sc)
    pl = Plain(X, Y, dtype=dt, **sc)
    p_out = pl.displacement()
    check(out, oracle.displacement(pb), p_out.detach(), ftol, "displacement")
    g = ops.pairwise_displacement_backward(X.to(DEV), Y.to(DEV), gpu_score(sc), G.to(DEV))
    compare_grads(g, oracle.displacement_backward(pb, G), gtol, "displacement", pl.grads(p_out, G))


@pytest.mark.parametrize("dt", [torch.float32, torch.float64])
@pytest.mark.parametrize("shape", ["ragged_split", "one_split", "padded"])
def test_svgd_direction(oracle, shape, dt):
    N, _, D, _ = SHAPES[shape]
    x = gen(31, (N, D), dt)
    s = -x + 0.1 * gen(32, (N, D), dt)
    gamma = 0.5 / D
    phi = ops.svgd_direction(x.to(DEV), s.to(DEV), gamma)
    check(phi, oracle.svgd_direction(x, s, gamma), plain_svgd(x, s, gamma, dt), tols(dt)[0], "svgd")


# ------------------------------------------------------------------------------------------------
# top-k
# ------------------------------------------------------------------------------------------------


def int_points(seed, shape, lo=-3, hi=3, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(dtype)


@pytest.mark.parametrize("dt", [torch.float32, torch.float64])
@pytest.mark.parametrize("metric", ["sqeuclidean", "linear"])
@pytest.mark.parametrize("largest", [False, True])
@pytest.mark.parametrize("k", [1, 3, 16, 32])
@pytest.mark.parametrize("NMD", [(300, 700, 5), (129, 33, 16), (64, 2000, 3)])
def test_topk_integer_exact(oracle, NMD, k, largest, metric, dt):
    """Integer-valued points: every score is exact, ties are frequent; values and indices must be
    identical to the oracle's (value, index)-ordered selection."""
    N, M, D = NMD
    X = int_points(41 + D, (N, D), dtype=dt)
    Y = int_points(42 + D, (M, D), dtype=dt)
    v, i = ops.pairwise_topk(X.to(DEV), Y.to(DEV), Score(metric), k, largest)
    ov, oi = oracle.topk(oracle.Problem(X, Y, metric=metric), k, largest)
    np.testing.assert_array_equal(i.cpu().numpy(), oi)
    np.testing.assert_array_equal(v.cpu().double().numpy(), ov)


@pytest.mark.parametrize("metric", ["sqeuclidean", "rbf", "linear"])
@pytest.mark.parametrize("D", [2, 30, 31, 32, 33, 62, 63, 64])
def test_topk_tc_feature_widths_exact(oracle, D, metric):
    """The tensor-core top-k at every feature-width boundary: the distance metrics fold the norms into
    the contraction where two spare feature columns exist (D <= 30, and 33 <= D <= 62) and add them per
    element otherwise. Integer points: the distances are exact, so the selection (indices, and for the
    distances the values) equals the oracle's; rbf values are fp32 exps of exact distances."""
    X = int_points(60 + D, (300, D), -4, 4)
    Y = int_points(61 + D, (1100, D), -4, 4)
    v, i = ops.pairwise_topk(X.to(DEV), Y.to(DEV), Score(metric, gamma=0.02), 16, metric == "linear")
    ov, oi = oracle.topk(oracle.Problem(X, Y, metric=metric, gamma=0.02), 16, metric == "linear")
    np.testing.assert_array_equal(i.cpu().numpy(), oi)
    if metric == "rbf":
        assert_close(v, ov, TOL_F32_FWD, "rbf topk values")
    else:
        np.testing.assert_array_equal(v.cpu().double().numpy(), ov)


@pytest.mark.parametrize("D", [16, 32, 48])
def test_topk_tc_same_points_exact(oracle, D):
    """X and Y the same tensor (self k-NN, every row's own point at distance 0 comes first among its
    ties): with folded norms the two operand sides differ, so they are split separately."""
    X = int_points(70 + D, (700, D), -3, 3).to(DEV)
    v, i = ops.pairwise_topk(X, X, Score("sqeuclidean"), 8, False)
    Xc = X.cpu()
    ov, oi = oracle.topk(oracle.Problem(Xc, Xc, metric="sqeuclidean"), 8, False)
    np.testing.assert_array_equal(i.cpu().numpy(), oi)
    np.testing.assert_array_equal(v.cpu().double().numpy(), ov)


@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("metric", ["sqeuclidean", "linear", "rbf"])
def test_topk_float(oracle, metric, affine):
    """Real-valued points: the selected values match within tolerance and every returned index
    carries the value returned beside it (near-ties may order differently in fp32)."""
    X, Y, _, sc = problem("ragged_split", torch.float32, metric, affine, False)
    k = 8
    v, i = ops.pairwise_topk(X.to(DEV), Y.to(DEV), gpu_score(sc), k, False)
    pb = oracle_problem(oracle, X, Y, sc)
    ov, oi = oracle.topk(pb, k, False)
    assert_close(v, ov, TOL_F32_FWD, "topk values")
    ii = i.cpu().numpy()
    for r in range(0, X.shape[0], 7):
        for t in range(k):
            assert abs(oracle.pair_score(pb, r, ii[r, t]) - float(v[r, t])) <= 1e-4 * (1 + abs(float(v[r, t])))
        assert len(set(ii[r].tolist())) == k


@pytest.mark.parametrize("dt", [torch.float32, torch.float64])
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("metric", ["sqeuclidean", "linear", "rbf"])
def test_topk_backward(oracle, metric, affine, dt):
    X, Y, _, sc = problem("ragged_split", dt, metric, affine, False)
    k = 5
    v, i = ops.pairwise_topk(X.to(DEV), Y.to(DEV), gpu_score(sc), k, False)
    gv = gen(51, (X.shape[0], k), dt)
    g = ops.pairwise_topk_backward(X.to(DEV), Y.to(DEV), gpu_score(sc), k, i, gv.to(DEV))
    pb = oracle_problem(oracle, X, Y, sc)
    # the oracle differentiates through the same selected pairs (indices are not differentiated)
    want = oracle.topk_backward(pb, k, i.cpu().numpy(), gv)
    pl = Plain(X, Y, dtype=dt, **sc)
    sel = pl.scores().gather(1, i.cpu())
    compare_grads(g, want, tols(dt)[1], "topk", pl.grads(sel, gv))


# ------------------------------------------------------------------------------------------------
# edge cases, autograd surface, determinism, native path
# ------------------------------------------------------------------------------------------------


def test_edge_single_point_exclude_self(oracle):
    z = torch.ones(1, 4, device=DEV)
    lse = ops.pairwise_logsumexp(z, z, Score("linear"), True)
    assert lse.item() == float("-inf")
    g = ops.pairwise_logsumexp_backward(z, z, Score("linear"), lse, torch.ones(1, device=DEV), True, same=True)
    assert torch.all(g["dX"] == 0)


@pytest.mark.parametrize("N,M,D,C", [(1, 1, 1, 1), (1, 77, 2, 3), (77, 1, 7, 1), (5, 3, 64, 64), (129, 65, 1, 64)])
def test_edge_shapes(oracle, N, M, D, C):
    X, Y, V = gen(61, (N, D), torch.float32), gen(62, (M, D), torch.float32), gen(63, (M, C), torch.float32)
    sc = dict(metric="rbf", gamma=0.3, scale=1.0, apply_exp=False)
    pb = oracle.Problem(X, Y, **sc)
    out = ops.pairwise_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))
    check(out, oracle.matmul(pb, V), Plain(X, Y, V=V, **sc).matmul().detach(), TOL_F32_FWD, "edge matmul")
    o, l = ops.pairwise_softmax_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))
    oo, ol = oracle.softmax_matmul(pb, V)
    pl = Plain(X, Y, V=V, **sc)
    p_o, _ = pl.softmax_matmul()
    check(o, oo, p_o.detach(), TOL_F32_FWD, "edge softmax")
    G = gen(64, (N, C), torch.float32)
    g = ops.pairwise_softmax_matmul_backward(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc), o, l, G.to(DEV))
    zero = {}
    if M == 1:  # one column: P = 1, dS = dP - delta = 0, so dX = dY = 0 up to rounding (size of the terms)
        t = float(G.abs().max() * V.abs().max()) * 2 * 0.3
        zero = {"dX": t * float((X.abs().max() + Y.abs().max())), "dY": t * float((X.abs().max() + Y.abs().max()))}
    compare_grads(g, oracle.softmax_matmul_backward(pb, V, oo, ol, G), TOL_F32_GRAD, "edge softmax",
                  pl.grads(p_o, G), zero_scale=zero)


def test_softmax_rows_sum_to_one_on_gpu():
    X, Y = gen(71, (300, 8), torch.float32).to(DEV), gen(72, (900, 8), torch.float32).to(DEV)
    out, _ = ops.pairwise_softmax_matmul(X, Y, torch.ones(900, 1, device=DEV), Score("sqeuclidean", scale=-0.5))
    assert torch.allclose(out, torch.ones_like(out), rtol=0, atol=1e-5)


def test_same_points_autograd_sums_both_sides(oracle):
    import lazy_score_matrix_gb300 as tp
    z0 = torch.nn.functional.normalize(gen(81, (333, 64), torch.float32), dim=1)
    z = z0.to(DEV).requires_grad_(True)
    lse = (tp.lazy(z, z, "linear") / 0.07).logsumexp(-1, exclude_self=True)
    (-lse.mean()).backward()
    pb = oracle.Problem(z0, z0, metric="linear", scale=1 / 0.07)
    ol = oracle.logsumexp(pb, True)
    g = oracle.logsumexp_backward(pb, ol, np.full(333, -1 / 333), True)
    assert_close(lse, ol, TOL_F32_FWD, "lse")
    assert_close(z.grad, g["dX"] + g["dY"], TOL_F32_GRAD, "z.grad")


def test_lazy_expression_folding_and_param_grads(oracle):
    import lazy_score_matrix_gb300 as tp
    X0, Y0 = gen(91, (150, 6), torch.float64), gen(92, (210, 6), torch.float64)
    b0, c0 = gen(93, (150,), torch.float64), gen(94, (210,), torch.float64)
    X, Y = X0.to(DEV).requires_grad_(True), Y0.to(DEV).requires_grad_(True)
    b, c = b0.to(DEV).requires_grad_(True), c0.to(DEV).requires_grad_(True)
    tau = 0.8
    loss = -(((-0.5 / tau) * tp.lazy(X, Y, "sqeuclidean")).add_rows(b).add_columns(c)).logsumexp(-1).mean()
    loss.backward()
    pb = oracle.Problem(X0, Y0, metric="sqeuclidean", scale=-0.5 / tau, row_bias=b0, col_bias=c0)
    ol = oracle.logsumexp(pb)
    g = oracle.logsumexp_backward(pb, ol, np.full(150, -1 / 150))
    assert abs(loss.item() - (-ol.mean())) < 1e-12 * abs(ol.mean()) + 1e-12
    for got, k in ((X.grad, "dX"), (Y.grad, "dY"), (b.grad, "d_row_bias"), (c.grad, "d_col_bias")):
        assert_close(got, g[k], TOL_F64, k)
    with pytest.raises(NotImplementedError):
        (tp.lazy(X, Y).add_rows(b) * 2.0)


def test_kernel_timer_times_every_launch():
    lib = _lib.load()
    X, Y, V, sc = problem("wide", torch.float32, "linear", False, False)
    Xd, Yd, Vd = X.to(DEV), Y.to(DEV), V.to(DEV)
    ops.pairwise_softmax_matmul(Xd, Yd, Vd, gpu_score(sc))
    torch.cuda.synchronize()
    _lib.launch_count(reset=True)
    _lib.check(lib.tp_timer_start(3), "tp_timer_start")
    for _ in range(2):
        ops.pairwise_softmax_matmul(Xd, Yd, Vd, gpu_score(sc))
    n = lib.tp_timer_stop()
    launched = _lib.launch_count()
    assert n == min(launched, 3) and launched >= 2
    name, ms = ctypes.c_char_p(), ctypes.c_float()
    for i in range(n):
        _lib.check(lib.tp_timer_read(i, ctypes.byref(name), ctypes.byref(ms)), "tp_timer_read")
        assert name.value and 0.0 < ms.value < 1e3
    assert lib.tp_timer_read(n, ctypes.byref(name), ctypes.byref(ms)) == _lib.TP_ERR_INVALID_ARG
    # a stopped timer records nothing more
    ops.pairwise_softmax_matmul(Xd, Yd, Vd, gpu_score(sc))
    assert lib.tp_timer_stop() == n


def test_deterministic_and_native(oracle):
    X, Y, V, sc = problem("wide", torch.float32, "linear", False, False)
    _lib.launch_count(reset=True)
    a = ops.pairwise_softmax_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))[0]
    b = ops.pairwise_softmax_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))[0]
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert _lib.launch_count() >= 2
    G = gen(99, a.shape, torch.float32).to(DEV)
    l = ops.pairwise_softmax_matmul(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc))[1]
    g1 = ops.pairwise_softmax_matmul_backward(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc), a, l, G)
    g2 = ops.pairwise_softmax_matmul_backward(X.to(DEV), Y.to(DEV), V.to(DEV), gpu_score(sc), a, l, G)
    for k in ("dX", "dY", "dV"):
        assert torch.equal(g1[k], g2[k]), k


@pytest.mark.parametrize("apply_exp", [False, True])
@pytest.mark.parametrize("exclude_self", [False, True])
@pytest.mark.parametrize("metric", ["sqeuclidean", "linear", "rbf"])
@pytest.mark.parametrize("dt", [torch.float32, torch.float64])
@pytest.mark.parametrize("ND", [(300, 16), (257, 64), (70, 3)])
def test_logsumexp_same_points_symmetric(oracle, ND, dt, metric, exclude_self, apply_exp):
    """X and Y the same points with no row/column parameters: libtp computes the summed gradient
    dX + dY in one symmetric sweep; it must equal the oracle's row and column loops added."""
    N, D = ND
    X = gen(101, (N, D), dt)
    scale = (-0.5 if metric == "sqeuclidean" else 0.5) / D ** 0.5 * (0.5 if apply_exp else 1.0)
    sc = dict(metric=metric, gamma=0.5 / D, scale=scale if metric != "rbf" else 0.8, apply_exp=apply_exp)
    gl = gen(102, (N,), dt)
    Xd = X.to(DEV)
    lse = ops.pairwise_logsumexp(Xd, Xd, gpu_score(sc), exclude_self)
    g = ops.pairwise_logsumexp_backward(Xd, Xd, gpu_score(sc), lse, gl.to(DEV), exclude_self, same=True)
    pb = oracle.Problem(X, X, **sc)
    ol = oracle.logsumexp(pb, exclude_self)
    og = oracle.logsumexp_backward(pb, ol, gl, exclude_self)
    ftol, gtol = tols(dt)
    pl = Plain(X, X, dtype=dt, same=True, **sc)
    p_lse = pl.logsumexp(exclude_self)
    check(lse, ol, p_lse.detach(), ftol, "lse")
    check(g["dX"], og["dX"] + og["dY"], pl.grads(p_lse, gl)["dX"], gtol, "dX + dY")
