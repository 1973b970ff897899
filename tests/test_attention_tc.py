"""GPU parity of the tensor-core attention path: softmax_matmul and its backward for fp32, D = C = 64,
linear score times a scale, no row/column parameters (the shape of attention in the torchpairwise
guide's Task Map). Ragged shapes from one point up to several tiles per persistent CTA, data scales far
from 1, peaked softmax rows, self-attention on the same points and partial gradient requests, against
the oracle at the fp32 tolerances (1e-4 forward, 5e-4 gradients)."""
import ctypes

import numpy as np
import pytest
import torch

from lazy_score_matrix_gb300 import _lib, ops
from lazy_score_matrix_gb300.ops import Score
from tests._plain import TC_SLACK, Plain, achievable
from tests._util import TOL_F32_FWD, TOL_F32_GRAD, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _n(seed, *shape, s=1.0):
    return s * torch.randn(*shape, generator=torch.Generator().manual_seed(seed), dtype=torch.float32)


def _check(oracle, Q, K, V, G, scale, want=ops.ALL, what="", grad_floor=None):
    """Against the oracle at the fp32 tolerances, or at twice what the plain dense fp32 evaluation
    (tests/_plain.py) reaches on the same inputs where that is larger; floor 1e-3 of the largest
    magnitude of each output. grad_floor: {key: magnitude} for gradients that are zero by the
    mathematics (measured against the size of the terms that cancel)."""
    grad_floor = grad_floor or {}
    sc = Score("linear", scale=scale)
    out, lse = ops.pairwise_softmax_matmul(Q.to(DEV), K.to(DEV), V.to(DEV), sc)
    g = ops.pairwise_softmax_matmul_backward(Q.to(DEV), K.to(DEV), V.to(DEV), sc, out, lse, G.to(DEV), want=want)
    pb = oracle.Problem(Q, K, metric="linear", scale=scale)
    oo, ol = oracle.softmax_matmul(pb, V)
    pl = Plain(Q, K, V=V, metric="linear", scale=scale)
    p_out, p_lse = pl.softmax_matmul()
    assert_close(out, oo, achievable(p_out.detach(), oo, TOL_F32_FWD, slack=TC_SLACK), f"{what} out")
    assert_close(lse, ol, achievable(p_lse.detach(), ol, TOL_F32_FWD, slack=TC_SLACK), f"{what} lse")
    # the backward takes out and lse as inputs: both sides get the same ones (with self-attention dK
    # moves by ~1e-3 for a 1e-6 relative change of out, through delta = dO . out)
    o32, l32 = out.double().cpu().numpy(), lse.double().cpu().numpy()
    og = oracle.softmax_matmul_backward(pb, V, o32, l32, G)
    pg = pl.grads(p_out, G)
    for k in ("dX", "dY", "dV"):
        if g.get(k) is not None:
            fl = grad_floor.get(k, 0.0)
            assert_close(g[k], og[k], achievable(pg[k], og[k], TOL_F32_GRAD, abs_floor=fl, slack=TC_SLACK), f"{what} {k}", abs_floor=fl)
    return g


def _tc_kernels(fn):
    """Names of the kernels fn launches (the library's own timer records each launch)."""
    lib = _lib.load()
    torch.cuda.synchronize()
    _lib.check(lib.tp_timer_start(64), "tp_timer_start")
    fn()
    n = lib.tp_timer_stop()
    names = set()
    name, ms = ctypes.c_char_p(), ctypes.c_float()
    for i in range(n):
        _lib.check(lib.tp_timer_read(i, ctypes.byref(name), ctypes.byref(ms)), "tp_timer_read")
        names.add(name.value.decode())
    return names


@pytest.mark.parametrize("N,M", [(1, 1), (5, 3), (127, 65), (129, 200), (300, 517), (2000, 1500), (3000, 2500)])
def test_attention_tc_matches_oracle(oracle, N, M):
    Q, K, V, G = _n(1, N, 64), _n(2, M, 64), _n(3, M, 64), _n(4, N, 64)
    zero = {}
    if M == 1:  # one key: P = 1, dS = dP - delta = 0, so dQ = dK = 0 up to rounding of |dO| |V| scale |K|
        t = 0.125 * float(G.abs().max() * V.abs().max())
        zero = {"dX": t * float(K.abs().max()), "dY": t * float(Q.abs().max())}
    _check(oracle, Q, K, V, G, 0.125, what=f"{N}x{M}", grad_floor=zero)


def test_attention_tc_runs_on_the_tensor_cores():
    Q, K, V, G = (_n(s, 300, 64).to(DEV) for s in (5, 6, 7, 8))
    sc = Score("linear", scale=0.125)
    holder = {}

    def fwd():
        holder["o"], holder["l"] = ops.pairwise_softmax_matmul(Q, K, V, sc)

    names = _tc_kernels(fwd)
    assert "attn_fwd_tc" in names and "lse_fwd_tc" not in names, names  # one sweep gives out and lse
    names = _tc_kernels(lambda: ops.pairwise_softmax_matmul_backward(Q, K, V, sc, holder["o"], holder["l"], G))
    assert {"attn_bwd_row_tc", "attn_bwd_col_tc"} <= names


@pytest.mark.parametrize("qs,ks,vs,gs", [(1024.0, 1 / 1024.0, 1e-3, 1e3), (1 / 512.0, 256.0, 300.0, 1e-4)])
def test_attention_tc_far_from_unit_scale(oracle, qs, ks, vs, gs):
    # rows far from unit size (split exponents ~20 apart between the two sides), the same scores
    N, M = 260, 333
    Q, K, V, G = _n(11, N, 64, s=qs), _n(12, M, 64, s=ks), _n(13, M, 64, s=vs), _n(14, N, 64, s=gs)
    _check(oracle, Q, K, V, G, 0.125, what="scaled")


@pytest.mark.parametrize("scale", [0.5, 1.0])
def test_attention_tc_peaked_rows(oracle, scale):
    # scores of std 4 or 8 (|S| up to ~22 or ~45), most of each row's mass on a few keys, most P far below
    # fp16's range; at scale 1 rounding S once to fp32 already moves out beyond 1e-4, so there the plain
    # fp32 evaluation's error sets the bound
    N, M = 400, 700
    Q, K, V, G = _n(21, N, 64), _n(22, M, 64), _n(23, M, 64), _n(24, N, 64)
    _check(oracle, Q, K, V, G, scale, what=f"peaked {scale}")


def _mixed_rows(seed, n, d, lo=-20):
    """Rows of N(0, 1) values each scaled by its own power of two in [2^lo, 2^0] (seeded): one matrix
    whose rows span 2^20 in magnitude."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g)
    e = torch.randint(lo, 1, (n, 1), generator=g).float()
    return x * torch.pow(2.0, e)


@pytest.mark.parametrize("which", ["Q", "K", "V", "dO", "all"])
def test_attention_tc_mixed_row_magnitudes(oracle, which):
    # the tensor-core attention gives each matrix ONE power of two and splits its elements into fp16
    # hi + lo; rows far below the matrix's largest keep fewer bits. Rows spread over 2^-20 .. 2^0 in
    # one matrix (or in all four) must still meet the bounds of the unit-scale case.
    N, M = 520, 700
    mats = {"Q": _n(71, N, 64), "K": _n(72, M, 64), "V": _n(73, M, 64), "dO": _n(74, N, 64)}
    for k, (n, seed) in {"Q": (N, 75), "K": (M, 76), "V": (M, 77), "dO": (N, 78)}.items():
        if which in (k, "all"):
            mats[k] = _mixed_rows(seed, n, 64)
    _check(oracle, mats["Q"], mats["K"], mats["V"], mats["dO"], 0.125, what=f"mixed {which}")


def test_attention_tc_zero_rows(oracle):
    N, M = 200, 150
    Q, K, V, G = _n(31, N, 64), _n(32, M, 64), _n(33, M, 64), _n(34, N, 64)
    Q[7] = 0
    K[100] = 0
    V[3] = 0
    G[9] = 0
    _check(oracle, Q, K, V, G, 0.125, what="zero rows")


def test_attention_tc_self_attention_same_points(oracle):
    X = _n(41, 390, 64)
    V, G = _n(42, 390, 64), _n(43, 390, 64)
    Xd = X.to(DEV)
    sc = Score("linear", scale=0.125)
    out, lse = ops.pairwise_softmax_matmul(Xd, Xd, V.to(DEV), sc)
    pb = oracle.Problem(X, X, metric="linear", scale=0.125)
    oo, ol = oracle.softmax_matmul(pb, V)
    pl = Plain(X, X.clone(), V=V, metric="linear", scale=0.125)
    p_out, _ = pl.softmax_matmul()
    assert_close(out, oo, achievable(p_out.detach(), oo, TOL_F32_FWD, slack=TC_SLACK), "self out")
    og = oracle.softmax_matmul_backward(pb, V, out.double().cpu().numpy(), lse.double().cpu().numpy(), G)
    g = ops.pairwise_softmax_matmul_backward(Xd, Xd, V.to(DEV), sc, out, lse, G.to(DEV))
    pg = pl.grads(p_out, G)
    for k in ("dX", "dY", "dV"):
        assert_close(g[k], og[k], achievable(pg[k], og[k], TOL_F32_GRAD, slack=TC_SLACK), f"self {k}")
    # one summed gradient for the shared points (dX and dY in one buffer)
    gs = ops.pairwise_softmax_matmul_backward(Xd, Xd, V.to(DEV), sc, out, lse, G.to(DEV), same=True)
    ps = Plain(X, X, V=V, metric="linear", scale=0.125, same=True)
    p_s, _ = ps.softmax_matmul()
    assert_close(gs["dX"], og["dX"] + og["dY"], achievable(ps.grads(p_s, G)["dX"], og["dX"] + og["dY"], TOL_F32_GRAD, slack=TC_SLACK),
                 "self summed")


@pytest.mark.parametrize("want", [(True, False, False), (False, True, False), (False, False, True),
                                  (False, True, True)])
def test_attention_tc_partial_requests(oracle, want):
    N, M = 333, 444
    Q, K, V, G = _n(51, N, 64), _n(52, M, 64), _n(53, M, 64), _n(54, N, 64)
    g = _check(oracle, Q, K, V, G, 0.125, want=want + (True,) * 4, what=f"want {want}")
    for k, w in zip(("dX", "dY", "dV"), want):
        assert (g[k] is not None) == w


def test_attention_tc_deterministic():
    Q, K, V, G = (_n(s, 1500, 64).to(DEV) for s in (61, 62, 63, 64))
    sc = Score("linear", scale=0.125)
    o1, l1 = ops.pairwise_softmax_matmul(Q, K, V, sc)
    o2, l2 = ops.pairwise_softmax_matmul(Q, K, V, sc)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = ops.pairwise_softmax_matmul_backward(Q, K, V, sc, o1, l1, G)
    g2 = ops.pairwise_softmax_matmul_backward(Q, K, V, sc, o1, l1, G)
    for k in ("dX", "dY", "dV"):
        assert torch.equal(g1[k], g2[k]), k
    assert np.isfinite(g1["dX"].cpu().numpy()).all()
