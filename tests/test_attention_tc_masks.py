"""GPU parity of the tensor-core attention path under index pair masks (torchpairwise guide "Using
Torchpairwise in Models", Task Map: softmax_matmul(V, mask=tp.masks.causal()); Score Expressions: band):
softmax_matmul and its backward for fp32, D = C = 64, against the oracle at the fp32 tolerances, on ragged
shapes with N < M, N = M and N > M, band widths from 0 to wider than a tile, rows and columns that the
band leaves empty, and the summed gradient of the same points on both sides."""
import ctypes

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


def _kernels(fn):
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


def _check(oracle, Q, K, V, G, mask, band=0, what="", grad_floor=None, zero_rows=0):
    """grad_floor: {key: magnitude} for gradients that are zero by the mathematics (measured against the
    size of the terms that cancel); zero_rows: the first rows of dX are such gradients (rows that keep one
    key), measured that way, the other rows at the tolerance."""
    grad_floor = grad_floor or {}
    sc = Score("linear", scale=0.125, pair_mask=mask, band=band)
    out, lse = ops.pairwise_softmax_matmul(Q.to(DEV), K.to(DEV), V.to(DEV), sc)
    g = ops.pairwise_softmax_matmul_backward(Q.to(DEV), K.to(DEV), V.to(DEV), sc, out, lse, G.to(DEV))
    pb = oracle.Problem(Q, K, metric="linear", scale=0.125, pair_mask=mask, band=band)
    oo, ol = oracle.softmax_matmul(pb, V)
    # the fp32 tolerances, or twice what the plain dense fp32 evaluation reaches on these inputs where
    # that is larger (tests/_plain.py), at the floor of 1e-3 of each output's largest magnitude
    pl = Plain(Q, K, V=V, metric="linear", scale=0.125, pair_mask=mask, band=band)
    p_out, p_lse = pl.softmax_matmul()
    assert_close(out, oo, achievable(p_out.detach(), oo, TOL_F32_FWD, slack=TC_SLACK), f"{what} out")
    assert_close(lse, ol, achievable(p_lse.detach(), ol, TOL_F32_FWD, slack=TC_SLACK), f"{what} lse")
    og = oracle.softmax_matmul_backward(pb, V, out.double().cpu().numpy(), lse.double().cpu().numpy(), G)
    pg = pl.grads(p_out, G)
    for k in ("dX", "dY", "dV"):
        got, want, pk = g[k], og[k], pg[k].numpy()
        if k == "dX" and zero_rows:
            t = 0.125 * float(G.abs().max() * V.abs().max() * K.abs().max())
            assert_close(got[:zero_rows], want[:zero_rows], TOL_F32_GRAD, f"{what} dX (one key)", abs_floor=t)
            got, want, pk = got[zero_rows:], want[zero_rows:], pk[zero_rows:]
        fl = grad_floor.get(k, 0.0)
        assert_close(got, want, achievable(pk, want, TOL_F32_GRAD, abs_floor=fl, slack=TC_SLACK), f"{what} {k}", abs_floor=fl)
    return out, lse, g


@pytest.mark.parametrize("N,M", [(5, 5), (129, 129), (300, 517), (517, 300), (2000, 2000)])
def test_causal_attention_tc_matches_oracle(oracle, N, M):
    Q, K, V, G = _n(1, N, 64), _n(2, M, 64), _n(3, M, 64), _n(4, N, 64)
    # row 0 keeps key 0 alone: P = 1, dS = dP - delta = 0, so dQ_0 = 0 up to rounding
    _check(oracle, Q, K, V, G, "causal", what=f"causal {N}x{M}", zero_rows=1)


@pytest.mark.parametrize("w", [0, 17, 64, 200])
@pytest.mark.parametrize("N,M", [(300, 517), (517, 300)])
def test_band_attention_tc_matches_oracle(oracle, N, M, w):
    Q, K, V, G = _n(11, N, 64), _n(12, M, 64), _n(13, M, 64), _n(14, N, 64)
    zero = {}
    if w == 0:  # one kept key per row: P = 1, dS = dP - delta = 0, so dQ = dK = 0 up to rounding
        t = 0.125 * float(G.abs().max() * V.abs().max())
        zero = {"dX": t * float(K.abs().max()), "dY": t * float(Q.abs().max())}
    out, lse, g = _check(oracle, Q, K, V, G, "band", band=w, what=f"band {w} {N}x{M}", grad_floor=zero)
    if N > M + w:  # rows i > M - 1 + w keep no key: lse -inf, output 0, no gradient
        empty = slice(M + w, N)
        assert torch.isneginf(lse[empty]).all()
        assert torch.all(out[empty] == 0) and torch.all(g["dX"][empty] == 0)
    if M > N + w:  # keys j > N - 1 + w meet no query
        assert torch.all(g["dY"][N + w:] == 0) and torch.all(g["dV"][N + w:] == 0)


@pytest.mark.parametrize("s", [0.4, 1.0])
def test_causal_self_attention_tc_summed(oracle, s):
    # the same points on both sides. At unit scale |x|^2 / 8 ~ 8 sits on the diagonal against ~N(0, 1)
    # off it: the early causal rows hold nearly all their mass on the self pair and dS = P (dP - delta)
    # cancels far below its terms, which fp32 itself does not resolve to 5e-4; at 0.4 the diagonal is
    # ~1.3, well inside fp32's conditioning
    X, V, G = _n(21, 390, 64, s=s), _n(22, 390, 64), _n(23, 390, 64)
    Xd = X.to(DEV)
    sc = Score("linear", scale=0.125, pair_mask="causal")
    out, lse = ops.pairwise_softmax_matmul(Xd, Xd, V.to(DEV), sc)
    pb = oracle.Problem(X, X, metric="linear", scale=0.125, pair_mask="causal")
    oo, _ = oracle.softmax_matmul(pb, V)
    pl = Plain(X, X, V=V, metric="linear", scale=0.125, pair_mask="causal", same=True)
    p_out, _ = pl.softmax_matmul()
    assert_close(out, oo, achievable(p_out.detach(), oo, TOL_F32_FWD, slack=TC_SLACK), "self out")
    og = oracle.softmax_matmul_backward(pb, V, out.double().cpu().numpy(), lse.double().cpu().numpy(), G)
    gs = ops.pairwise_softmax_matmul_backward(Xd, Xd, V.to(DEV), sc, out, lse, G.to(DEV), same=True)
    pg = pl.grads(p_out, G)
    want = og["dX"] + og["dY"]
    assert_close(gs["dX"], want, achievable(pg["dX"], want, TOL_F32_GRAD, slack=TC_SLACK), "self summed")
    assert_close(gs["dV"], og["dV"], achievable(pg["dV"], og["dV"], TOL_F32_GRAD, slack=TC_SLACK), "self dV")
    names = _kernels(lambda: ops.pairwise_softmax_matmul_backward(Xd, Xd, V.to(DEV), sc, out, lse, G.to(DEV),
                                                                  same=True))
    assert {"attn_bwd_row_tc", "attn_bwd_col_tc"} <= names


@pytest.mark.parametrize("mask,tc", [("causal", True), ("band", True), ("same_group", False)])
def test_index_masks_run_on_the_tensor_cores(mask, tc):
    Q, K, V, G = (_n(s, 300, 64).to(DEV) for s in (31, 32, 33, 34))
    grp = (torch.arange(300, dtype=torch.int32) % 3).to(DEV)
    kw = dict(row_group=grp, col_group=grp) if mask == "same_group" else {}
    sc = Score("linear", scale=0.125, pair_mask=mask, band=9, **kw)
    holder = {}

    def fwd():
        holder["o"], holder["l"] = ops.pairwise_softmax_matmul(Q, K, V, sc)

    names = _kernels(fwd) | _kernels(
        lambda: ops.pairwise_softmax_matmul_backward(Q, K, V, sc, holder["o"], holder["l"], G))
    want = {"attn_fwd_tc", "attn_bwd_row_tc", "attn_bwd_col_tc"}
    assert (want <= names) == tc, names


@pytest.mark.parametrize("D", [64, 16])
def test_band_wider_than_the_problem_keeps_every_pair(oracle, D):
    # widths of N + M and far beyond (the tensor-core schedule adds the width to point indices): every
    # pair is kept, on the tensor cores (D = 64) and on the streamed sweeps (D = 16)
    N, M = 300, 517
    C = 64 if D == 64 else 8
    Q, K, V, G = _n(41, N, D), _n(42, M, D), _n(43, M, C), _n(44, N, C)
    unmasked, _ = oracle.softmax_matmul(oracle.Problem(Q, K, metric="linear", scale=0.125), V)
    for w in (N + M, 2 ** 40, 2 ** 62):
        out, _, _ = _check(oracle, Q, K, V, G, "band", band=w, what=f"band {w} D {D}")
        p_un, _ = Plain(Q, K, V=V, metric="linear", scale=0.125).softmax_matmul()
        assert_close(out, unmasked, achievable(p_un.detach(), unmasked, TOL_F32_FWD, slack=TC_SLACK), f"band {w} D {D} vs unmasked")
