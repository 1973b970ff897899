"""Torch-tensor entry points over the C ABI: argument checks, output and workspace allocation from
PyTorch's caching allocator, the current CUDA stream, and the libtp call. Every step of the
computation runs in libtp's kernels; nothing here computes on the data.

Each function mirrors one C entry point of include/tp.h (same name without the ``tp_`` prefix).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

_DT = {torch.float32: _lib.TP_F32, torch.float64: _lib.TP_F64}


@dataclass
class Score:
    """The canonical score: base (metric), then scale * w_row * w_col * base + b_row + b_col, then
    an optional exp (torchpairwise guide "Score Expressions"); optionally a pair mask ("all",
    "causal": j <= i, "band": |i - j| <= band, "same_group": row_group[i] == col_group[j], int32 ids)
    whose masked pairs leave the consumer's reduction."""
    metric: str = "linear"
    gamma: float = 1.0
    scale: float = 1.0
    apply_exp: bool = False
    row_bias: Optional[torch.Tensor] = None
    col_bias: Optional[torch.Tensor] = None
    row_weight: Optional[torch.Tensor] = None
    col_weight: Optional[torch.Tensor] = None
    pair_mask: str = "all"
    band: int = 0
    row_group: Optional[torch.Tensor] = None
    col_group: Optional[torch.Tensor] = None

    def params(self):
        return (self.row_bias, self.col_bias, self.row_weight, self.col_weight)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libtp runs on CUDA tensors only (no CPU fallback)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def _contig(t, dtype, name, shape=None):
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.contiguous()


class _Call:
    """Marshalled problem: the tp_pairs / tp_score structs plus the tensors they point into."""

    def __init__(self, X, Y, score: Score):
        if X.dim() != 2 or Y.dim() != 2 or X.shape[1] != Y.shape[1]:
            raise ValueError("X [N,D] and Y [M,D] expected")
        if X.dtype not in _DT:
            raise TypeError("float32 or float64 expected")
        self.dtype = X.dtype
        self.X = _contig(X, X.dtype, "X")
        self.Y = self.X if Y is X else _contig(Y, X.dtype, "Y")
        self.N, self.D = self.X.shape
        self.M = self.Y.shape[0]
        self.rb = _contig(score.row_bias, self.dtype, "row_bias", (self.N,))
        self.cb = _contig(score.col_bias, self.dtype, "col_bias", (self.M,))
        self.rw = _contig(score.row_weight, self.dtype, "row_weight", (self.N,))
        self.cw = _contig(score.col_weight, self.dtype, "col_weight", (self.M,))
        if score.pair_mask not in _lib.PAIR_MASKS:
            raise ValueError(f"unknown pair mask {score.pair_mask!r}")
        groups = score.pair_mask == "same_group"
        self.rg = _contig(score.row_group, torch.int32, "row_group", (self.N,)) if groups else None
        self.cg = _contig(score.col_group, torch.int32, "col_group", (self.M,)) if groups else None
        if groups and (self.rg is None or self.cg is None):
            raise ValueError("a same_group mask needs row_group [N] and col_group [M]")
        self.device = _need_cuda(self.X, self.Y, self.rb, self.cb, self.rw, self.cw, self.rg, self.cg)
        if score.metric not in _lib.METRICS:
            raise ValueError(f"unknown metric {score.metric!r}")
        self.pairs = _lib.tp_pairs(_DT[self.dtype], self.N, self.M, self.D, self.X.data_ptr(), self.Y.data_ptr())
        self.score = _lib.tp_score(_lib.METRICS[score.metric], float(score.gamma), float(score.scale),
                                   int(bool(score.apply_exp)), _ptr(self.rb), _ptr(self.cb), _ptr(self.rw),
                                   _ptr(self.cw), _lib.PAIR_MASKS[score.pair_mask], int(score.band),
                                   _ptr(self.rg), _ptr(self.cg))
        self.gamma = float(score.gamma)
        self.lib = _lib.load()
        self.stream = ctypes.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)

    def empty(self, *shape, dtype=None):
        return torch.empty(*shape, dtype=dtype or self.dtype, device=self.device)

    def workspace(self, entry: str, C: int = 0, k: int = 0):
        n = self.lib.tp_workspace_size(entry.encode(), ctypes.byref(self.pairs), int(C), int(k))
        if n == ctypes.c_size_t(-1).value:
            raise ValueError(f"invalid sizes for {entry}")
        if n == 0:
            return None, 0
        return torch.empty(n, dtype=torch.uint8, device=self.device), n

    def args(self):
        return ctypes.byref(self.pairs), ctypes.byref(self.score)


def _ws_args(ws):
    t, n = ws
    return _ptr(t), n


# ------------------------------------------------------------------------------------------------
# forward
# ------------------------------------------------------------------------------------------------


def pairwise_matmul(X, Y, V, score: Score):
    c = _Call(X, Y, score)
    V = _contig(V, c.dtype, "V", (c.M, V.shape[-1]))
    _need_cuda(V)
    C = V.shape[1]
    out = c.empty(c.N, C)
    _lib.check(c.lib.tp_pairwise_matmul(*c.args(), _ptr(V), C, _ptr(out), *_ws_args(c.workspace(
        "pairwise_matmul", C)), c.stream), "tp_pairwise_matmul")
    return out


def pairwise_logsumexp(X, Y, score: Score, exclude_self: bool = False):
    c = _Call(X, Y, score)
    lse = c.empty(c.N)
    _lib.check(c.lib.tp_pairwise_logsumexp(*c.args(), int(bool(exclude_self)), _ptr(lse),
                                           *_ws_args(c.workspace("pairwise_logsumexp")), c.stream),
               "tp_pairwise_logsumexp")
    return lse


def pairwise_softmax_matmul(X, Y, V, score: Score):
    c = _Call(X, Y, score)
    V = _contig(V, c.dtype, "V", (c.M, V.shape[-1]))
    _need_cuda(V)
    C = V.shape[1]
    out = c.empty(c.N, C)
    lse = c.empty(c.N)
    _lib.check(c.lib.tp_pairwise_softmax_matmul(*c.args(), _ptr(V), C, _ptr(out), _ptr(lse),
                                                *_ws_args(c.workspace("pairwise_softmax_matmul", C)), c.stream),
               "tp_pairwise_softmax_matmul")
    return out, lse


def pairwise_displacement(X, Y, score: Score):
    c = _Call(X, Y, score)
    out = c.empty(c.N, c.D)
    _lib.check(c.lib.tp_pairwise_displacement(*c.args(), _ptr(out), *_ws_args(c.workspace("pairwise_displacement")),
                                              c.stream), "tp_pairwise_displacement")
    return out


def svgd_direction(x, score_values, gamma: float, y=None):
    """phi_i = (1/n) sum_j k(x_j, x_i) (score_j - 2 gamma (x_j - x_i)), one sweep."""
    y = x if y is None else y
    c = _Call(x, y, Score("rbf", gamma=gamma))
    sv = _contig(score_values, c.dtype, "score", (c.M, c.D))
    _need_cuda(sv)
    phi = c.empty(c.N, c.D)
    _lib.check(c.lib.tp_svgd_direction(ctypes.byref(c.pairs), float(gamma), _ptr(sv), _ptr(phi),
                                       *_ws_args(c.workspace("svgd_direction")), c.stream), "tp_svgd_direction")
    return phi


def pairwise_topk(X, Y, score: Score, k: int, largest: bool = False):
    c = _Call(X, Y, score)
    vals = c.empty(c.N, k)
    idx = c.empty(c.N, k, dtype=torch.int64)
    _lib.check(c.lib.tp_pairwise_topk(*c.args(), int(k), int(bool(largest)), _ptr(vals), _ptr(idx),
                                      *_ws_args(c.workspace("pairwise_topk", 0, k)), c.stream), "tp_pairwise_topk")
    return vals, idx


# ------------------------------------------------------------------------------------------------
# backward (gradients are allocated for the requested outputs only; `same` = X and Y are the same
# points and one summed gradient is wanted for them)
# ------------------------------------------------------------------------------------------------


def _grad_outputs(c: _Call, want, C: int = 0, same: bool = False):
    wX, wY, wV, wrb, wcb, wrw, wcw = want
    g = {}
    if same and (wX or wY):
        g["dX"] = c.empty(c.N, c.D)
        g["dY"] = g["dX"]
    else:
        g["dX"] = c.empty(c.N, c.D) if wX else None
        g["dY"] = c.empty(c.M, c.D) if wY else None
    g["dV"] = c.empty(c.M, C) if (wV and C) else None
    g["d_row_bias"] = c.empty(c.N) if (wrb and c.rb is not None) else None
    g["d_col_bias"] = c.empty(c.M) if (wcb and c.cb is not None) else None
    g["d_row_weight"] = c.empty(c.N) if (wrw and c.rw is not None) else None
    g["d_col_weight"] = c.empty(c.M) if (wcw and c.cw is not None) else None
    return g


def _gp(g):
    return [_ptr(g["d_row_bias"]), _ptr(g["d_col_bias"]), _ptr(g["d_row_weight"]), _ptr(g["d_col_weight"])]


ALL = (True,) * 7


def pairwise_matmul_backward(X, Y, V, score: Score, grad_out, want=ALL, same=False):
    c = _Call(X, Y, score)
    V = _contig(V, c.dtype, "V", (c.M, V.shape[-1]))
    C = V.shape[1]
    go = _contig(grad_out, c.dtype, "grad_out", (c.N, C))
    _need_cuda(V, go)
    g = _grad_outputs(c, want, C, same)
    _lib.check(c.lib.tp_pairwise_matmul_backward(*c.args(), _ptr(V), C, _ptr(go), _ptr(g["dX"]), _ptr(g["dY"]),
                                                 _ptr(g["dV"]), *_gp(g),
                                                 *_ws_args(c.workspace("pairwise_matmul_backward", C)), c.stream),
               "tp_pairwise_matmul_backward")
    return g


def pairwise_logsumexp_backward(X, Y, score: Score, lse, grad_lse, exclude_self=False, want=ALL, same=False):
    c = _Call(X, Y, score)
    lse = _contig(lse, c.dtype, "lse", (c.N,))
    gl = _contig(grad_lse, c.dtype, "grad_lse", (c.N,))
    _need_cuda(lse, gl)
    g = _grad_outputs(c, want, 0, same)
    _lib.check(c.lib.tp_pairwise_logsumexp_backward(*c.args(), int(bool(exclude_self)), _ptr(lse), _ptr(gl),
                                                    _ptr(g["dX"]), _ptr(g["dY"]), *_gp(g),
                                                    *_ws_args(c.workspace("pairwise_logsumexp_backward")), c.stream),
               "tp_pairwise_logsumexp_backward")
    return g


def pairwise_softmax_matmul_backward(X, Y, V, score: Score, out, lse, grad_out, want=ALL, same=False):
    c = _Call(X, Y, score)
    V = _contig(V, c.dtype, "V", (c.M, V.shape[-1]))
    C = V.shape[1]
    out = _contig(out, c.dtype, "out", (c.N, C))
    lse = _contig(lse, c.dtype, "lse", (c.N,))
    go = _contig(grad_out, c.dtype, "grad_out", (c.N, C))
    _need_cuda(V, out, lse, go)
    g = _grad_outputs(c, want, C, same)
    _lib.check(c.lib.tp_pairwise_softmax_matmul_backward(
        *c.args(), _ptr(V), C, _ptr(out), _ptr(lse), _ptr(go), _ptr(g["dX"]), _ptr(g["dY"]), _ptr(g["dV"]),
        *_gp(g), *_ws_args(c.workspace("pairwise_softmax_matmul_backward", C)), c.stream),
        "tp_pairwise_softmax_matmul_backward")
    return g


def pairwise_displacement_backward(X, Y, score: Score, grad_out, want=ALL, same=False):
    c = _Call(X, Y, score)
    go = _contig(grad_out, c.dtype, "grad_out", (c.N, c.D))
    _need_cuda(go)
    g = _grad_outputs(c, want, 0, same)
    _lib.check(c.lib.tp_pairwise_displacement_backward(*c.args(), _ptr(go), _ptr(g["dX"]), _ptr(g["dY"]), *_gp(g),
                                                       *_ws_args(c.workspace("pairwise_displacement_backward")),
                                                       c.stream), "tp_pairwise_displacement_backward")
    return g


def pairwise_topk_backward(X, Y, score: Score, k, indices, grad_values, want=ALL, same=False):
    c = _Call(X, Y, score)
    idx = _contig(indices, torch.int64, "indices", (c.N, k))
    gv = _contig(grad_values, c.dtype, "grad_values", (c.N, k))
    _need_cuda(idx, gv)
    g = _grad_outputs(c, want, 0, same)
    _lib.check(c.lib.tp_pairwise_topk_backward(*c.args(), int(k), _ptr(idx), _ptr(gv), _ptr(g["dX"]), _ptr(g["dY"]),
                                               *_gp(g), *_ws_args(c.workspace("pairwise_topk_backward", 0, k)),
                                               c.stream), "tp_pairwise_topk_backward")
    return g
