"""Lazy pairwise scores: bind X and Y, fold the expression nodes, consume once.

Follows the torchpairwise guide "Using Torchpairwise in Models": ``lazy(X, Y, metric)`` is a logical
[N,M] score matrix that is never stored (introduction); arithmetic on it builds a score expression
("Score Expressions": scalar scale, add_rows, add_columns, weight_rows, weight_columns, exp); a
consumer call evaluates it on libtp's fused kernels ("Task Map": softmax_matmul, @ / matmul,
logsumexp with exclude_self, topk / argmin / min, displacement) and first derivatives replay the
pairs in libtp's backward kernels.

The expression is folded into one canonical form, ``S = [exp](scale * w_row * w_col * base + b_row + b_col)``.
Orders that do not fold into it (a scalar applied after a bias, two biases on the same side, an
exp followed by more arithmetic, ...) raise NotImplementedError; the guide sends such expressions
to a tile path, which this library does not have.
"""
from __future__ import annotations

from collections import namedtuple
from dataclasses import dataclass, replace
from typing import Optional

import torch

from . import ops
from .masks import PairMask
from .ops import Score

TopK = namedtuple("TopK", ["values", "indices"])


@dataclass(frozen=True)
class _Meta:
    metric: str
    gamma: float
    scale: float
    apply_exp: bool
    pair: Optional[PairMask] = None

    def score(self, rb, cb, rw, cw) -> Score:
        if self.pair is None:
            return Score(self.metric, self.gamma, self.scale, self.apply_exp, rb, cb, rw, cw)
        return Score(self.metric, self.gamma, self.scale, self.apply_exp, rb, cb, rw, cw, self.pair.kind,
                     self.pair.width, self.pair.row_group, self.pair.col_group)


def _unsupported(what: str):
    raise NotImplementedError(f"{what} does not fold into the fused score form "
                              "[exp](scale * w_row * w_col * base + b_row + b_col)")


class LazyScores:
    """A logical [N,M] pairwise score matrix over X [N,D] and Y [M,D] (never materialised)."""

    def __init__(self, X: torch.Tensor, Y: Optional[torch.Tensor] = None, metric: str = "linear",
                 gamma: float = 1.0):
        self.X = X
        self.Y = X if Y is None else Y
        self._meta = _Meta(metric, float(gamma), 1.0, False)
        self.row_bias = self.col_bias = self.row_weight = self.col_weight = None

    @property
    def shape(self):
        return torch.Size([self.X.shape[0], self.Y.shape[0]])

    def _with(self, **kw) -> "LazyScores":
        o = LazyScores.__new__(LazyScores)
        o.X, o.Y, o._meta = self.X, self.Y, self._meta
        o.row_bias, o.col_bias, o.row_weight, o.col_weight = self.row_bias, self.col_bias, self.row_weight, self.col_weight
        o._row_keep, o._col_keep = getattr(self, "_row_keep", None), getattr(self, "_col_keep", None)
        for k, v in kw.items():
            if k == "meta":
                o._meta = v
            else:
                setattr(o, k, v)
        return o

    # --- expression nodes ----------------------------------------------------------------------
    def __mul__(self, s):
        if isinstance(s, torch.Tensor):
            if s.dim() != 0:
                _unsupported("multiplying by a non-scalar tensor")
            s = float(s)
        if not isinstance(s, (int, float)):
            return NotImplemented
        if self._meta.apply_exp or self.row_bias is not None or self.col_bias is not None:
            _unsupported("a scalar factor after a bias or exp")
        return self._with(meta=replace(self._meta, scale=self._meta.scale * float(s)))

    __rmul__ = __mul__

    def __truediv__(self, t):
        if isinstance(t, torch.Tensor):
            t = float(t)
        return self * (1.0 / float(t))

    def __neg__(self):
        return self * -1.0

    def weight_rows(self, w: torch.Tensor) -> "LazyScores":
        if self._meta.apply_exp or self.row_bias is not None or self.col_bias is not None or self.row_weight is not None:
            _unsupported("weight_rows after a bias, exp or another row weight")
        return self._with(row_weight=w)

    def weight_columns(self, w: torch.Tensor) -> "LazyScores":
        if self._meta.apply_exp or self.row_bias is not None or self.col_bias is not None or self.col_weight is not None:
            _unsupported("weight_columns after a bias, exp or another column weight")
        return self._with(col_weight=w)

    def add_rows(self, b: torch.Tensor) -> "LazyScores":
        if self._meta.apply_exp or self.row_bias is not None:
            _unsupported("add_rows after exp or another row bias")
        return self._with(row_bias=b)

    def add_columns(self, b: torch.Tensor) -> "LazyScores":
        if self._meta.apply_exp or self.col_bias is not None:
            _unsupported("add_columns after exp or another column bias")
        return self._with(col_bias=b)

    def exp(self) -> "LazyScores":
        if self._meta.apply_exp:
            _unsupported("exp of exp")
        return self._with(meta=replace(self._meta, apply_exp=True))

    def score(self) -> Score:
        return self._meta.score(self.row_bias, self.col_bias, self.row_weight, self.col_weight)

    @property
    def T(self) -> "LazyScores":
        """The transposed [M,N] matrix: S^T_ji = S_ij. Exact, because every base is symmetric in its two
        points; the row and column parameters trade places."""
        o = self._with(row_bias=self.col_bias, col_bias=self.row_bias, row_weight=self.col_weight,
                       col_weight=self.row_weight)
        if self._meta.pair is not None:
            o._meta = replace(self._meta, pair=self._meta.pair.transposed())
        o.X, o.Y = self.Y, self.X
        return o

    def mask_pairs(self, mask: PairMask) -> "LazyScores":
        """Remove the pairs a pair mask (``masks.causal()``, ``masks.band(w)``, ``masks.same_group(g)``)
        masks from every consumer of this score (Task Map: softmax_matmul with mask=...)."""
        if not isinstance(mask, PairMask):
            raise TypeError("mask_pairs expects a masks.PairMask")
        if self._meta.pair is not None:
            _unsupported("a second pair mask")
        return self._with(meta=replace(self._meta, pair=mask))

    def mask_columns(self, keep: torch.Tensor) -> "LazyScores":
        """Boolean column mask ("Score Expressions": boolean row/column masks stay fused): columns with
        keep[j] False drop out of every reduction over a row. Lowered onto the fused form: a column
        bias of -inf for logsumexp / softmax_matmul (their terms exp(-inf) = 0) and for K @ V, sum and
        mean of an exp score; a zero column weight for K @ V, sum and mean without exp or biases; a
        column bias of +inf (smallest) or -inf (largest) for top-k, so masked columns are never chosen
        while k does not exceed the kept columns. logsumexp / softmax_matmul of an exp score cannot
        be masked this way (exp(-inf) = 0 is still a term) and raise NotImplementedError."""
        keep = keep.to(device=self.Y.device, dtype=torch.bool)
        if keep.shape != (self.Y.shape[0],):
            raise ValueError("mask_columns: keep must be a bool vector of length M")
        o = self._with()
        o._col_keep = keep if getattr(self, "_col_keep", None) is None else (self._col_keep & keep)
        return o

    def mask_rows(self, keep: torch.Tensor) -> "LazyScores":
        """Boolean row mask: rows with keep[i] False drop out of every reduction over a column (dim=-2)."""
        keep = keep.to(device=self.X.device, dtype=torch.bool)
        if keep.shape != (self.X.shape[0],):
            raise ValueError("mask_rows: keep must be a bool vector of length N")
        o = self._with()
        o._row_keep = keep if getattr(self, "_row_keep", None) is None else (self._row_keep & keep)
        return o

    def _masked(self, kind: str) -> "LazyScores":
        """The expression with the column mask folded in, for a reduction over each row of `kind`
        ("lse", "sum", "topk_min", "topk_max"). A row mask only affects reductions over columns."""
        keep = getattr(self, "_col_keep", None)
        if keep is None:
            return self
        dtype = self.Y.dtype
        if kind == "lse" and self._meta.apply_exp:
            _unsupported("a column mask on logsumexp / softmax_matmul of an exp score (exp(-inf) = 0 still counts)")
        if kind in ("lse", "topk_max", "topk_min") or (kind == "sum" and self._meta.apply_exp):
            fill = float("inf") if kind == "topk_min" else float("-inf")
            extra = torch.where(keep, torch.zeros((), dtype=dtype, device=keep.device),
                                torch.full((), fill, dtype=dtype, device=keep.device))
            cb = extra if self.col_bias is None else self.col_bias + extra
            o = self._with(col_bias=cb)
        elif kind == "sum":
            if self.row_bias is not None or self.col_bias is not None:
                _unsupported("a column mask on K @ V with biases and no exp")
            w = keep.to(dtype)
            o = self._with(col_weight=w if self.col_weight is None else self.col_weight * w)
        else:
            raise ValueError(kind)
        o._col_keep = None
        return o

    def _params(self):
        return (self.row_bias, self.col_bias, self.row_weight, self.col_weight)

    # --- consumers -----------------------------------------------------------------------------
    def matmul(self, V: torch.Tensor) -> torch.Tensor:
        """out_i = sum_j S_ij V_j ("Task Map", kernel attention; [V | ones] gives the row mass)."""
        e = self._masked("sum")
        return _MatmulFn.apply(e.X, e.Y, V, *e._params(), e._meta)

    def sum(self, dim: int = -1) -> torch.Tensor:
        """sum_j S_ij per row (dim=-1) or sum_i S_ij per column (dim=-2): K @ ones."""
        if dim in (-2, 0):
            return self._col_view().sum(-1)
        if dim not in (-1, 1):
            raise ValueError("sum: dim must be -1 or -2")
        ones = torch.ones(self.Y.shape[0], 1, dtype=self.Y.dtype, device=self.Y.device)
        return self.matmul(ones)[:, 0]

    def mean(self, dim: int = -1) -> torch.Tensor:
        """Mean over each row (dim=-1) or column (dim=-2), over the kept entries under a mask."""
        if dim in (-2, 0):
            return self._col_view().mean(-1)
        keep = getattr(self, "_col_keep", None)
        count = float(self.Y.shape[0]) if keep is None else keep.sum().to(self.Y.dtype)
        return self.sum(-1) / count

    def _col_view(self) -> "LazyScores":
        """The transposed matrix with the row mask turned into its column mask."""
        t = self.T
        t._col_keep, t._row_keep = getattr(self, "_row_keep", None), getattr(self, "_col_keep", None)
        return t

    __matmul__ = matmul

    def logsumexp(self, dim: int = -1, exclude_self: bool = False) -> torch.Tensor:
        """lse_i = log sum_j exp S_ij over each row ("Task Map", InfoNCE)."""
        if dim in (-2, 0):
            return self._col_view().logsumexp(-1, exclude_self)
        if dim not in (-1, 1):
            raise ValueError("logsumexp: dim must be -1 or -2")
        e = self._masked("lse")
        return _LseFn.apply(e.X, e.Y, *e._params(), e._meta, bool(exclude_self))

    def softmax_matmul(self, V: torch.Tensor, mask=None) -> torch.Tensor:
        """out_i = sum_j softmax_j(S_ij) V_j ("Task Map", attention), over the pairs a pair mask keeps."""
        if mask is not None:
            return self.mask_pairs(mask).softmax_matmul(V)
        e = self._masked("lse")
        return _SoftmaxFn.apply(e.X, e.Y, V, *e._params(), e._meta)

    def displacement(self) -> torch.Tensor:
        """disp_i = sum_j S_ij (y_j - x_i) ("Stein Variational Gradient Descent")."""
        e = self._masked("sum")
        return _DispFn.apply(e.X, e.Y, *e._params(), e._meta)

    def topk(self, k: int, dim: int = -1, largest: bool = True) -> TopK:
        """k best entries per row, sorted, ties by lower column index ("Task Map", k-NN)."""
        if dim in (-2, 0):
            v, i = self._col_view().topk(k, -1, largest)
            return TopK(v.t(), i.t())
        if dim not in (-1, 1):
            raise ValueError("topk: dim must be -1 or -2")
        e = self._masked("topk_max" if largest else "topk_min")
        v, i = _TopkFn.apply(e.X, e.Y, *e._params(), e._meta, int(k), bool(largest))
        return TopK(v, i)

    def min(self, dim: int = -1) -> TopK:
        """Smallest entry per row (dim=-1) or per column (dim=-2), with its index ("Task Map",
        Chamfer-style losses: D.min(-1) and D.min(-2))."""
        v, i = self.topk(1, dim=dim, largest=False)
        return TopK(v.reshape(-1), i.reshape(-1))

    def max(self, dim: int = -1) -> TopK:
        v, i = self.topk(1, dim=dim, largest=True)
        return TopK(v.reshape(-1), i.reshape(-1))

    def argmin(self, dim: int = -1) -> torch.Tensor:
        return self.min(dim).indices

    def argmax(self, dim: int = -1) -> torch.Tensor:
        return self.max(dim).indices


def lazy(X: torch.Tensor, Y: Optional[torch.Tensor] = None, metric: str = "linear", gamma: float = 1.0) -> LazyScores:
    """Bind a lazy [N,M] score matrix (torchpairwise guide, introduction)."""
    return LazyScores(X, Y, metric=metric, gamma=gamma)


def svgd_direction(x: torch.Tensor, score: torch.Tensor, *, gamma: float) -> torch.Tensor:
    """(K @ score - 2 gamma K.displacement()) / n for the rbf kernel, one fused sweep
    ("Stein Variational Gradient Descent"). Forward only."""
    return ops.svgd_direction(x, score, gamma)


# ------------------------------------------------------------------------------------------------
# autograd functions (argument marshalling only; both directions run in libtp)
# ------------------------------------------------------------------------------------------------


def _want(ctx, first_param: int, has_v: bool):
    n = ctx.needs_input_grad
    wx, wy = n[0], n[1]
    wv = n[2] if has_v else False
    p = first_param
    return (wx, wy, wv, n[p], n[p + 1], n[p + 2], n[p + 3])


def _ret_xy(ctx, g):
    if ctx.same:
        return g["dX"], None
    return g["dX"], g["dY"]


def _ret_params(g):
    return g["d_row_bias"], g["d_col_bias"], g["d_row_weight"], g["d_col_weight"]


class _MatmulFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, Y, V, rb, cb, rw, cw, meta):
        out = ops.pairwise_matmul(X, Y, V, meta.score(rb, cb, rw, cw))
        ctx.save_for_backward(X, Y, V, rb, cb, rw, cw)
        ctx.meta, ctx.same = meta, X is Y
        return out

    @staticmethod
    def backward(ctx, go):
        X, Y, V, rb, cb, rw, cw = ctx.saved_tensors
        g = ops.pairwise_matmul_backward(X, Y, V, ctx.meta.score(rb, cb, rw, cw), go, _want(ctx, 3, True), ctx.same)
        return (*_ret_xy(ctx, g), g["dV"], *_ret_params(g), None)


class _LseFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, Y, rb, cb, rw, cw, meta, exclude_self):
        lse = ops.pairwise_logsumexp(X, Y, meta.score(rb, cb, rw, cw), exclude_self)
        ctx.save_for_backward(X, Y, rb, cb, rw, cw, lse)
        ctx.meta, ctx.same, ctx.excl = meta, X is Y, exclude_self
        return lse

    @staticmethod
    def backward(ctx, gl):
        X, Y, rb, cb, rw, cw, lse = ctx.saved_tensors
        g = ops.pairwise_logsumexp_backward(X, Y, ctx.meta.score(rb, cb, rw, cw), lse, gl, ctx.excl,
                                            _want(ctx, 2, False), ctx.same)
        return (*_ret_xy(ctx, g), *_ret_params(g), None, None)


class _SoftmaxFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, Y, V, rb, cb, rw, cw, meta):
        out, lse = ops.pairwise_softmax_matmul(X, Y, V, meta.score(rb, cb, rw, cw))
        ctx.save_for_backward(X, Y, V, rb, cb, rw, cw, out, lse)
        ctx.meta, ctx.same = meta, X is Y
        return out

    @staticmethod
    def backward(ctx, go):
        X, Y, V, rb, cb, rw, cw, out, lse = ctx.saved_tensors
        g = ops.pairwise_softmax_matmul_backward(X, Y, V, ctx.meta.score(rb, cb, rw, cw), out, lse, go,
                                                 _want(ctx, 3, True), ctx.same)
        return (*_ret_xy(ctx, g), g["dV"], *_ret_params(g), None)


class _DispFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, Y, rb, cb, rw, cw, meta):
        out = ops.pairwise_displacement(X, Y, meta.score(rb, cb, rw, cw))
        ctx.save_for_backward(X, Y, rb, cb, rw, cw)
        ctx.meta, ctx.same = meta, X is Y
        return out

    @staticmethod
    def backward(ctx, go):
        X, Y, rb, cb, rw, cw = ctx.saved_tensors
        g = ops.pairwise_displacement_backward(X, Y, ctx.meta.score(rb, cb, rw, cw), go, _want(ctx, 2, False),
                                               ctx.same)
        return (*_ret_xy(ctx, g), *_ret_params(g), None)


class _TopkFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, Y, rb, cb, rw, cw, meta, k, largest):
        vals, idx = ops.pairwise_topk(X, Y, meta.score(rb, cb, rw, cw), k, largest)
        ctx.mark_non_differentiable(idx)
        ctx.save_for_backward(X, Y, rb, cb, rw, cw, idx)
        ctx.meta, ctx.same, ctx.k = meta, X is Y, k
        return vals, idx

    @staticmethod
    def backward(ctx, gv, _gi):
        X, Y, rb, cb, rw, cw, idx = ctx.saved_tensors
        g = ops.pairwise_topk_backward(X, Y, ctx.meta.score(rb, cb, rw, cw), ctx.k, idx, gv, _want(ctx, 2, False),
                                       ctx.same)
        return (*_ret_xy(ctx, g), *_ret_params(g), None, None, None)
