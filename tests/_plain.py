"""Plain dense evaluation of each consumer in the working precision (PyTorch on the CPU): what that
precision achieves on the exact inputs.

Parity tests hold the GPU to max(tolerance, ACHIEVABLE_SLACK x the error of this evaluation against the
oracle), measured with the same floor (1e-3 of the largest magnitude). Where the consumer is well
conditioned the tolerance decides; where its outputs cancel far below their terms (weighted sums of
many random-sign rows, exp of exp, a softmax row carrying all its mass on one pair) any evaluation in
fp32 misses the tolerance, and this evaluation measures by how much, on the test's own inputs.

The score matrix is built densely ([N, M] in memory: test sizes only) from its definition (torchpairwise
guide "Using Torchpairwise in Models", Score Expressions, in the canonical order scale * w_row * w_col *
base + b_row + b_col, then exp), distances by the direct difference; the reductions are PyTorch's
logsumexp, softmax and matrix products; gradients are PyTorch autograd of that expression. Nothing here
is shared with the oracle or with libtp.
"""
from __future__ import annotations

import torch

from tests._util import FLOOR, rel_err

# An evaluation in a different summation order (the GPU's tiles and two-level sums, the hardware exp2)
# has rounding errors of the same size as this one, not the same errors: their largest elementwise
# values can differ by a small factor. Twice the measured error.
ACHIEVABLE_SLACK = 2.0
# The tensor-core kernels split each fp32 operand into fp16 hi + lo: 22 significant bits instead of
# fp32's 24, and the products' low parts (lo x lo) are dropped. Two bits of operand precision are a
# factor 4 in the rounding error of every product, so their bound is four times the plain fp32 error.
TC_SLACK = 4.0


def _t(a, dtype):
    if a is None:
        return None
    if not isinstance(a, torch.Tensor):
        a = torch.as_tensor(a)
    return a.detach().cpu().to(dtype).clone()


def _keep(N, M, pair_mask="all", band=0, row_group=None, col_group=None, exclude_self=False):
    i = torch.arange(N)[:, None]
    j = torch.arange(M)[None, :]
    keep = torch.ones(N, M, dtype=torch.bool)
    if pair_mask == "causal":
        keep &= j <= i
    elif pair_mask == "band":
        keep &= (i - j).abs() <= band
    elif pair_mask == "same_group":
        rg, cg = torch.as_tensor(row_group).cpu().long(), torch.as_tensor(col_group).cpu().long()
        keep &= rg[:, None] == cg[None, :]
    if exclude_self:
        keep &= i != j
    return keep


class Plain:
    """Dense scores S [N, M] in `dtype` with autograd on X, Y, V and the row/column parameters."""

    def __init__(self, X, Y, dtype=torch.float32, metric="linear", gamma=1.0, scale=1.0, apply_exp=False,
                 row_bias=None, col_bias=None, row_weight=None, col_weight=None, pair_mask="all", band=0,
                 row_group=None, col_group=None, V=None, same=False):
        self.dtype = dtype
        self.X = _t(X, dtype).requires_grad_(True)
        self.Y = self.X if same else _t(Y, dtype).requires_grad_(True)
        self.same = same
        self.V = None if V is None else _t(V, dtype).requires_grad_(True)
        self.p = {k: (None if v is None else _t(v, dtype).requires_grad_(True))
                  for k, v in (("d_row_bias", row_bias), ("d_col_bias", col_bias),
                               ("d_row_weight", row_weight), ("d_col_weight", col_weight))}
        self.metric, self.gamma, self.scale, self.apply_exp = metric, gamma, scale, apply_exp
        self.mask = dict(pair_mask=pair_mask, band=band, row_group=row_group, col_group=col_group)

    def scores(self):
        X, Y = self.X, self.Y
        if self.metric == "linear":
            base = X @ Y.T
        else:
            d2 = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
            base = d2 if self.metric == "sqeuclidean" else torch.exp(-self.gamma * d2)
        t = self.scale * base
        if self.p["d_row_weight"] is not None:
            t = t * self.p["d_row_weight"][:, None]
        if self.p["d_col_weight"] is not None:
            t = t * self.p["d_col_weight"][None, :]
        if self.p["d_row_bias"] is not None:
            t = t + self.p["d_row_bias"][:, None]
        if self.p["d_col_bias"] is not None:
            t = t + self.p["d_col_bias"][None, :]
        return torch.exp(t) if self.apply_exp else t

    def keep(self, exclude_self=False):
        return _keep(self.X.shape[0], self.Y.shape[0], exclude_self=exclude_self, **self.mask)

    # ---- forwards
    def matmul(self):
        S = self.scores()
        return torch.where(self.keep(), S, torch.zeros((), dtype=self.dtype)) @ self.V

    def logsumexp(self, exclude_self=False):
        S = self.scores()
        return torch.logsumexp(torch.where(self.keep(exclude_self), S, torch.tensor(float("-inf"), dtype=self.dtype)),
                               dim=1)

    def softmax_matmul(self):
        S = torch.where(self.keep(), self.scores(), torch.tensor(float("-inf"), dtype=self.dtype))
        lse = torch.logsumexp(S, dim=1)
        P = torch.exp(S - torch.where(torch.isfinite(lse), lse, torch.zeros((), dtype=self.dtype))[:, None])
        return P @ self.V, lse

    def displacement(self):
        S = torch.where(self.keep(), self.scores(), torch.zeros((), dtype=self.dtype))
        return S @ self.Y - S.sum(1, keepdim=True) * self.X

    # ---- gradients of sum(G * out): autograd of the dense expression
    def grads(self, out, G):
        G = _t(G, self.dtype)
        ins = {"dX": self.X}
        if not self.same:
            ins["dY"] = self.Y
        if self.V is not None:
            ins["dV"] = self.V
        ins.update({k: v for k, v in self.p.items() if v is not None})
        keys = list(ins)
        gs = torch.autograd.grad((out * G).sum(), [ins[k] for k in keys], allow_unused=True)
        res = {k: (torch.zeros_like(ins[k]) if g is None else g) for k, g in zip(keys, gs)}
        if self.same:
            res["dY"] = None  # summed into dX
        return res


@torch.no_grad()
def attention_rows(Q, K, V, scale, dtype=torch.float32, chunk=1024):
    """out = softmax(scale Q K^T) V and its row log-sum-exp, densely in `dtype`, a chunk of rows at a time
    (the same arithmetic per row as Plain.softmax_matmul, without the [N, M] matrix in memory at once)."""
    Q, K, V = _t(Q, dtype), _t(K, dtype), _t(V, dtype)
    outs, lses = [], []
    for r in range(0, Q.shape[0], chunk):
        S = scale * (Q[r:r + chunk] @ K.T)
        lse = torch.logsumexp(S, dim=1)
        outs.append(torch.exp(S - lse[:, None]) @ V)
        lses.append(lse)
    return torch.cat(outs), torch.cat(lses)


def svgd_direction(x, score, gamma, dtype=torch.float32):
    """phi = (K @ score - 2 gamma K.displacement()) / n with K = exp(-gamma |x_i - x_j|^2) (the guide's
    Stein Variational Gradient Descent section), densely in `dtype`."""
    x, s = _t(x, dtype), _t(score, dtype)
    K = torch.exp(-gamma * ((x[:, None, :] - x[None, :, :]) ** 2).sum(-1))
    disp = K @ x - K.sum(1, keepdim=True) * x
    return (K @ s - 2 * gamma * disp) / x.shape[0]


def achievable(plain_out, want, tol, floor_frac=FLOOR, abs_floor=0.0, slack=ACHIEVABLE_SLACK):
    """The bound a GPU result is held to: the tolerance, or `slack` x what the plain evaluation in the
    working precision reaches against the oracle, whichever is larger (same error measure)."""
    return max(tol, slack * rel_err(plain_out, want, floor_frac, abs_floor))
