"""Pair masks for lazy scores: torchpairwise guide "Using Torchpairwise in Models", Task Map (attention:
``softmax_matmul(V, mask=...)`` with ``tp.masks.causal()``, band, same_group) and Score Expressions.

A masked pair leaves the consumer's reduction: no term in K @ V, a log-sum-exp, a softmax or a
displacement, never selected by top-k (rows with fewer than k kept pairs pad with value +-inf and
index -1), no gradient; a softmax row with no kept pair returns 0. The masks run inside libtp's
streamed sweeps; attention (fp32, D = C = 64) under a causal or band mask runs on its tensor-core kernels,
which skip the tiles a mask removes whole (the guide runs pair masks on materialised tiles).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class PairMask:
    """kind: "causal" (keep j <= i), "band" (keep |i - j| <= width), "same_group" (keep
    row_group[i] == col_group[j])."""
    kind: str
    width: int = 0
    row_group: Optional[torch.Tensor] = None
    col_group: Optional[torch.Tensor] = None

    def transposed(self) -> "PairMask":
        """The mask of the transposed matrix (pair (j, i) of S^T is pair (i, j) of S)."""
        if self.kind == "causal":
            raise NotImplementedError("a causal mask transposes into j >= i, which libtp's masks do not hold")
        if self.kind == "same_group":
            return PairMask("same_group", 0, self.col_group, self.row_group)
        return self


def causal() -> PairMask:
    """Keep the pairs j <= i (row i sees columns up to its own index)."""
    return PairMask("causal")


def band(width: int) -> PairMask:
    """Keep the pairs with |i - j| <= width."""
    if int(width) < 0:
        raise ValueError("band width must be >= 0")
    return PairMask("band", int(width))


def same_group(row_group: torch.Tensor, col_group: Optional[torch.Tensor] = None) -> PairMask:
    """Keep the pairs whose row and column carry the same group id (integer tensors [N] and [M]; the
    column ids default to the row ids, for scores of a set with itself)."""
    rg = row_group.to(torch.int32).contiguous()
    cg = rg if col_group is None else col_group.to(torch.int32).contiguous()
    return PairMask("same_group", 0, rg, cg)
