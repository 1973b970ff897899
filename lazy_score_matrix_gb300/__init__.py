"""lazy_score_matrix_gb300: streamed pairwise score consumers on GB300 (sm_103a).

A pairwise score S[i,j] = f(x_i, y_j) is evaluated tile by tile in libtp's CUDA kernels, consumed in
the same pass and never stored; first derivatives replay the pairs (torchpairwise guide "Using
Torchpairwise in Models"). The C ABI is include/tp.h; this package is its Python binding.
"""
from . import masks
from .lazy import LazyScores, TopK, lazy, svgd_direction
from .losses import mmd_statistics, sinkhorn_divergence
from .ops import Score

__all__ = ["LazyScores", "TopK", "lazy", "svgd_direction", "mmd_statistics", "sinkhorn_divergence", "Score", "masks"]
