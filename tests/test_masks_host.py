"""Host logic of the pair masks (CPU only): the constructors of tp.masks (torchpairwise guide "Using
Torchpairwise in Models", Task Map and Score Expressions: causal, band, same_group), how each mask
transposes with the lazy matrix, the expressions that do not fold into one fused score, and the product
path refusing CPU tensors (there is no CPU fallback)."""
import pytest
import torch

import lazy_score_matrix_gb300 as tp


def test_mask_constructors():
    assert tp.masks.causal().kind == "causal"
    b = tp.masks.band(3)
    assert (b.kind, b.width) == ("band", 3)
    with pytest.raises(ValueError):
        tp.masks.band(-1)
    rg = torch.tensor([0, 1, 1, 2], dtype=torch.int64)
    g = tp.masks.same_group(rg)
    assert g.row_group.dtype == torch.int32 and torch.equal(g.col_group, g.row_group)
    cg = torch.tensor([2, 2, 0])
    g2 = tp.masks.same_group(rg, cg)
    assert torch.equal(g2.col_group, cg.to(torch.int32))


def test_masks_transpose_with_the_matrix():
    # pair (j, i) of S^T is pair (i, j) of S: a band is symmetric, the group arrays trade places, and a
    # causal mask would become j >= i, which no mask holds
    X, Y = torch.randn(5, 3), torch.randn(6, 3)
    L = tp.lazy(X, Y, "linear")
    assert L.mask_pairs(tp.masks.band(2)).T._meta.pair == tp.masks.band(2)
    rg, cg = torch.arange(5) % 2, torch.arange(6) % 3
    t = L.mask_pairs(tp.masks.same_group(rg, cg)).T._meta.pair
    assert torch.equal(t.row_group, cg.to(torch.int32)) and torch.equal(t.col_group, rg.to(torch.int32))
    with pytest.raises(NotImplementedError):
        L.mask_pairs(tp.masks.causal()).T
    with pytest.raises(NotImplementedError):  # a reduction over columns goes through the transpose
        L.mask_pairs(tp.masks.causal()).logsumexp(dim=-2)


def test_mask_expressions_that_do_not_fold():
    L = tp.lazy(torch.randn(4, 3), torch.randn(4, 3))
    with pytest.raises(TypeError):
        L.mask_pairs("causal")
    with pytest.raises(NotImplementedError):
        L.mask_pairs(tp.masks.causal()).mask_pairs(tp.masks.band(1))


def test_consumers_refuse_cpu_tensors():
    L = tp.lazy(torch.randn(6, 3), torch.randn(6, 3), "linear")
    with pytest.raises(ValueError, match="CUDA tensors only"):
        L.softmax_matmul(torch.randn(6, 2), mask=tp.masks.causal())
