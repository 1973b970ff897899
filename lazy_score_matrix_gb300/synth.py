"""Seeded synthetic inputs for the five benchmark workloads (and smaller versions of them).

Shared by the tests (both sides of every comparison get the same bits) and the bench. Holds no part of the
method's arithmetic: only random draws, the unit-normalisation the InfoNCE workload prescribes for
its inputs, and constant upstream gradients. Every tensor is drawn on the CPU from
``torch.Generator().manual_seed(1000 * workload + tensor_index)`` in the workload's dtype.

Workloads (shapes and distributions of the torchpairwise guide's "Task Map" and "Stein Variational
Gradient Descent" rows):
  1 rbf kernel product, fp32: X, Y [1024,3] ~ N(0,1), gamma 0.5, V = [N(0,1) [1024,3] | ones], dout = ones.
  2 InfoNCE row logsumexp, fp32: z [8192,64] ~ N(0,1), rows L2-normalised, scale 1/0.07, exclude_self,
    loss = -mean(lse) so grad_lse = -1/N.
  3 exact k-NN, fp32: X [65536,16], R [1048576,16], integers uniform in [-8, 8], sqeuclidean, k = 16.
  4 attention softmax_matmul, fp32: Q, K, V [16384,64] ~ N(0,1), scale 64^-0.5, dO = ones.
  5 SVGD direction, fp64: x [131072,8] ~ N(0,1), score = -x, rbf gamma 0.1.
"""
from __future__ import annotations

import torch

FULL = {
    1: dict(N=1024, M=1024, D=3, C=4),
    2: dict(N=8192, M=8192, D=64),
    3: dict(N=65536, M=1048576, D=16, k=16),
    4: dict(N=16384, M=16384, D=64, C=64),
    5: dict(N=131072, M=131072, D=8),
}

NAMES = {
    1: "rbf_kernel_matmul_f32_X1024x3_Y1024x3_V1024x4",
    2: "infonce_logsumexp_f32_z8192x64",
    3: "knn_topk16_f32_X65536x16_R1048576x16",
    4: "attention_softmax_matmul_f32_QKV16384x64",
    5: "svgd_direction_f64_x131072x8",
}


def _gen(cfg: int, idx: int) -> torch.Generator:
    return torch.Generator().manual_seed(1000 * cfg + idx)


def normal(cfg, idx, shape, dtype=torch.float32):
    return torch.randn(*shape, generator=_gen(cfg, idx), dtype=dtype)


def integers(cfg, idx, shape, lo, hi, dtype=torch.float32):
    """Uniform integers in [lo, hi] inclusive, stored in `dtype`."""
    return torch.randint(lo, hi + 1, shape, generator=_gen(cfg, idx)).to(dtype)


def workload(cfg: int, **over) -> dict:
    """CPU tensors and scalars of workload `cfg`; keyword overrides shrink the sizes."""
    s = dict(FULL[cfg])
    s.update(over)
    if cfg == 1:
        N, M, D, C = s["N"], s["M"], s["D"], s["C"]
        V = torch.cat([normal(1, 2, (M, C - 1)), torch.ones(M, 1)], 1)
        return dict(X=normal(1, 0, (N, D)), Y=normal(1, 1, (M, D)), V=V, gamma=0.5, metric="rbf",
                    grad_out=torch.ones(N, C))
    if cfg == 2:
        N, D = s["N"], s["D"]
        z = normal(2, 0, (N, D))
        z = z / z.norm(dim=1, keepdim=True)
        return dict(z=z, scale=1.0 / 0.07, metric="linear", exclude_self=True, grad_lse=torch.full((N,), -1.0 / N))
    if cfg == 3:
        N, M, D = s["N"], s["M"], s["D"]
        return dict(X=integers(3, 0, (N, D), -8, 8), R=integers(3, 1, (M, D), -8, 8), k=s.get("k", 16),
                    metric="sqeuclidean")
    if cfg == 4:
        N, M, D, C = s["N"], s["M"], s["D"], s["C"]
        return dict(Q=normal(4, 0, (N, D)), K=normal(4, 1, (M, D)), V=normal(4, 2, (M, C)), scale=D ** -0.5,
                    metric="linear", grad_out=torch.ones(N, C))
    if cfg == 5:
        N, D = s["N"], s["D"]
        x = normal(5, 0, (N, D), torch.float64)
        return dict(x=x, score=-x, gamma=0.1)
    raise ValueError(cfg)
