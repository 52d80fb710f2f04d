"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers: it holds none of the quantization or GEMM
arithmetic.  Tensors are drawn with torch generators on the requested device; a
check that compares the CUDA path with the oracle copies the SAME bytes to the
host, so the device a tensor was drawn on never matters for parity.

Workloads follow the shapes of the dense layers of the 5120-hidden model the
NVFP4 pretraining news page describes (¶1): hidden 5120, FFN 20480.
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, then rounded to ``dtype``."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def student_t(shape, dof: int, seed: int, scale: float = 1.0, dtype=torch.bfloat16,
              device="cpu") -> torch.Tensor:
    """Student-t with integer ``dof``: z / sqrt(chi2_dof / dof), chi2 = sum of dof squared normals."""
    g = _gen(seed, device)
    z = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros_like(z)
    for _ in range(dof):
        n = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(n, n)
    t = z / torch.sqrt(chi2 / dof)
    if scale != 1.0:
        t.mul_(scale)
    return t.to(dtype)


def outlier_columns(x: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Scale round(frac * C) seeded columns of ``x`` by ``factor`` (in place; returns x)."""
    C = x.shape[-1]
    n = int(round(frac * C))
    if n == 0:
        return x
    g = _gen(seed, "cpu")
    cols = torch.randperm(C, generator=g)[:n].to(x.device)
    x[..., cols] = (x[..., cols].float() * factor).to(x.dtype)
    return x


def outlier_rows(x: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Scale round(frac * R) seeded rows of ``x`` by ``factor`` (in place; returns x)."""
    R = x.shape[0]
    n = int(round(frac * R))
    if n == 0:
        return x
    g = _gen(seed, "cpu")
    rows = torch.randperm(R, generator=g)[:n].to(x.device)
    x[rows] = (x[rows].float() * factor).to(x.dtype)
    return x


# ---- the workloads ---------------------------------------------------------------

def linear_layer(M: int, K: int, N: int, seed: int = 0, dtype=torch.bfloat16, device="cpu"):
    """One linear layer: X [M,K] ~ N(0,1), W [N,K] ~ N(0,0.02), dY [M,N] ~ N(0,1e-3).

    Data seeds: X = seed, W = seed + 1, dY = seed + 2.
    """
    X = normal((M, K), 1.0, seed, dtype, device)
    W = normal((N, K), 0.02, seed + 1, dtype, device)
    dY = normal((M, N), 1e-3, seed + 2, dtype, device)
    return X, W, dY


def heavy_tailed_layer(M: int, K: int, N: int, seed: int = 0, device="cpu"):
    """Heavy-tailed stress layer: X Student-t(3) with 1% of channels x50, W ~ N(0,0.02),
    dY = Student-t(4) x 1e-3; all bf16."""
    X = student_t((M, K), 3, seed, device=device)
    outlier_columns(X, 0.01, 50.0, seed + 100)
    W = normal((N, K), 0.02, seed + 1, torch.bfloat16, device)
    dY = student_t((M, N), 4, seed + 2, scale=1e-3, device=device)
    return X, W, dY


def heavy_tailed_token_outliers(M: int, K: int, N: int, seed: int = 0, device="cpu"):
    """The heavy-tailed layer with its outliers along the tokens (the Wgrad contraction axis)
    instead of the channels: X Student-t(3) and dY Student-t(4) x 1e-3 with the same seeded
    1% of tokens (rows of both) x50, W ~ N(0,0.02); all bf16.  An outlier token dominates
    every 16-token block of the column (Wgrad) quantization it falls in."""
    X = student_t((M, K), 3, seed, device=device)
    W = normal((N, K), 0.02, seed + 1, torch.bfloat16, device)
    dY = student_t((M, N), 4, seed + 2, scale=1e-3, device=device)
    outlier_rows(X, 0.01, 50.0, seed + 200)
    outlier_rows(dY, 0.01, 50.0, seed + 200)
    return X, W, dY


def sweep_tensor(R: int, C: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Quantizer sweep input: bf16 [R, C] ~ N(0,1) with 0.1% of columns x100."""
    x = normal((R, C), 1.0, seed, torch.bfloat16, device)
    return outlier_columns(x, 0.001, 100.0, seed + 100)


def sweep_rows(p: int, C: int) -> int:
    """Rows for a sweep tensor of about 2^p elements with C columns (a multiple of 16)."""
    return max(16, int(round((2 ** p) / C / 16)) * 16)
