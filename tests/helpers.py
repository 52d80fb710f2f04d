"""Test-side glue between the CUDA path (torch tensors) and the oracle (numpy).

Only data movement and layout bookkeeping live here; the method's arithmetic is
in oracle/ (expected values) and in the CUDA kernels (values under test).
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_input(t: torch.Tensor) -> np.ndarray:
    """The exact bytes the GPU quantizer reads, as the oracle's input array."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


def mma_layout_from_canonical(scales: np.ndarray, rows: int, cols: int, tile2d: bool = False) -> np.ndarray:
    """Expected tensor-core scale buffer (include/nvfp4.h layout) from canonical scales.

    tile2d: `scales` is the [rows/16, cols/16] tile grid, expanded to every row.
    """
    nrb = (rows + 127) // 128
    nkb = (cols + 255) // 256
    out = np.zeros(nrb * nkb * 2048, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    s = np.arange(cols // 16)[None, :]
    off = (((r >> 7) * nkb + (s >> 4)) << 11) + (((s >> 2) & 3) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (s & 3)
    vals = np.repeat(scales, 16, axis=0)[:rows] if tile2d else scales
    out[off.reshape(-1)] = vals.reshape(-1)
    return out


def qtensor_to_oracle(q, block: int) -> dict:
    """A GPU-produced quantized operand as the oracle's dict (canonical scales)."""
    return dict(codes=q.codes.cpu().numpy(), scales=q.scales.cpu().numpy(), s_dec=float(q.s_dec[0].item()),
                rows=q.rows, cols=q.cols, block=block)


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    d = np.linalg.norm((got.astype(np.float64) - ref.astype(np.float64)).ravel())
    n = np.linalg.norm(ref.astype(np.float64).ravel())
    return float(d / n) if n > 0 else float(d)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (RNE) and back, through torch's fp32 -> bf16 cast.

    fp64 -> fp32 first can double-round; the bf16 comparisons use a Frobenius
    bound far above that effect."""
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def mx_mma_layout_from_canonical(scales: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Expected MXFP4 tensor-core scale buffer (1 KB tiles, include/nvfp4.h) from [rows, cols/32] scales."""
    nrb = (rows + 127) // 128
    nkb = (cols + 255) // 256
    out = np.zeros(nrb * nkb * 1024, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    s = np.arange(cols // 32)[None, :]
    off = (((r >> 7) * nkb + (s >> 3)) << 10) + (((s >> 2) & 1) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (s & 3)
    out[off.reshape(-1)] = scales.reshape(-1)
    return out
