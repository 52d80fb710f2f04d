"""GB300-native NVFP4 quantized linear layer.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI of
include/nvfp4.h (``libnvfp4_gb300.so``); this package marshals torch tensors
(device memory and the current stream) into those calls.  There is no CPU or
library fallback: every function raises if the CUDA library is missing.

Method: news page "NVIDIA NVFP4 paper: 4-bit pretrain hits FP8 parity (12B,
10T tokens)", ¶2 -- E2M1 in 16-element blocks with E4M3 block scales and an
FP32 tensor scale; 16x16 2D blocks for weights; a 16x16 RHT on the Wgrad
inputs; stochastic rounding on gradients only.
"""
from __future__ import annotations

from .api import (QTensor, quantize, quantize_dual, gemm, linear_fprop, linear_dgrad, linear_wgrad, quantize_weight,
                  status_query, dev_status, reset_status, scales_mma_bytes, NVFP4Error, sqrelu_forward,
                  sqrelu_backward, gemm_sqrelu_backward, gemm_sqrelu_maxima, MXTensor, mx_quantize, mx_gemm, mx_scales_mma_bytes,
                  reset_gemm_workspaces)
from ._lib import F32, BF16, RNE, SR, ROW, COL, TILE16, EXPORTS, LIB_PATH

__all__ = ["QTensor", "quantize", "quantize_dual", "gemm", "linear_fprop", "linear_dgrad", "linear_wgrad", "quantize_weight",
           "status_query", "dev_status", "reset_status", "scales_mma_bytes", "NVFP4Error", "sqrelu_forward",
           "sqrelu_backward", "gemm_sqrelu_backward", "gemm_sqrelu_maxima", "MXTensor", "mx_quantize", "mx_gemm", "mx_scales_mma_bytes",
           "reset_gemm_workspaces",
           "F32", "BF16", "RNE", "SR", "ROW", "COL", "TILE16", "EXPORTS", "LIB_PATH"]
