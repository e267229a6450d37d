"""Dense block-scaled FP4 linear layer (FP64 oracle; test infrastructure only).

"Serve Kimi-K2.5-MXFP4 on MI355X with ATOM", section "Stage C: MXFP4 Linear
GEMM": the f4gemm kernels take bf16 activations, quantise them per 1x32 on
the fly and multiply block-scaled FP4 operands with the scaled matrix
instruction (scales applied inside the product), writing bf16:

    a = dequant(quantize(x))        MXFP4 per 32 (NVFP4: per 16, one tensor
                                    scale over x), the quantisers of quant.py
    y = a . W^T,  W = dequant(codes, scales[, g_w])

The products are exact in float64 (MXFP4: multiples of 2**-2 of bounded
exponent range; NVFP4: exact block products rounded once per sum).  The GPU
stores y as bf16; its tolerance is |gpu - y| <= 2**-8 |y| + 1e-3 S with
S = sum_k |a_k W_k| (the form the layer's tolerance takes for one
contraction).
"""
from __future__ import annotations

import numpy as np

from . import quant as Q


def linear_forward(x_f64: np.ndarray, w_codes: np.ndarray, w_scales: np.ndarray, fmt: str, g_w=None):
    """x [T, K] exact bf16 values; w_codes [N, K] unpacked FP4 codes, w_scales
    the matching block scale bytes.  Returns y [T, N], S [T, N] and the
    quantised activations (codes, scales, g_x)."""
    xc, xs, gx = Q.quantize(x_f64, fmt)
    a = Q.dequant(xc, xs, fmt, gx)
    W = Q.dequant(w_codes, w_scales, fmt, g_w)
    return a @ W.T, np.abs(a) @ np.abs(W).T, (xc, xs, gx)


def tolerance(y: np.ndarray, S: np.ndarray) -> np.ndarray:
    return 2.0 ** -8 * np.abs(y) + 1e-3 * S
