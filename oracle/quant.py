"""MXFP4 and NVFP4 quantisation (FP64 oracle; test infrastructure only).

MXFP4 ("Serve Kimi-K2.5-MXFP4 on MI355X with ATOM", sections "The
Kimi-K2.5-MXFP4 Model on gfx950" and "Stage B: Dynamic Activation
Quantization"): each block of 32 consecutive K values shares one E8M0 scale;
elements are E2M1.  The pages fix neither the scale rule nor the rounding;
the reading used here is the OCP MX rule

    e = floor(log2(amax)) - 2   (clamped to [-127, 127]; amax = 0 -> e = -127)
    scale byte = e + 127,  code_i = RNE_E2M1(v_i / 2**e)  saturating at 6,

where the code keeps the sign bit of v_i (so -0.1 becomes -0).

NVFP4 ("Serving NVFP4 models on AMD Instinct MI355 accelerators", section
"Weight Dequantization and Activation QDQ"): E2M1 elements, one E4M3 scale per
16 values and one FP32 scale per tensor.  The reading used here, every step a
correctly rounded FP32 operation in this order:

    g    = fp32(amax_tensor / 2688)                   (2688 = 6 * 448)
    s_b  = RNE_E4M3(fp32(amax_block / fp32(6 * g)))   saturating at 448
    d_b  = fp32(value(s_b) * g)
    code = RNE_E2M1(fp32(v / d_b))                     (d_b = 0 -> signed zero)

and the dequantised value is E2M1(code) * value(s_b) * g, exactly.
"""
from __future__ import annotations

import numpy as np

from .formats import (E2M1_TABLE, E4M3_TABLE, e2m1_encode, e4m3_encode,
                      floor_log2)

MX_BLOCK = 32
NV_BLOCK = 16


def mx_quantize(v: np.ndarray):
    """MXFP4 quantisation along the last axis.

    Returns (codes uint8 [..., K] unpacked 4-bit codes, scale bytes uint8
    [..., K/32]).  ``v`` holds exact float64 values (bf16 or fp32 inputs)."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % MX_BLOCK == 0
    blk = v.reshape(v.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.max(np.abs(blk), axis=-1)
    e = np.where(amax > 0, floor_log2(np.where(amax > 0, amax, 1.0)) - 2, -127)
    e = np.clip(e, -127, 127)
    scaled = np.ldexp(blk, -e[..., None])
    codes = e2m1_encode(scaled).reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def mx_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact values of unpacked MXFP4 codes [..., K] with E8M0 bytes [..., K/32]."""
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1]
    vals = E2M1_TABLE[codes].reshape(codes.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    s = np.asarray(scales, dtype=np.int64)
    out = np.ldexp(vals, (s - 127)[..., None])
    out = np.where((s == 255)[..., None], np.nan, out)
    return out.reshape(codes.shape)


def nv_global_scale(amax: float) -> np.float32:
    """Per-tensor FP32 scale g = fp32(amax / (6 * 448))."""
    return np.float32(amax) / np.float32(2688.0)


def nv_quantize(v: np.ndarray, g: np.float32 | None = None):
    """NVFP4 quantisation along the last axis with one tensor scale over all of ``v``.

    Returns (codes uint8 [..., K] unpacked, scale bytes uint8 [..., K/16],
    g float32).  ``v`` must hold values exactly representable in fp32."""
    v = np.asarray(v, dtype=np.float64)
    v32 = v.astype(np.float32)
    assert np.array_equal(v32.astype(np.float64), v, equal_nan=True), "inputs must be fp32 values"
    K = v.shape[-1]
    assert K % NV_BLOCK == 0
    if g is None:
        g = nv_global_scale(np.max(np.abs(v32)) if v32.size else np.float32(0))
    g = np.float32(g)
    blk = v32.reshape(v.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    amax_b = np.max(np.abs(blk), axis=-1)
    six_g = np.float32(6.0) * g
    with np.errstate(divide="ignore", invalid="ignore"):
        q_s = np.where(six_g > 0, amax_b / six_g, np.float32(0.0)).astype(np.float32)
    s_byte = e4m3_encode(q_s.astype(np.float64)) & np.uint8(0x7F)
    d_b = (E4M3_TABLE[s_byte].astype(np.float32) * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(d_b[..., None] > 0, blk / d_b[..., None], np.float32(0.0) * blk)
    scaled = scaled.astype(np.float32).astype(np.float64)
    # keep the sign of zero inputs (np.where above already gives +-0 for d_b == 0)
    codes = e2m1_encode(scaled).reshape(v.shape)
    return codes, s_byte.astype(np.uint8), g


def nv_dequant(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """Exact values of unpacked NVFP4 codes [..., K] with E4M3 bytes [..., K/16]
    and tensor scale g."""
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1]
    vals = E2M1_TABLE[codes].reshape(codes.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    s = E4M3_TABLE[np.asarray(scales, dtype=np.uint8)]
    return (vals * s[..., None] * float(g)).reshape(codes.shape)


def quantize(v: np.ndarray, fmt: str, g=None):
    """Dispatch on format: returns (codes, scales, g or None)."""
    if fmt == "mxfp4":
        c, s = mx_quantize(v)
        return c, s, None
    return nv_quantize(v, g)


def dequant(codes, scales, fmt: str, g=None) -> np.ndarray:
    if fmt == "mxfp4":
        return mx_dequant(codes, scales)
    return nv_dequant(codes, scales, g)
