"""Exact MXFP4 -> FP8 E4M3 per-channel conversion (FP64 oracle; test only).

"Kimi-K2.7-Code on Gaudi 2", section "Exact MXFP4 to FP8 per-channel
conversion": an MXFP4 element is an E2M1 value times the power-of-two E8M0
scale of its 32-block.  For each output row one power-of-two channel scale 2**k
is chosen, k = (exponent of the row's largest element) - 7, so that every
element becomes an E4M3 normal with exponent in [-5, 7] and magnitude at most
192; this holds whenever the row's E8M0 scales span at most 9 binades.  The
-5 floor keeps a copy halved at load time normal.

Steps per row, in that order:

    v_i   = E2M1(c_i) * 2**(s_b - 127)
    e_max = floor(log2(max |v_i|))
    k     = e_max - 7
    byte  = RNE_E4M3(v_i / 2**k)         (exact for in-contract rows)
    scale = 2**k as fp32                 (may be an fp32 subnormal; exact)

Readings where the page is silent:
  * all-zero row: k = 0, scale 1.0, bytes keep the zero's sign (0x00 / 0x80);
  * a scale byte 255 (NaN) in the row: status NAN_SCALE, bytes 0, scale NaN;
  * an element whose shifted exponent falls below -5: status BELOW_FLOOR; its
    byte is still the round-to-nearest-even E4M3 value (possibly subnormal
    or zero), so the row is flagged rather than silently inexact.
"""
from __future__ import annotations

import numpy as np

from .formats import E2M1_TABLE, e4m3_encode, floor_log2, unpack_nibbles

ST_OK = 0
ST_BELOW_FLOOR = 1
ST_NAN_SCALE = 2

SHIFT = 7     # k = e_max - SHIFT puts the row's largest element at exponent 7
FLOOR = -5    # lowest element exponent the conversion promises
E8M0_BIAS = 127


def mxfp4_to_fp8_rowscale(codes: np.ndarray, scales: np.ndarray):
    """codes uint8 [R, K/2] (packed), scales uint8 [R, K/32].  Returns
    (fp8 bytes uint8 [R, K], row_scale float32 [R], status uint8 [R])."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    R = codes.shape[0]
    K = 2 * codes.shape[1]
    c = unpack_nibbles(codes).reshape(R, K // 32, 32)
    s = scales.astype(np.int64)
    nan_row = np.any(s == 255, axis=1)
    v = np.ldexp(E2M1_TABLE[c], (np.where(s == 255, E8M0_BIAS, s) - E8M0_BIAS)[..., None]).reshape(R, K)
    mag = np.abs(v)
    nz = mag > 0
    rowmax = np.max(mag, axis=1)
    has = rowmax > 0
    e_max = np.where(has, floor_log2(np.where(has, rowmax, 1.0)), SHIFT)
    k = np.where(has, e_max - SHIFT, 0)
    w = np.ldexp(v, -k[:, None])
    out = e4m3_encode(w)
    ex = np.where(nz, floor_log2(np.where(nz, w, 1.0)), 0)
    below = np.any(nz & (ex < FLOOR), axis=1)
    status = np.where(below, ST_BELOW_FLOOR, ST_OK).astype(np.uint8)
    row_scale = np.ldexp(np.ones(R), k).astype(np.float32)
    out[nan_row] = 0
    row_scale[nan_row] = np.float32(np.nan)
    status[nan_row] = ST_NAN_SCALE
    return out, row_scale, status


def scale_span(scales: np.ndarray) -> np.ndarray:
    """Binades spanned by each row's E8M0 scales (max - min byte)."""
    s = np.asarray(scales, dtype=np.int64)
    return s.max(axis=1) - s.min(axis=1)
