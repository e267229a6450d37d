"""Element and scale formats of block-scaled FP4.

* E2M1: the 4-bit element of MXFP4 and NVFP4 ("Serve Kimi-K2.5-MXFP4 on MI355X
  with ATOM", section "The Kimi-K2.5-MXFP4 Model on gfx950": FP4 E2M1 payload,
  packed two per byte).  Bit 3 is the sign, bits 2..1 the exponent (bias 1),
  bit 0 the mantissa; exponent field 0 is subnormal (0.5 * m).  No Inf/NaN.
* E8M0: the MXFP4 block scale (same section): byte b encodes 2**(b - 127);
  255 is NaN.
* E4M3 (OCP "FN"): the NVFP4 block scale ("Serving NVFP4 models on AMD Instinct
  MI355 accelerators") and the output of the FP8 conversion ("Kimi-K2.7-Code on
  Gaudi 2", section "Exact MXFP4 to FP8 per-channel conversion").  Bias 7,
  three mantissa bits, subnormals m * 2**-9, only S.1111.111 is NaN, max 448.

Encoders round to nearest with ties to the even code and saturate at the
largest finite magnitude.  Encoders take exact float64 values.
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Exact value of a 4-bit E2M1 code (negative zero for code 8)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e8m0_value(b: int) -> float:
    return float("nan") if b == 255 else 2.0 ** (b - 127)


def e4m3_value(b: int) -> float:
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(b) for b in range(256)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)

# Non-negative finite grids, indexed by code: value is increasing in the code,
# and the code's least significant bit is the mantissa's.
_E2M1_POS = E2M1_TABLE[:8]
_E4M3_POS = E4M3_TABLE[:127]


def _rne_grid(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid point nearest to each non-negative magnitude; a tie
    goes to the even index; magnitudes beyond the last point saturate.

    With mids[i] the midpoint of grid[i] and grid[i+1], the nearest point of
    a magnitude is the number of midpoints strictly below it; a magnitude on
    a midpoint lies between an odd and an even index and takes the even one."""
    mag = np.asarray(mag, dtype=np.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    if len(mids) <= 16:  # short grid: count the midpoints one by one
        idx = np.zeros(mag.shape, dtype=np.int64)
        on_mid = np.zeros(mag.shape, dtype=bool)
        for m in mids:
            idx += mag > m
            on_mid |= mag == m
    else:
        idx = np.searchsorted(mids, mag, side="left")
        on_mid = np.take(mids, np.minimum(idx, len(mids) - 1)) == mag
    idx += on_mid & ((idx & 1) == 1)
    return idx


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even E2M1 code of each value, saturating to +-6.  The
    code carries the sign bit of the input, zero included."""
    v = np.asarray(v, dtype=np.float64)
    code = _rne_grid(np.abs(v), _E2M1_POS)
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even E4M3 byte of each value, saturating to +-448."""
    v = np.asarray(v, dtype=np.float64)
    code = _rne_grid(np.abs(v), _E4M3_POS)
    return (code | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes along the last axis: element 2j in the low nibble of
    byte j, element 2j+1 in the high nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def floor_log2(v: np.ndarray) -> np.ndarray:
    """Exact floor(log2(|v|)) for finite non-zero float64 values."""
    _, ex = np.frexp(np.abs(np.asarray(v, dtype=np.float64)))
    return ex.astype(np.int64) - 1
