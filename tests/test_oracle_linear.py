"""Pins of the dense block-scaled FP4 linear oracle: every output equals the
exact block-scaled sum computed with Python integers and fractions (MXFP4:
E2M1 integers times power-of-two scales; NVFP4: the two-level form
g_a g_w sum_b s_a,b s_w,b sum_k q_a q_w), and a loop-by-loop recomputation."""
from fractions import Fraction
import math

import numpy as np

from oracle import formats as F
from oracle import linear as LIN
from oracle import quant as Q


def _inputs(T, K, N, fmt, seed=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, K)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)  # bf16 values
    if fmt == "mxfp4":
        codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
        scales = (127 + rng.integers(-10, -5, size=(N, 1)) - rng.choice([0, 1, 2], size=(N, K // 32),
                                                                          p=[.7, .25, .05])).astype(np.uint8)
        return x, codes, scales, None
    wb = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    wb = (wb.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)
    c, s, g = Q.nv_quantize(wb)
    return x, c, s, g


def test_mx_linear_is_the_exact_block_scaled_sum():
    x, wc, ws, _ = _inputs(3, 256, 16, "mxfp4")
    y, S, (xc, xs, _) = LIN.linear_forward(x, wc, ws, "mxfp4")
    for t in range(3):
        for n in (0, 5, 15):
            tot = Fraction(0)
            for b in range(256 // 32):
                blk = sum(int(2 * F.E2M1_TABLE[xc[t, k]]) * int(2 * F.E2M1_TABLE[wc[n, k]])
                          for k in range(32 * b, 32 * b + 32))
                tot += Fraction(blk, 4) * Fraction(2) ** (int(xs[t, b]) - 127) * Fraction(2) ** (int(ws[n, b]) - 127)
            assert Fraction(float(y[t, n])) == tot
            assert S[t, n] >= abs(y[t, n])


def test_nv_linear_is_the_two_level_block_sum():
    x, wc, ws, gw = _inputs(2, 256, 8, "nvfp4")
    y, _, (xc, xs, gx) = LIN.linear_forward(x, wc, ws, "nvfp4", gw)
    for t in range(2):
        for n in (0, 7):
            tot = Fraction(0)
            for b in range(256 // 16):
                blk = sum(int(2 * F.E2M1_TABLE[xc[t, k]]) * int(2 * F.E2M1_TABLE[wc[n, k]])
                          for k in range(16 * b, 16 * b + 16))
                tot += Fraction(blk, 4) * Fraction(F.E4M3_TABLE[xs[t, b]]) * Fraction(F.E4M3_TABLE[ws[n, b]])
            exact = tot * Fraction(float(gx)) * Fraction(float(gw))
            assert abs(Fraction(float(y[t, n])) - exact) <= abs(exact) * Fraction(2) ** -50


def test_linear_matches_loops():
    x, wc, ws, _ = _inputs(2, 64, 4, "mxfp4")
    y, _, _ = LIN.linear_forward(x, wc, ws, "mxfp4")
    for t in range(2):
        xc, xs = Q.mx_quantize(x[t:t + 1])
        a = [F.E2M1_TABLE[xc[0, k]] * 2.0 ** (int(xs[0, k // 32]) - 127) for k in range(64)]
        for n in range(4):
            w = [F.E2M1_TABLE[wc[n, k]] * 2.0 ** (int(ws[n, k // 32]) - 127) for k in range(64)]
            assert y[t, n] == math.fsum(a[k] * w[k] for k in range(64))
