"""Pins of the oracle's MXFP4 / NVFP4 quantisers: hand-derived blocks, brute
force, idempotence, torch's E4M3 rounding and the block-scaled product
invariant."""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quant as Q

GOLDEN = Path(__file__).parent / "golden"


def _golden_blocks():
    out = []
    for line in (GOLDEN / "mx_blocks.txt").read_text().splitlines():
        if not line or line.startswith("#"):
            continue
        name, vals, byte, codes = [p.strip() for p in line.split("|")]
        if "*" in vals:
            v, n = vals.split("*")
            block = [float(v)] * int(n)
        else:
            block = [float(x) for x in vals.split()]
        block = block + [0.0] * (32 - len(block))
        out.append((name, np.array(block), int(byte), [int(c) for c in codes.split()]))
    return out


@pytest.mark.parametrize("name,block,byte,codes", _golden_blocks())
def test_mx_hand_blocks(name, block, byte, codes):
    c, s = Q.mx_quantize(block[None, :])
    assert int(s[0, 0]) == byte
    assert c[0, :8].tolist() == codes


def test_mx_nearest_grid_point():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    v = v.astype(np.float32).astype(np.float64)
    c, s = Q.mx_quantize(v)
    e = s.astype(np.int64) - 127
    scaled = np.ldexp(v.reshape(64, 8, 32), -e[..., None])
    assert np.all(np.max(np.abs(scaled), axis=-1) >= 4) and np.all(np.max(np.abs(scaled), axis=-1) < 8)
    grid = F.E2M1_TABLE
    for r in range(4):
        for b in range(8):
            for i in range(32):
                x = scaled[r, b, i]
                d = np.abs(grid - x)
                d[np.signbit(grid) != np.signbit(x)] = np.inf
                best = np.flatnonzero(d == d.min())
                best = best[best % 2 == 0] if len(best) > 1 else best
                assert c[r, b * 32 + i] == best[0]


def test_mx_idempotent():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((16, 128)).astype(np.float32).astype(np.float64)
    c, s = Q.mx_quantize(v)
    d = Q.mx_dequant(c, s)
    c2, s2 = Q.mx_quantize(d)
    assert np.array_equal(s, s2)
    assert np.array_equal(Q.mx_dequant(c2, s2), d)


def test_mx_dequant_nan_scale():
    c = np.zeros((1, 32), dtype=np.uint8)
    assert np.all(np.isnan(Q.mx_dequant(c, np.array([[255]], dtype=np.uint8))))


def _int_block_dot(qa, qb, sa, sb, blk, scale_val):
    """Block-scaled product with exact integer inner sums (2*E2M1 is an integer)."""
    K = qa.shape[-1]
    tot = Fraction(0)
    ia = (2 * F.E2M1_TABLE[qa]).astype(np.int64)
    ib = (2 * F.E2M1_TABLE[qb]).astype(np.int64)
    for b in range(K // blk):
        inner = int(np.dot(ia[b * blk:(b + 1) * blk], ib[b * blk:(b + 1) * blk]))
        tot += Fraction(inner, 4) * Fraction(scale_val(sa[b])) * Fraction(scale_val(sb[b]))
    return tot


def test_mx_block_scaled_product_invariant():
    rng = np.random.default_rng(5)
    for _ in range(10):
        a = rng.standard_normal(256).astype(np.float32).astype(np.float64)
        w = (rng.standard_normal(256) * 0.02).astype(np.float32).astype(np.float64)
        ca, sa = Q.mx_quantize(a[None])
        cw, sw = Q.mx_quantize(w[None])
        lhs = float(np.dot(Q.mx_dequant(ca, sa)[0], Q.mx_dequant(cw, sw)[0]))
        rhs = _int_block_dot(ca[0], cw[0], sa[0], sw[0], 32, lambda b: F.E8M0_TABLE[b])
        assert Fraction(lhs) == rhs


def test_nv_qdq_gemm_equals_block_scaled_product():
    """'Serving NVFP4 models on AMD Instinct MI355 accelerators': activations
    pass through NVFP4 QDQ and both operands enter a higher-precision GEMM; that
    product must equal the block-scaled form g_a g_w sum_b s_a s_w sum q q."""
    rng = np.random.default_rng(6)
    for _ in range(10):
        a = rng.standard_normal((1, 512)).astype(np.float32).astype(np.float64)
        w = (rng.standard_normal((1, 512)) * 0.02).astype(np.float32).astype(np.float64)
        ca, sa, ga = Q.nv_quantize(a)
        cw, sw, gw = Q.nv_quantize(w)
        da, dw = Q.nv_dequant(ca, sa, ga)[0], Q.nv_dequant(cw, sw, gw)[0]
        lhs = float(np.dot(da, dw))
        rhs = _int_block_dot(ca[0], cw[0], sa[0], sw[0], 16, lambda b: F.E4M3_TABLE[b])
        rhs *= Fraction(float(ga)) * Fraction(float(gw))
        # the dequantised operands are exact in float64 (<= 31 significant
        # bits); their products round once at 2^-53, the sum adds its own
        assert abs(Fraction(lhs) - rhs) <= Fraction(2.0 ** -50) * Fraction(float(np.dot(np.abs(da), np.abs(dw))))


def test_nv_steps_against_torch_and_brute_force():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((8, 64)) * np.exp2(rng.integers(-6, 6, (8, 1)))).astype(np.float32)
    v64 = v.astype(np.float64)
    c, s, g = Q.nv_quantize(v64)
    amax = np.float32(np.max(np.abs(v)))
    assert g == np.float32(amax / np.float32(2688.0))
    six_g = np.float32(6.0) * g
    amax_b = np.max(np.abs(v.reshape(8, 4, 16)), axis=-1)
    qs = (amax_b / six_g).astype(np.float32)
    s_torch = torch.tensor(qs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s, s_torch)
    d = (F.E4M3_TABLE[s].astype(np.float32) * g).astype(np.float32)
    sc = (v.reshape(8, 4, 16) / d[..., None]).astype(np.float32).astype(np.float64)
    grid = F.E2M1_TABLE
    for r in range(8):
        for b in range(4):
            for i in range(16):
                x = min(abs(sc[r, b, i]), 6.0) * (1 if sc[r, b, i] >= 0 else -1)
                dd = np.abs(grid - x)
                dd[np.signbit(grid) != np.signbit(sc[r, b, i])] = np.inf
                best = np.flatnonzero(dd == dd.min())
                best = best[best % 2 == 0] if len(best) > 1 else best
                assert c[r, b * 16 + i] == best[0]


def test_nv_block_scale_hits_448():
    v = np.zeros((1, 32))
    v[0, 0] = 1000.0
    v[0, 16] = 1.0
    c, s, g = Q.nv_quantize(v)
    assert g == np.float32(np.float32(1000.0) / np.float32(2688.0))
    assert int(s[0, 0]) == 0x7E  # 1000 / (6 g) rounds to 448
    assert int(c[0, 0]) == 7


def test_nv_all_zero():
    c, s, g = Q.nv_quantize(np.zeros((2, 32)))
    assert g == 0 and not c.any() and not s.any()
