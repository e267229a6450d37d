"""Pins of the oracle's exact MXFP4 -> FP8 per-channel conversion ("Kimi-K2.7-Code
on Gaudi 2", section "Exact MXFP4 to FP8 per-channel conversion" and the
"Correctness" table): lossless round trip through torch's E4M3 decoding, the
[-5, 7] exponent window and 192 bound, the span <= 9 theorem and its floor
edge, E8M0 bytes 0 / 254 / 255, the halving replay, and a mutation suite."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from oracle import convert as C
from oracle import formats as F
from oracle import quant as Q


def _torch_e4m3_values(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _exact_roundtrip(codes, scales, fp8, row_scale):
    """decode(fp8) * scale == dequant(MXFP4) for every element (exact)."""
    R = codes.shape[0]
    ref = Q.mx_dequant(F.unpack_nibbles(codes), scales)
    got = _torch_e4m3_values(fp8) * row_scale.astype(np.float64)[:, None]
    return np.all(got == ref, axis=1) & np.all(np.signbit(got) == np.signbit(ref), axis=1)


def _rows_with_span(rng, n, K, span):
    nb = K // 32
    codes = rng.integers(0, 256, (n, K // 2), dtype=np.uint8)
    lo = rng.integers(1, 254 - span, n)
    sc = lo[:, None] + rng.integers(0, span + 1, (n, nb))
    sc[:, 0] = lo
    sc[:, -1] = lo + span
    return codes, sc.astype(np.uint8)


def test_synthetic_weights_roundtrip_exactly():
    cfg = synth.configs()["tiny"]
    codes, scales = synth.gen_mx_weight(cfg, "w13", 3)
    fp8, rs, st = C.mxfp4_to_fp8_rowscale(codes, scales)
    assert np.all(st == C.ST_OK)
    assert np.all(_exact_roundtrip(codes, scales, fp8, rs))


@pytest.mark.parametrize("span", [0, 1, 2, 5, 9])
def test_span_at_most_9_is_lossless(span):
    rng = np.random.default_rng(20 + span)
    codes, scales = _rows_with_span(rng, 200, 512, span)
    fp8, rs, st = C.mxfp4_to_fp8_rowscale(codes, scales)
    assert np.all(st == C.ST_OK)
    assert np.all(_exact_roundtrip(codes, scales, fp8, rs))
    vals = _torch_e4m3_values(fp8)
    assert np.max(np.abs(vals)) <= 192
    nz = vals != 0
    ex = F.floor_log2(np.where(nz, vals, 1.0))
    assert ex[nz].min() >= -5 and ex[nz].max() <= 7


def test_floor_edge_rows():
    codes, scales, names = synth.adversarial_conversion_rows()
    fp8, rs, st = C.mxfp4_to_fp8_rowscale(codes, scales)
    got = dict(zip(names, st.tolist()))
    assert got["span9"] == C.ST_OK and got["span9_low"] == C.ST_OK
    assert got["span10"] == C.ST_BELOW_FLOOR
    assert got["span12_mild"] == C.ST_OK  # the span rule is sufficient, not necessary
    assert got["e8m0_0"] == C.ST_OK and got["e8m0_254"] == C.ST_OK
    assert got["e8m0_255"] == C.ST_NAN_SCALE
    i = names.index("e8m0_255")
    assert np.isnan(rs[i]) and not fp8[i].any()
    ok = st != C.ST_NAN_SCALE
    rt = _exact_roundtrip(codes[ok], scales[ok], fp8[ok], rs[ok])
    assert np.all(rt)  # even span10 is exact here: E4M3 exponent -6 is still normal
    i = names.index("e8m0_0")
    assert rs[i] == np.float32(2.0 ** -132)  # fp32 subnormal, not flushed
    i = names.index("e8m0_254")
    assert rs[i] == np.float32(2.0 ** 122)
    i = names.index("all_zero")
    assert rs[i] == 1.0 and not fp8[i].any()
    i = names.index("neg_zero")
    assert np.all(fp8[i] == 0x80)


def test_below_floor_rounds_to_nearest():
    # one block at scale 2^12, the rest at 2^0: elements 0.5 land at 2^-1-12+... < 2^-9
    K = 64
    codes = np.full((1, K // 2), 0x11, dtype=np.uint8)
    codes[0, :16] = 0x77
    scales = np.array([[127 + 14, 127]], dtype=np.uint8)
    fp8, rs, st = C.mxfp4_to_fp8_rowscale(codes, scales)
    assert st[0] == C.ST_BELOW_FLOOR
    # largest 6 * 2^14 -> k = 16 - 7 = 9; 0.5 / 2^9 = 2^-10 -> half of the
    # smallest subnormal 2^-9 -> ties to even -> 0
    assert rs[0] == 2.0 ** 9
    assert np.all(fp8[0, 32:] == 0)


def test_halving_replay_stays_normal():
    rng = np.random.default_rng(30)
    codes, scales = _rows_with_span(rng, 100, 256, 9)
    fp8, rs, st = C.mxfp4_to_fp8_rowscale(codes, scales)
    vals = _torch_e4m3_values(fp8)
    half = vals / 2
    back = torch.tensor(half).to(torch.float8_e4m3fn)
    assert np.array_equal(back.to(torch.float64).numpy(), half)
    bits = back.view(torch.uint8).numpy()
    nz = half != 0
    assert np.all(((bits >> 3) & 15)[nz] >= 1)  # exponent field >= 1: normal


# ---------------------------------------------------------------- mutations
# Each mutation plants one mistake in the oracle (by patching the module) and
# must make the check suite below fail.

def _swapped_unpack(p):
    out = F.unpack_nibbles(p)
    out[..., 0::2], out[..., 1::2] = out[..., 1::2].copy(), out[..., 0::2].copy()
    return out


def _signless_encode(v):
    return F.e4m3_encode(np.abs(v))


def _truncating_encode(v):
    # converted elements carry significand 1.0 or 1.5: drop the 0.5 (bit 2)
    return F.e4m3_encode(v) & np.uint8(0xFB)


MUTANTS = {
    "shift_6": ("SHIFT", 6),
    "shift_8": ("SHIFT", 8),
    "floor_minus_6": ("FLOOR", -6),
    "e8m0_bias_126": ("E8M0_BIAS", 126),
    "swap_nibbles": ("unpack_nibbles", _swapped_unpack),
    "drop_sign": ("e4m3_encode", _signless_encode),
    "lose_half_significand": ("e4m3_encode", _truncating_encode),
    "nan_as_ok": ("ST_NAN_SCALE", 0),
    "floor_as_ok": ("ST_BELOW_FLOOR", 0),
}


def _suite(conv):
    """The checks above, as one predicate over a converter."""
    rng = np.random.default_rng(40)
    codes, scales = _rows_with_span(rng, 64, 256, 9)
    a_c, a_s, names = synth.adversarial_conversion_rows()
    try:
        fp8, rs, st = conv(codes, scales)
        if not np.all(st == 0) or not np.all(_exact_roundtrip(codes, scales, fp8, rs)):
            return False
        vals = _torch_e4m3_values(fp8)
        nz = vals != 0
        ex = F.floor_log2(np.where(nz, vals, 1.0))
        if np.max(np.abs(vals)) > 192 or ex[nz].min() < -5 or ex[nz].max() > 7:
            return False
        fp8, rs, st = conv(a_c, a_s)
        want = {"span9": 0, "span10": 1, "e8m0_255": 2, "e8m0_0": 0, "span12_mild": 0}
        for n, v in want.items():
            if st[names.index(n)] != v:
                return False
        ok = np.array([n != "e8m0_255" for n in names])
        return bool(np.all(_exact_roundtrip(a_c[ok], a_s[ok], fp8[ok], rs[ok])))
    except Exception:
        return False


def test_suite_accepts_oracle():
    assert _suite(C.mxfp4_to_fp8_rowscale)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutation_is_caught(name, monkeypatch):
    attr, val = MUTANTS[name]
    monkeypatch.setattr(C, attr, val)
    assert not _suite(C.mxfp4_to_fp8_rowscale), name
