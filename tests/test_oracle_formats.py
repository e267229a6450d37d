"""Pins of the oracle's element and scale formats against torch's float8
dtypes, the OCP E2M1 table and brute force."""
import math
from pathlib import Path

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = Path(__file__).parent / "golden"


def test_e2m1_table_matches_ocp_values():
    rows = [l.split() for l in (GOLDEN / "e2m1_values.txt").read_text().splitlines()
            if l and not l.startswith("#")]
    want = np.array([float(v) for _, v in rows])
    assert [int(c) for c, _ in rows] == list(range(16))
    assert np.array_equal(F.E2M1_TABLE, want)
    assert np.array_equal(np.signbit(F.E2M1_TABLE), np.signbit(want))


def test_e2m1_values_exact_in_e4m3_and_bf16():
    t = torch.tensor(F.E2M1_TABLE, dtype=torch.float64)
    assert torch.equal(t.to(torch.float8_e4m3fn).to(torch.float64), t)
    assert torch.equal(t.to(torch.bfloat16).to(torch.float64), t)


def test_e8m0_decode_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = F.E8M0_TABLE
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    # torch flushes 2^-127 (byte 0) through float32's subnormal range exactly
    assert np.array_equal(ours[:255], ref[:255])


def test_e4m3_decode_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(F.E4M3_TABLE))
    assert nan.sum() == 2
    assert np.array_equal(F.E4M3_TABLE[~nan], ref[~nan])
    assert np.array_equal(np.signbit(F.E4M3_TABLE[~nan]), np.signbit(ref[~nan]))
    assert F.E4M3_TABLE[0x7E] == 448.0


def _e4m3_probe_values():
    pos = F.E4M3_TABLE[:127]
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(1)
    rand = rng.uniform(0, 448, 20000)
    tiny = rng.uniform(0, 2.0 ** -6, 5000)
    v = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), rand, tiny])
    v = v.astype(np.float32).astype(np.float64)  # torch converts from fp32
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_rne():
    v = _e4m3_probe_values()
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = F.e4m3_encode(v)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates():
    assert F.e4m3_encode(np.array([448.0, 460.0, 1e9, -1e9])).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]


def _brute_e2m1(v):
    """Nearest E2M1 code of the same sign by enumerating all codes; a tie goes
    to the even code."""
    neg = math.copysign(1.0, v) < 0
    cands = [c for c in range(16) if bool(c >> 3) == neg]
    dist = [abs(F.E2M1_TABLE[c] - v) for c in cands]
    best = min(dist)
    ties = [c for c, d in zip(cands, dist) if d == best]
    even = [c for c in ties if c % 2 == 0]
    return (even or ties)[0]


def test_e2m1_encode_brute_force():
    pos = F.E2M1_TABLE[:8]
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(2)
    v = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 9), rng.uniform(0, 6, 3000),
                        [0.0, 6.0]])
    v = np.concatenate([v, -v])
    ours = F.e2m1_encode(v)
    for x, c in zip(v, ours):
        assert c == _brute_e2m1(x), (x, c)
    # beyond 6 saturates with sign
    assert F.e2m1_encode(np.array([6.5, 100.0, -7.0])).tolist() == [7, 7, 15]


@pytest.mark.parametrize("v,code", [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4),
                                    (3.5, 6), (5.0, 6), (-0.0, 8), (0.0, 0), (-0.2, 8)])
def test_e2m1_ties_to_even(v, code):
    assert int(F.e2m1_encode(np.array([v]))[0]) == code


def test_nibble_order():
    codes = np.array([[1, 2, 3, 15]], dtype=np.uint8)
    packed = F.pack_nibbles(codes)
    assert packed.tolist() == [[0x21, 0xF3]]
    assert np.array_equal(F.unpack_nibbles(packed), codes)


def test_floor_log2_exact():
    for k in range(-149, 128):
        x = 2.0 ** k
        assert F.floor_log2(np.array([x]))[0] == k
        assert F.floor_log2(np.array([np.nextafter(x, 0)]))[0] == k - 1
