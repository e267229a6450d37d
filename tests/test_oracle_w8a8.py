"""Pins of the W8A8 oracle (exactly converted FP8 weights, per-token dynamic
E4M3 activations): the E4M3 encoding against torch's float8_e4m3fn cast, the
scale rule's fixed points, the weight side against the MXFP4 values it was
converted from, exact integer dot products, a loop-by-loop recomputation of
the tiny layer, and the ambiguity allowance on planted boundaries."""
from fractions import Fraction
import math

import numpy as np
import torch

import synth
from oracle import formats as F
from oracle import inputs as OI
from oracle import quant as Q
from oracle import w8a8 as W


def _rows(seed=0):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((64, 96)) * np.exp2(rng.integers(-30, 30, size=(64, 1)))
    v[3] = 0.0
    v[4, :5] = [-0.0, 0.0, -0.0, 0.0, -0.0]
    v[4, 5:] = 0.0
    v[5] = np.where(np.arange(96) % 2, 1e-40, -1e-40)  # fp32 subnormals
    return v.astype(np.float32).astype(np.float64)


def test_fp8_codes_match_torch_cast():
    v = _rows()
    codes, sig = W.fp8_quantize(v)
    nz = sig > 0
    scaled = torch.from_numpy((v[nz].astype(np.float32) / sig[nz][:, None]).astype(np.float32))
    inrange = scaled.abs() <= 448
    want = scaled.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codes[nz]
    assert np.array_equal(got[inrange.numpy()], want[inrange.numpy()])
    # values that round past 448 saturate to the largest code
    assert np.all(F.E4M3_TABLE[got[~inrange.numpy()]] == np.sign(scaled[~inrange].numpy()) * 448)


def test_row_maximum_maps_to_448_and_zero_rows_keep_signs():
    v = _rows(1)
    codes, sig = W.fp8_quantize(v)
    vals = np.abs(F.E4M3_TABLE[codes])
    nz = sig > 0
    assert np.all(np.max(vals[nz], axis=1) == 448.0)
    # all-zero rows: scale 0, codes carry the sign of each zero
    assert sig[3] == 0 and np.all(codes[3] == 0)
    assert sig[4] == 0 and list(codes[4, :5]) == [0x80, 0x00, 0x80, 0x00, 0x80]
    # dequantised values stay within half an E4M3 step of the inputs
    d = W.fp8_dequant(codes, sig)
    ok = nz[:, None] & (np.abs(v) >= 2.0 ** -6 * sig[:, None])
    assert np.all(np.abs(d - v)[ok] <= 2.0 ** -4 * np.abs(v)[ok] * (1 + 2.0 ** -20))


def test_converted_weights_equal_their_mxfp4_values():
    cfg = synth.configs()["tiny"]
    for which, e in (("w13", 0), ("w2", 3)):
        codes, scales = synth.gen_mx_weight(cfg, which, e)
        mx = Q.mx_dequant(F.unpack_nibbles(codes), scales)
        assert np.array_equal(W.converted_weight(codes, scales), mx)


def test_w8a8_products_are_exact():
    cfg = synth.configs()["tiny"]
    x, _, _ = OI.layer_inputs(cfg)
    xc, xs = W.fp8_quantize(x)
    codes, scales = synth.gen_mx_weight(cfg, "w13", 1)
    from oracle.convert import mxfp4_to_fp8_rowscale
    w8, rs, _ = mxfp4_to_fp8_rowscale(codes, scales)
    Wv = F.E4M3_TABLE[w8] * rs.astype(np.float64)[:, None]
    a = W.fp8_dequant(xc, xs)
    g = a @ Wv.T
    ia = (F.E4M3_TABLE[xc] * 512).astype(np.int64)   # E4M3 values are multiples of 2^-9
    iw = (F.E4M3_TABLE[w8] * 512).astype(np.int64)
    for t in range(cfg.T):
        for n in (0, 7, cfg.I + 5, 2 * cfg.I - 1):
            exact = Fraction(int(ia[t] @ iw[n])) / 2 ** 18 * Fraction(float(xs[t])) * Fraction(float(rs[n]))
            assert Fraction(float(g[t, n])) == exact


def _loop_token(cfg, x, wr, b, ws, t):
    """One token of the tiny W8A8 layer with scalar loops (torch's E4M3 cast
    for the encoding)."""
    H, I, k = cfg.H, cfg.I, cfg.top_k

    def q8(row):
        amax = np.float32(max(abs(float(v)) for v in row))
        s = np.float32(amax / np.float32(448.0))
        sc = torch.tensor([np.float32(np.float32(v) / s) for v in row], dtype=torch.float32)
        codes = sc.clamp(-448, 448).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
        return [float(c) * float(s) for c in codes]

    l = [math.fsum(x[t, h] * wr[e, h] for h in range(H)) for e in range(cfg.E)]
    s = [0.5 * (1 + math.tanh(v / 2)) for v in l]
    c = [s[e] + float(b[e]) for e in range(cfg.E)]
    chosen = sorted(range(cfg.E), key=lambda e: (-c[e], e))[:k]
    tot = math.fsum(s[e] for e in chosen)
    a = q8(x[t])
    out = [0.0] * H
    for e in chosen:
        wt = s[e] / tot * cfg.routed_scaling
        W13, W2 = ws.get("w13", e), ws.get("w2", e)
        h = []
        for n in range(I):
            gate = math.fsum(a[j] * W13[n, j] for j in range(H))
            up = math.fsum(a[j] * W13[I + n, j] for j in range(H))
            h.append(float(np.float32(gate * (0.5 * (1 + math.tanh(gate / 2))) * up)))
        hd = q8(h)
        for o in range(H):
            out[o] += wt * math.fsum(hd[i] * W2[o, i] for i in range(I))
    return np.array(out)


def test_tiny_layer_matches_loops():
    cfg = synth.configs()["tiny"]
    x, wr, b = OI.layer_inputs(cfg)
    ws = W.fp8_weight_source(cfg)
    for t in (0, 3):
        ref = W.token_forward_fp8(cfg, x[t:t + 1], wr, b, ws)["ref"][0]
        np.testing.assert_allclose(ref, _loop_token(cfg, x, wr, b, ws, t), rtol=1e-12, atol=1e-15)


def test_ambiguity_allowance_on_planted_boundaries():
    # scale 1 (amax 448); 3.125 lies exactly between the E4M3 values 3.0 and 3.25
    h = np.zeros((1, 16))
    h[0, 0] = 448.0
    h[0, 1] = 3.125
    hq, sig = W.fp8_quantize(h)
    assert sig[0] == 1.0 and F.E4M3_TABLE[hq[0, 1]] == 3.0  # ties to the even code
    none, _ = W._h_candidates_fp8(h, np.zeros_like(h), hq, sig)
    assert not none.any()
    dh = np.zeros_like(h)
    dh[0, 1] = 1e-6
    dmax, _ = W._h_candidates_fp8(h, dh, hq, sig)
    assert dmax[0, 1] == 0.25 and dmax[0, 2:].max() == 0.0
    # an uncertain row maximum moves the row scale, so every code may move
    dmax2, (lo, hi) = W._h_candidates_fp8(h, np.full_like(h, 1e-3), hq, sig)
    assert lo[0] < sig[0] < hi[0] and dmax2[0, 0] > 0
