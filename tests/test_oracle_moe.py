"""Pins of the oracle's expert MLP and combine: exact integer accumulation of
the MXFP4 products, a loop-by-loop recomputation of the tiny layer, the
ambiguity allowance on planted boundary cases, and the NVFP4 layer path."""
from dataclasses import replace
from fractions import Fraction
import math

import numpy as np

import synth
from oracle import formats as F
from oracle import inputs as OI
from oracle import moe as M
from oracle import quant as Q


def _exact_dot(qa, ea, qw, ew):
    """sum_k E2M1(qa_k) 2^ea_k * E2M1(qw_k) 2^ew_k with Python integers."""
    ia = [int(2 * F.E2M1_TABLE[c]) for c in qa]
    iw = [int(2 * F.E2M1_TABLE[c]) for c in qw]
    ex = [int(a + b) - 2 for a, b in zip(ea, ew)]
    m = min(ex)
    tot = sum((x * y) << (e - m) for x, y, e in zip(ia, iw, ex))
    return Fraction(tot) * Fraction(2) ** m


def test_mx_gate_up_is_exact():
    cfg = synth.configs()["tiny"]
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    out = M.layer_forward(cfg, x, wr, b, ws)
    xc, xs = out["xc"], out["xs"]
    for e, info in list(out["experts"].items())[:2]:
        wc, wsc, _ = ws.get("w13", e)
        W = Q.mx_dequant(wc, wsc)
        for r in range(min(2, len(info["tok"]))):
            t = info["tok"][r]
            a = Q.mx_dequant(xc[t:t + 1], xs[t:t + 1])[0]
            g = a @ W.T
            for n in (0, 5, cfg.I + 3):
                ea = np.repeat(xs[t].astype(np.int64) - 127, 32)
                ew = np.repeat(wsc[n].astype(np.int64) - 127, 32)
                assert Fraction(float(g[n])) == _exact_dot(xc[t], ea, wc[n], ew)


def _loop_layer(cfg, x, wr, b, ws):
    """The tiny layer recomputed route by route with scalar loops."""
    T, H, I, k = cfg.T, cfg.H, cfg.I, cfg.top_k
    out = np.zeros((T, H))
    xc, xs = Q.mx_quantize(x)
    for t in range(T):
        l = [math.fsum(x[t, h] * wr[e, h] for h in range(H)) for e in range(cfg.E)]
        s = [0.5 * (1 + math.tanh(v / 2)) for v in l]
        c = [s[e] + float(b[e]) for e in range(cfg.E)]
        chosen = sorted(range(cfg.E), key=lambda e: (-c[e], e))[:k]
        tot = math.fsum(s[e] for e in chosen)
        a = Q.mx_dequant(xc[t:t + 1], xs[t:t + 1])[0]
        for e in chosen:
            wt = s[e] / tot * cfg.routed_scaling
            wc, wsc, _ = ws.get("w13", e)
            W13 = Q.mx_dequant(wc, wsc)
            gate = np.array([math.fsum(a * W13[n]) for n in range(I)])
            up = np.array([math.fsum(a * W13[I + n]) for n in range(I)])
            sig = 0.5 * (1 + np.tanh(gate / 2))
            h = (gate * sig * up).astype(np.float32).astype(np.float64)
            hc, hsc = Q.mx_quantize(h[None])
            hd = Q.mx_dequant(hc, hsc)[0]
            wc2, wsc2, _ = ws.get("w2", e)
            W2 = Q.mx_dequant(wc2, wsc2)
            out[t] += wt * np.array([math.fsum(hd * W2[o]) for o in range(H)])
    return out


def test_tiny_layer_matches_loops():
    cfg = synth.configs()["tiny"]
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    ref = M.layer_forward(cfg, x, wr, b, ws)["ref"]
    loops = _loop_layer(cfg, x, wr, b, ws)
    np.testing.assert_allclose(ref, loops, rtol=1e-12, atol=1e-15)


def test_ambiguity_allowance_on_planted_midpoint():
    h = np.zeros((1, 32))
    h[0, 0] = 6.0          # scale 2^0
    h[0, 1] = 2.5          # exactly between 2 and 3 -> 2 by ties-to-even
    hq, hs = Q.mx_quantize(h)
    none, _ = M._h_candidates_mx(h, np.zeros_like(h), hq, hs)
    assert not none.any()
    dh = np.full_like(h, 1e-9)
    dmax, _ = M._h_candidates_mx(h, dh, hq, hs)
    assert dmax[0, 1] == 1.0 and dmax[0, 0] == 0.0 and dmax[0, 2:].max() == 0.0
    # amax next to a power of two: the whole block may take the other scale
    h2 = np.zeros((1, 32))
    h2[0, 0] = 4.0
    h2[0, 1] = 1.0
    hq2, hs2 = Q.mx_quantize(h2)
    dmax2, (lo, hi) = M._h_candidates_mx(h2, np.full_like(h2, 1e-9), hq2, hs2)
    assert lo[0, 0] == 126 and hi[0, 0] == 127
    assert dmax2[0, 0] > 0


def test_nvfp4_layer_small():
    cfg = replace(synth.configs()["deepseek_nvfp4"], T=6, H=128, I=64, E=16, top_k=4,
                  n_group=4, topk_group=2)
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    out = M.layer_forward(cfg, x, wr, b, ws)
    assert out["gx"] == Q.nv_global_scale(np.max(np.abs(x)))
    for e, info in out["experts"].items():
        g_h = info["g_h"]
        assert g_h == Q.nv_global_scale(np.max(np.abs(info["h32"])))
    # the layer output equals the per-route sum recomputed from intermediates
    re = np.zeros_like(out["ref"])
    for e, info in out["experts"].items():
        w2 = ws.get("w2", e)
        W2 = Q.nv_dequant(*w2)
        y = Q.nv_dequant(info["hq"], info["hs"], info["g_h"]) @ W2.T
        for r, t in enumerate(info["tok"]):
            re[t] += info["wt"][r] * y[r]
    np.testing.assert_allclose(out["ref"], re, rtol=1e-13, atol=1e-16)
    assert np.all(M.tolerance(out["ref"], out["S"], out["A"]) > 0)


def test_shared_expert_gets_every_token_with_weight_one():
    cfg = replace(synth.configs()["tiny"], n_shared=1)
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    out = M.layer_forward(cfg, x, wr, b, ws)
    sh = out["experts"][cfg.E]
    assert list(sh["tok"]) == list(range(cfg.T)) and np.all(sh["wt"] == 1.0)
    base = M.layer_forward(replace(cfg, n_shared=0), x, wr, b, ws)["ref"]
    W2 = Q.mx_dequant(*ws.get("sh2", 0)[:2])
    y = Q.mx_dequant(sh["hq"], sh["hs"]) @ W2.T
    np.testing.assert_allclose(out["ref"], base + y, rtol=1e-13, atol=1e-16)


def test_token_forward_matches_layer_forward():
    cfg = replace(synth.configs()["tiny"], n_shared=1)
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    full = M.layer_forward(cfg, x, wr, b, ws)
    for t in range(cfg.T):
        one = M.token_forward(cfg, x[t:t + 1], wr, b, ws)
        assert np.array_equal(one["idx"][0], full["idx"][t])
        np.testing.assert_allclose(one["ref"][0], full["ref"][t], rtol=1e-13, atol=1e-16)
        np.testing.assert_allclose(one["S"][0], full["S"][t], rtol=1e-13, atol=1e-16)


# ------------------------------------------------------------------ NVFP4 flip allowance
def _nv_case(n_blocks=2):
    """One row of n_blocks NVFP4 blocks: element 0 holds the tensor maximum
    2688 * 2^-10, so g = 2^-10 exactly and block 0's scale is 448
    (d = 448 g = 0.4375); element 1 sits on the E2M1 midpoint 2.5 d."""
    h = np.zeros((1, 16 * n_blocks))
    h[0, 0] = 2688 * 2.0 ** -10
    h[0, 1] = 2.5 * 0.4375
    return h


def _nv_sampled_alternatives(h, dh, hq, hs, g_h, rng, n=400):
    """Brute force: quantise fp32 points h' of the box |h' - h| <= dh (its
    corners, random points, and the points that move only the tensor
    maximum) with their own tensor scale; return the largest change of each
    dequantised element and the range of block-scale bytes seen."""
    ref = Q.nv_dequant(hq, hs, g_h)
    worst = np.zeros_like(h)
    s_lo = hs.astype(np.int64).copy()
    s_hi = hs.astype(np.int64).copy()
    for i in range(n):
        mode = i % 3
        d = rng.choice([-1.0, 1.0], h.shape) if mode == 0 else rng.uniform(-1, 1, h.shape)
        if mode == 2:
            d = np.zeros_like(h)
            d.flat[int(np.argmax(np.abs(h)))] = rng.choice([-1.0, 1.0])
        hp = (h + d * dh).astype(np.float32).astype(np.float64)
        hp = np.where(np.abs(hp - h) <= dh, hp, h)
        c, s, g = Q.nv_quantize(hp)
        worst = np.maximum(worst, np.abs(Q.nv_dequant(c, s, g) - ref))
        s_lo = np.minimum(s_lo, s.astype(np.int64))
        s_hi = np.maximum(s_hi, s.astype(np.int64))
    return worst, (s_lo, s_hi)


def test_nv_allowance_planted_midpoint():
    """An element on the E2M1 midpoint 2.5 d under a fixed block scale
    (nothing else may move): the allowance is exactly one grid step d there
    (2 d by ties-to-even, 3 d on the other side) and zero elsewhere; with no
    interval it is zero everywhere."""
    h = _nv_case()
    hq, hs, g = Q.nv_quantize(h)
    assert g == np.float32(2.0 ** -10) and F.E4M3_TABLE[hs[0, 0]] == 448.0
    assert F.E2M1_TABLE[hq[0, 1]] == 2.0
    none, (lo, hi) = M._h_candidates_nv(h, np.zeros_like(h), hq, hs, g)
    assert not none.any() and np.array_equal(lo, hs) and np.array_equal(hi, hs)
    dh = np.zeros_like(h)
    dh[0, 1] = 2.0 ** -20
    dmax, (lo, hi) = M._h_candidates_nv(h, dh, hq, hs, g)
    assert dmax[0, 1] == 0.4375
    assert np.count_nonzero(dmax) == 1
    assert np.array_equal(lo, hs) and np.array_equal(hi, hs)
    worst, (slo, shi) = _nv_sampled_alternatives(h, dh, hq, hs, g, np.random.default_rng(31))
    assert np.array_equal(worst, dmax)


def test_nv_allowance_planted_block_scale_boundary():
    """Block 1's maximum makes amax_b / (6 g) = 8.5, the midpoint of the
    E4M3 values 8 and 9, and may move by one fp32 step: its scale byte may
    be either (8 by ties-to-even),
    and its maximum element, 6 * 8 g under scale 8, becomes 6 * 9 g under 9."""
    h = _nv_case()
    g = 2.0 ** -10
    h[0, 16] = 8.5 * 6 * g
    hq, hs, gq = Q.nv_quantize(h)
    assert gq == np.float32(g) and F.E4M3_TABLE[hs[0, 1]] == 8.0
    dh = np.zeros_like(h)
    dh[0, 16] = float(np.spacing(np.float32(h[0, 16])))  # one fp32 step: the box holds amax_b +- that step
    dmax, (lo, hi) = M._h_candidates_nv(h, dh, hq, hs, gq)
    assert F.E4M3_TABLE[lo[0, 1]] == 8.0 and F.E4M3_TABLE[hi[0, 1]] == 9.0
    assert lo[0, 0] == hi[0, 0] == hs[0, 0]
    assert dmax[0, 16] == 6 * g
    assert np.count_nonzero(dmax) == 1
    worst, (slo, shi) = _nv_sampled_alternatives(h, dh, hq, hs, gq, np.random.default_rng(32))
    assert np.array_equal(worst, dmax)
    assert np.array_equal(slo, lo) and np.array_equal(shi, hi)


def test_nv_allowance_planted_tensor_scale_change():
    """The tensor maximum may move by one fp32 step either way, which moves
    g = amax / 2688 and with it every quotient of the tensor: the midpoint
    element, with no interval of its own, may round to 3 * 448 g_lo (the
    smaller g) instead of 2 * 448 g.  The allowance admits that flip; it
    exceeds the exact largest change by at most the spread of the grid
    value times 448 (g_hi - g_lo), its bilinear corner bound."""
    h = _nv_case()
    hq, hs, g = Q.nv_quantize(h)
    dh = np.zeros_like(h)
    dh[0, 0] = float(np.spacing(np.float32(h[0, 0])))
    dmax, (lo, hi) = M._h_candidates_nv(h, dh, hq, hs, g)
    g_lo = float(Q.nv_global_scale(np.float32(h[0, 0] - dh[0, 0])))
    g_hi = float(Q.nv_global_scale(np.float32(h[0, 0] + dh[0, 0])))
    assert g_lo < g < g_hi and np.array_equal(lo, hs) and np.array_equal(hi, hs)
    exact = 3 * 448 * g_lo - 2 * 448 * float(g)  # dequantised values are E2M1 * E4M3 * g exactly
    assert exact <= dmax[0, 1] <= exact + 3 * 448 * (g_hi - g_lo)
    worst, _ = _nv_sampled_alternatives(h, dh, hq, hs, g, np.random.default_rng(33))
    assert worst[0, 1] == exact
    assert np.all(worst <= dmax) and np.all((dmax > 0) == (h != 0))


def test_nv_allowance_bounds_random_boxes():
    """Soundness on random rows with intervals wide enough to cross many
    boundaries: no sampled quantisation of the box changes an element by
    more than the allowance, and every sampled scale byte is in its range."""
    rng = np.random.default_rng(34)
    for trial in range(6):
        h = (rng.standard_normal((3, 64)) * 2.0 ** rng.integers(-8, 4)).astype(np.float32).astype(np.float64)
        dh = np.abs(h) * 2.0 ** -rng.integers(6, 14) + 2.0 ** -40
        hq, hs, g = Q.nv_quantize(h)
        dmax, (lo, hi) = M._h_candidates_nv(h, dh, hq, hs, g)
        worst, (slo, shi) = _nv_sampled_alternatives(h, dh, hq, hs, g, rng, n=300)
        assert np.all(worst <= dmax * (1 + 1e-12)), (trial, float(np.max(worst - dmax)))
        assert np.all(slo >= lo) and np.all(shi <= hi)


def test_mx_allowance_bounds_random_boxes():
    """The MXFP4 allowance, the same way: no sampled fp32 point of a wide box
    quantises to a value further from the reference than the allowance, and
    every sampled scale byte lies in the allowed range."""
    rng = np.random.default_rng(35)
    for trial in range(6):
        h = (rng.standard_normal((3, 64)) * 2.0 ** rng.integers(-8, 4)).astype(np.float32).astype(np.float64)
        dh = np.abs(h) * 2.0 ** -rng.integers(4, 12) + 2.0 ** -40
        hq, hs = Q.mx_quantize(h)
        dmax, (lo, hi) = M._h_candidates_mx(h, dh, hq, hs)
        ref = Q.mx_dequant(hq, hs)
        for i in range(300):
            d = rng.choice([-1.0, 1.0], h.shape) if i % 2 else rng.uniform(-1, 1, h.shape)
            hp = (h + d * dh).astype(np.float32).astype(np.float64)
            hp = np.where(np.abs(hp - h) <= dh, hp, h)
            c, s = Q.mx_quantize(hp)
            assert np.all(np.abs(Q.mx_dequant(c, s) - ref) <= dmax), (trial, i)
            assert np.all(s >= lo) and np.all(s <= hi)
