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
