"""W8A8 expert MLP on the exactly converted FP8 weights (FP64 oracle; test
infrastructure only).

"Kimi-K2.7-Code on Gaudi 2", section "Exact MXFP4 to FP8 per-channel
conversion": the converted experts are E4M3 weights with one power-of-two
scale per output row (channel); they load through an FP8 method with
per-channel weights and dynamic per-token activations, so the expert GEMMs
become W8A8 ("Activations become FP8 per token").  The pages fix no rule for
the activation scale.  The reading used here, every step one correctly
rounded fp32 operation in this order:

    sigma = fp32(amax_row / 448)                  (448: the largest E4M3 value)
    code  = RNE_E4M3(fp32(v / sigma))             saturating at 448;
                                                  sigma = 0 -> signed zero
    value = E4M3(code) * sigma

applied to each token's x (a row of H values) and to each route's
intermediate h (a row of I values, the W8A8 counterpart of the A4W4
requantisation).

Per route (token t, expert e, routing weight w):

    a       = dequant(quantize(x[t]))
    [g | u] = a . W13[e]^T,   W = E4M3(byte) * row_scale
    h       = silu(g) * u, rounded to fp32
    h_hat   = dequant(quantize(h))
    y       = h_hat . W2[e]^T
    out[t] += w * y                                (shared experts: w = 1)

On rows the conversion marks exact, W equals the MXFP4 weight values
element for element, so this layer differs from the A4W4 one only in how the
activations and the intermediate are quantised.  Products of E4M3 values
are multiples of 2**-18 below 2**18 in magnitude, so every dot product here
is exact in float64 before the two scales multiply it.

Tolerance: as for the A4W4 layer, |gpu - ref| <= 2**-8 |ref| + 1e-3 S + A,
with A covering elements of h whose interval h +- dh admits another FP8
quantisation (another code, or another row scale when the row's largest
element is itself uncertain).
"""
from __future__ import annotations

import numpy as np

from .convert import ST_OK, mxfp4_to_fp8_rowscale
from .formats import E4M3_TABLE, e4m3_encode
from .moe import EPS_EXP_PER_G, EPS_SWIGLU, GAMMA, SILU_LIP, silu
from .router import decision_margins, route, router_logits

FP8_MAX = 448.0


def fp8_quantize(v: np.ndarray):
    """Per-row dynamic E4M3 quantisation along the last axis.  ``v`` holds
    values exactly representable in fp32.  Returns (codes uint8 [..., K],
    sigma float32 [...])."""
    v = np.asarray(v, dtype=np.float64)
    v32 = v.astype(np.float32)
    assert np.array_equal(v32.astype(np.float64), v, equal_nan=True), "inputs must be fp32 values"
    amax = np.max(np.abs(v32), axis=-1) if v32.shape[-1] else np.zeros(v32.shape[:-1], np.float32)
    sigma = (amax / np.float32(FP8_MAX)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = np.where(sigma[..., None] > 0, v32 / sigma[..., None], np.float32(0.0) * v32)
    codes = e4m3_encode(scaled.astype(np.float32).astype(np.float64))
    return codes, sigma


def fp8_dequant(codes: np.ndarray, sigma: np.ndarray) -> np.ndarray:
    """Exact values of E4M3 codes [..., K] with per-row scales [...]."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)] * np.asarray(sigma, dtype=np.float64)[..., None]


def converted_weight(codes_packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Values of an MXFP4 weight matrix after the exact per-channel FP8
    conversion: E4M3(byte) * row_scale, row by row."""
    fp8, rs, st = mxfp4_to_fp8_rowscale(codes_packed, scales)
    assert np.all(st == ST_OK), "W8A8 weights come from rows the conversion marks exact"
    return E4M3_TABLE[fp8] * rs.astype(np.float64)[:, None]


def fp8_weight_source(cfg):
    """Expert weights of the W8A8 layer: the oracle's own conversion of the
    synthetic MXFP4 weights; get(which, e) returns the value matrix."""
    import synth
    from .moe import WeightSource

    def fn(which, e):
        codes, scales = synth.gen_mx_weight(cfg, which, e)
        return converted_weight(codes, scales)
    return WeightSource(fn)


def _h_candidates_fp8(h: np.ndarray, dh: np.ndarray, hq: np.ndarray, sig: np.ndarray, cap: int = 64):
    """Largest change of each dequantised element of h over every FP8
    quantisation of some h' with |h' - h| <= dh (h' rounded to fp32), and the
    range of admissible row scales.  The row scale depends on the row's
    largest |h'|; every fp32 value between its two extremes is tried (rows
    with more than ``cap`` candidates use the bound |q(v) - v| <= 2**-4 |v| +
    2**-10 sigma instead)."""
    n, I = h.shape
    lo, hi = h - dh, h + dh
    amax_hi = np.max(np.maximum(np.abs(lo), np.abs(hi)), axis=-1)
    amin = np.where((lo <= 0) & (hi >= 0), 0.0, np.minimum(np.abs(lo), np.abs(hi)))
    amax_lo = np.max(amin, axis=-1)
    # the row maximum of an fp32 h' lies between the fp32 values nearest to
    # amax_lo from above and to amax_hi from below
    f_lo = amax_lo.astype(np.float32)
    f_lo = np.where(f_lo < amax_lo, np.nextafter(f_lo, np.float32(np.inf)), f_lo).astype(np.float32)
    f_hi = amax_hi.astype(np.float32)
    f_hi = np.where(f_hi > amax_hi, np.nextafter(f_hi, np.float32(-np.inf)), f_hi).astype(np.float32)
    s_lo = (f_lo / np.float32(FP8_MAX)).astype(np.float32)
    s_hi = (f_hi / np.float32(FP8_MAX)).astype(np.float32)
    ref = fp8_dequant(hq, sig)
    dmax = np.zeros_like(h)
    for r in range(n):
        cands, s = [], np.float32(s_lo[r])
        while s <= s_hi[r] and len(cands) <= cap:
            cands.append(s)
            s = np.nextafter(s, np.float32(np.inf))
        if len(cands) > cap:
            vmax = np.maximum(np.abs(lo[r]), np.abs(hi[r]))
            bound = 2.0 ** -4 * vmax + 2.0 ** -10 * float(s_hi[r])
            dmax[r] = np.maximum(np.abs(lo[r] - ref[r]), np.abs(hi[r] - ref[r])) + bound
            continue
        for s in cands:
            for v in (lo[r], hi[r]):
                with np.errstate(divide="ignore", invalid="ignore"):
                    sc = (v.astype(np.float32) / s).astype(np.float32) if s > 0 else np.float32(0.0) * v
                alt = E4M3_TABLE[e4m3_encode(sc.astype(np.float64))] * float(s)
                dmax[r] = np.maximum(dmax[r], np.abs(alt - ref[r]))
    return dmax, (s_lo, s_hi)


def expert_rows_fp8(cfg, e: int, a: np.ndarray, wts: np.ndarray, weights, gamma: float = GAMMA,
                    with_ambiguity: bool = True) -> dict:
    """W8A8 MLP of expert e (ids >= E: shared experts) for the dequantised
    activation rows a [n, H] routed to it with weights wts [n]."""
    E, I = cfg.E, cfg.I
    W13 = weights.get("w13", e) if e < E else weights.get("sh13", e - E)
    W2 = weights.get("w2", e) if e < E else weights.get("sh2", e - E)
    gu = a @ W13.T
    g, u = gu[:, :I], gu[:, I:]
    h = silu(g) * u
    h32 = h.astype(np.float32).astype(np.float64)
    hq, sig = fp8_quantize(h32)
    hd = fp8_dequant(hq, sig)
    y = hd @ W2.T
    info = {"wt": wts, "h": h, "h32": h32, "hq": hq, "hsig": sig, "y": y}
    if with_ambiguity:
        gu_abs = np.abs(a) @ np.abs(W13).T
        W2a = np.abs(W2)
        info["Sy"] = np.abs(hd) @ W2a.T
        dg = gamma * gu_abs[:, :I] + 2.0 ** -22 * np.abs(g)
        du = gamma * gu_abs[:, I:] + 2.0 ** -22 * np.abs(u)
        dh = (SILU_LIP * dg * (np.abs(u) + du) + np.abs(silu(g)) * du
              + (EPS_SWIGLU + EPS_EXP_PER_G * np.abs(g)) * np.abs(h) + 2.0 ** -140)
        dmax, srange = _h_candidates_fp8(h32, dh, hq, sig)
        info.update({"dh": dh, "dmax": dmax, "scale_range": srange, "Ay": dmax @ W2a.T,
                     "n_ambiguous": int(np.count_nonzero(dmax))})
    else:
        info["Sy"] = np.zeros_like(y)
        info["Ay"] = np.zeros_like(y)
    return info


def token_forward_fp8(cfg, x_rows_f64: np.ndarray, wr_f64: np.ndarray, bias_f32: np.ndarray, weights,
                      gamma: float = GAMMA, with_ambiguity: bool = True):
    """The W8A8 layer output of individual tokens x_rows [n, H] (both
    quantisations act row by row, so a token's output depends on its own
    routes alone).  Returns routing, quantised activations, the routes'
    intermediates and ref / S / A [n, H]."""
    E, k, ns = cfg.E, cfg.top_k, cfg.n_shared
    logits, lsum = router_logits(x_rows_f64, wr_f64)
    idx, w = route(logits, bias_f32, k, cfg.n_group, cfg.topk_group, cfg.routed_scaling, cfg.renormalize)
    xc, xsig = fp8_quantize(x_rows_f64)
    n, H = x_rows_f64.shape
    ref, S, A = np.zeros((n, H)), np.zeros((n, H)), np.zeros((n, H))
    routes = []
    for i in range(n):
        a = fp8_dequant(xc[i:i + 1], xsig[i:i + 1])
        per = []
        for j, e in enumerate(list(idx[i]) + list(range(E, E + ns))):
            wt = w[i, j] if j < k else 1.0
            info = expert_rows_fp8(cfg, int(e), a, np.array([wt]), weights, gamma, with_ambiguity)
            ref[i] += wt * info["y"][0]
            S[i] += abs(wt) * info["Sy"][0]
            A[i] += abs(wt) * info["Ay"][0]
            info["expert"] = int(e)
            per.append(info)
        routes.append(per)
    margins = [decision_margins(logits[i], bias_f32, k, cfg.n_group, cfg.topk_group) for i in range(n)]
    return {"logits": logits, "lsum": lsum, "idx": idx, "w": w, "margins": margins, "xc": xc, "xsig": xsig,
            "routes": routes, "ref": ref, "S": S, "A": A}
