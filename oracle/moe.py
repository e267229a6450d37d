"""Expert MLP, weighted combine and output tolerance (FP64 oracle; test only).

Per route (token t, expert e, routing weight w) the layer computes, following
the block-scaled dataflow of "Serve Kimi-K2.5-MXFP4 on MI355X with ATOM"
(Figure 1 and section "When Is the Scale Applied?": scales enter inside the
product, both operands block-scaled FP4) and the fused-MoE stages of section
"Stage D: MXFP4 Fused MoE":

    a       = dequant(quantize(x[t]))                  activations (A4)
    [g | u] = a . W13[e]^T                             gate rows, then up rows
    h       = silu(g) * u,   silu(g) = g / (1 + exp(-g))
    h_hat   = dequant(quantize(fp32(h)))               A4W4 intermediate
    y       = h_hat . W2[e]^T
    out[t] += w * y                                    (shared experts: w = 1)

"Serving NVFP4 models on AMD Instinct MI355 accelerators" (section "Weight
Dequantization and Activation QDQ") fixes what a block-scaled product equals:
the operands pass through quantise-dequantise and are multiplied in higher
precision, which is what the float64 products here do.  The dequantised
operands are exact float64 values.  For MXFP4, with the bounded exponent range
of these inputs, every product and partial sum is exact too; for NVFP4 the
products carry up to 62 significant bits and round at 2**-53.

Readings where the pages are silent: the intermediate h is rounded to fp32
before it is quantised; for NVFP4 its tensor scale is one per expert
(amax over that expert's h), the activation x has one per call.

Tolerance.  An output element passes when

    |gpu - ref| <= 2**-8 |ref| + 1e-3 * S + A,

S = sum_j |w_j| sum_i |h_hat_ji * W2[e_j, h, i]| (plus shared experts), and A
allows for the quantised intermediate flipping where the GPU's fp32 h may fall
on the other side of a rounding or scale boundary: A sums, over every element
whose interval [h - dh, h + dh] admits another quantisation, the largest change
of its dequantised value times |w_j * W2|.  dh follows from the accumulation
error bound GAMMA * sum_k |a_k * w_k| of the fp32 GEMM.
"""
from __future__ import annotations

import numpy as np

from . import quant as Q
from .formats import E2M1_TABLE, E4M3_TABLE, e2m1_encode, e4m3_encode, floor_log2
from .permute import permute
from .router import decision_margins, route, router_logits

# Relative accumulation-error bound of an fp32 GEMM output:
# |acc_gpu - acc_exact| <= GAMMA * sum_k |a_k * w_k|.
GAMMA = 2.0 ** -16
# Relative error allowed for the fp32 SwiGLU arithmetic: a few roundings
# (EPS_SWIGLU) plus, for an exponential evaluated with the hardware unit, an
# error that grows with the argument: at most 2 + 1.173 |g| units in the last
# place of e^-g (the documented bound of CUDA's fast exponential), which the
# sigmoid passes on at most once.  The pages fix no precision for this step.
EPS_SWIGLU = 2.0 ** -20
EPS_EXP_PER_G = 2.5 * 2.0 ** -24
SILU_LIP = 1.1  # max |silu'|


def silu(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def _h_candidates_mx(h: np.ndarray, dh: np.ndarray, hq: np.ndarray, hs: np.ndarray):
    """Largest change of each dequantised element over every MXFP4 quantisation
    of some h' with |h' - h| <= dh.  Also returns the candidate scale-byte
    range per block (for checking the GPU's own choice)."""
    n, I = h.shape
    B = Q.MX_BLOCK
    hb = h.reshape(n, I // B, B)
    db = dh.reshape(n, I // B, B)
    lo = hb - db
    hi = hb + db
    amax_hi = np.max(np.maximum(np.abs(lo), np.abs(hi)), axis=-1)
    amin = np.where((lo <= 0) & (hi >= 0), 0.0, np.minimum(np.abs(lo), np.abs(hi)))
    amax_lo = np.max(amin, axis=-1)

    def exp_of(a):
        return np.clip(np.where(a > 0, floor_log2(np.where(a > 0, a, 1.0)) - 2, -127), -127, 127)

    e_lo = exp_of(amax_lo)
    e_hi = exp_of(amax_hi)
    ref = Q.mx_dequant(hq, hs).reshape(n, I // B, B)
    dmax = np.zeros_like(hb)
    for de in range(0, int(np.max(e_hi - e_lo)) + 1 if e_hi.size else 1):
        e = e_lo + de
        ok = e <= e_hi
        for v in (lo, hi):
            c = e2m1_encode(np.ldexp(v, -e[..., None])).astype(np.int64)
            alt = np.ldexp(E2M1_TABLE[c], e[..., None])
            d = np.where(ok[..., None], np.abs(alt - ref), 0.0)
            dmax = np.maximum(dmax, d)
    return dmax.reshape(n, I), (e_lo + 127, e_hi + 127)


def _h_candidates_nv(h: np.ndarray, dh: np.ndarray, hq: np.ndarray, hs: np.ndarray, g_h):
    """NVFP4 counterpart of _h_candidates_mx.  Any h' of the box moves the
    tensor scale within [g_lo, g_hi] (from the box's smallest and largest
    tensor maximum) and each block scale within [s_min, s_max] (from the
    block's smallest and largest maximum at both ends of g).  For a block
    scale s, the fp32 quotient v / fp32(s g) is monotone in v and in g, so
    over the element's interval and [g_lo, g_hi] it spans the range between
    its values at the four corners, and the code takes every E2M1 grid value
    between theirs.  A dequantised value E2M1 * s * g is bilinear in the grid
    value and g, so its largest distance from the reference over that range
    is reached at a corner of (grid value, g)."""
    n, I = h.shape
    B = Q.NV_BLOCK
    hb = h.reshape(n, I // B, B)
    db = dh.reshape(n, I // B, B)
    lo = hb - db
    hi = hb + db
    amax_hi_t = float(np.max(np.abs(h) + dh)) if h.size else 0.0
    amax_lo_t = float(np.max(np.maximum(np.abs(h) - dh, 0.0))) if h.size else 0.0
    g_cands = sorted({float(Q.nv_global_scale(amax_lo_t)), float(Q.nv_global_scale(amax_hi_t)), float(g_h)})
    g_ends = (np.float32(g_cands[0]), np.float32(g_cands[-1]))
    amax_b_hi = np.max(np.maximum(np.abs(lo), np.abs(hi)), axis=-1)
    amin = np.where((lo <= 0) & (hi >= 0), 0.0, np.minimum(np.abs(lo), np.abs(hi)))
    amax_b_lo = np.max(amin, axis=-1)
    ref = Q.nv_dequant(hq, hs, g_h).reshape(n, I // B, B)
    dmax = np.zeros_like(hb)
    s_min = np.full(amax_b_lo.shape, 255, dtype=np.int64)
    s_max = np.full(amax_b_lo.shape, -1, dtype=np.int64)
    for g32 in g_ends:
        six_g = np.float32(6.0) * g32
        for ab in (amax_b_lo, amax_b_hi):
            q_s = (ab.astype(np.float32) / six_g).astype(np.float32) if six_g > 0 else np.zeros_like(ab, dtype=np.float32)
            sb = (e4m3_encode(q_s.astype(np.float64)) & 0x7F).astype(np.int64)
            s_min = np.minimum(s_min, sb)
            s_max = np.maximum(s_max, sb)
    for ds in range(0, int(np.max(s_max - s_min)) + 1 if s_max.size else 1):
        sb = np.minimum(s_min + ds, 126)
        ok = (s_min + ds) <= s_max
        sv = E4M3_TABLE[sb][..., None]
        quots = []
        for g32 in g_ends:
            d_b = (E4M3_TABLE[sb].astype(np.float32) * g32).astype(np.float32)[..., None]
            for v in (lo, hi):
                with np.errstate(divide="ignore", invalid="ignore"):
                    q = np.where(d_b > 0, v.astype(np.float32) / d_b, 0.0)
                quots.append(q.astype(np.float32).astype(np.float64))
        grid_lo = E2M1_TABLE[e2m1_encode(np.minimum.reduce(quots)).astype(np.int64)]
        grid_hi = E2M1_TABLE[e2m1_encode(np.maximum.reduce(quots)).astype(np.int64)]
        for gv in (grid_lo, grid_hi):
            for g32 in g_ends:
                d = np.where(ok[..., None], np.abs(gv * sv * float(g32) - ref), 0.0)
                dmax = np.maximum(dmax, d)
    return dmax.reshape(n, I), (s_min, s_max)


class WeightSource:
    """Oracle-side expert weights.  ``get(which, e)`` returns (codes unpacked
    [rows, K], scale bytes, tensor scale or None) for which in
    {"w13", "w2", "sh13", "sh2"}."""

    def __init__(self, fn):
        self._fn = fn
        self._cache = {}

    def get(self, which, e):
        key = (which, e)
        if key not in self._cache:
            self._cache[key] = self._fn(which, e)
        return self._cache[key]

    def drop(self, which, e):
        self._cache.pop((which, e), None)


def expert_rows(cfg, e: int, a: np.ndarray, wts: np.ndarray, weights: WeightSource,
                gamma: float = GAMMA, with_ambiguity: bool = True) -> dict:
    """The MLP of expert e (ids >= E are shared experts) for the dequantised
    activation rows a [n, H] routed to it with weights wts [n].  Returns the
    intermediates and y, the S term and the ambiguity term per row."""
    E, I, fmt = cfg.E, cfg.I, cfg.fmt
    if e < E:
        w13, w2 = weights.get("w13", e), weights.get("w2", e)
    else:
        w13, w2 = weights.get("sh13", e - E), weights.get("sh2", e - E)
    W13 = Q.dequant(w13[0], w13[1], fmt, w13[2])
    gu = a @ W13.T
    gu_abs = np.abs(a) @ np.abs(W13).T if with_ambiguity else None
    del W13
    g, u = gu[:, :I], gu[:, I:]
    h = silu(g) * u
    h32 = h.astype(np.float32).astype(np.float64)
    if fmt == "mxfp4":
        hq, hs = Q.mx_quantize(h32)
        g_h = None
    else:
        hq, hs, g_h = Q.nv_quantize(h32)
    hd = Q.dequant(hq, hs, fmt, g_h)
    W2 = Q.dequant(w2[0], w2[1], fmt, w2[2])
    y = hd @ W2.T
    W2a = np.abs(W2) if with_ambiguity else None
    Sy = np.abs(hd) @ W2a.T if with_ambiguity else None
    info = {"wt": wts, "h": h, "h32": h32, "hq": hq, "hs": hs, "g_h": g_h, "y": y, "Sy": Sy,
            "gu_abs": gu_abs}
    if with_ambiguity:
        dg = gamma * gu_abs[:, :I] + 2.0 ** -22 * np.abs(g)
        du = gamma * gu_abs[:, I:] + 2.0 ** -22 * np.abs(u)
        sg = silu(g)
        dh = (SILU_LIP * dg * (np.abs(u) + du) + np.abs(sg) * du
              + (EPS_SWIGLU + EPS_EXP_PER_G * np.abs(g)) * np.abs(h) + 2.0 ** -140)
        if fmt == "mxfp4":
            dmax, srange = _h_candidates_mx(h32, dh, hq, hs)
        else:
            dmax, srange = _h_candidates_nv(h32, dh, hq, hs, g_h)
        info.update({"dh": dh, "dmax": dmax, "scale_range": srange, "Ay": dmax @ W2a.T,
                     "n_ambiguous": int(np.count_nonzero(dmax))})
    else:
        info["Ay"] = np.zeros_like(y)
    return info


def layer_forward(cfg, x_bits_f64: np.ndarray, wr_f64: np.ndarray, bias_f32: np.ndarray,
                  weights: WeightSource, tokens=None, gamma: float = GAMMA,
                  with_ambiguity: bool = True):
    """The whole layer with routing over all T tokens; outputs for the tokens
    in ``tokens`` (default: all).  Every expert a chosen token uses is
    evaluated on all of its routed rows (NVFP4's per-expert tensor scale of h
    depends on all of them).

    x_bits_f64 / wr_f64 hold the exact values of the bf16 inputs.  Returns a
    dict with routing, quantised activations, permutation, per-expert
    intermediates, and for the chosen tokens ref / S / A [len(tokens), H]."""
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.top_k
    ns = cfg.n_shared
    fmt = cfg.fmt
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    logits, lsum = router_logits(x_bits_f64, wr_f64)
    idx, w = route(logits, bias_f32, k, cfg.n_group, cfg.topk_group, cfg.routed_scaling,
                   cfg.renormalize)
    xc, xs, gx = Q.quantize(x_bits_f64, fmt)
    counts, offsets, ptok, pslot = permute(idx, E, ns)

    need = sorted(set(int(e) for t in tokens for e in idx[t]) | set(range(E, E + ns)))
    tok_pos = {int(t): i for i, t in enumerate(tokens)}
    ref = np.zeros((len(tokens), H))
    S = np.zeros((len(tokens), H))
    A = np.zeros((len(tokens), H))
    experts = {}
    for e in need:
        rows = np.arange(offsets[e], offsets[e + 1])
        toks = ptok[rows]
        slots = pslot[rows]
        wts = w[toks, np.minimum(slots, k - 1)] if e < E else np.ones(len(rows))
        a = Q.dequant(xc[toks], xs[toks], fmt, gx)
        info = expert_rows(cfg, e, a, wts, weights, gamma, with_ambiguity)
        info.update({"rows": rows, "tok": toks, "slot": slots})
        for r in range(len(rows)):
            t = int(toks[r])
            if t in tok_pos:
                i = tok_pos[t]
                ref[i] += wts[r] * info["y"][r]
                S[i] += abs(wts[r]) * info["Sy"][r]
                A[i] += abs(wts[r]) * info["Ay"][r]
        experts[e] = info
    margins = [decision_margins(logits[t], bias_f32, k, cfg.n_group, cfg.topk_group)
               for t in range(T)]
    return {"logits": logits, "lsum": lsum, "idx": idx, "w": w, "margins": margins,
            "xc": xc, "xs": xs, "gx": gx, "counts": counts, "offsets": offsets,
            "perm_tok": ptok, "perm_slot": pslot, "experts": experts,
            "tokens": tokens, "ref": ref, "S": S, "A": A}


def token_forward(cfg, x_rows_f64: np.ndarray, wr_f64: np.ndarray, bias_f32: np.ndarray,
                  weights: WeightSource, gamma: float = GAMMA, with_ambiguity: bool = True):
    """MXFP4 only: the layer output of individual tokens x_rows [n, H].  With
    MXFP4 both quantisations (x and h) act row by row, so one token's output
    depends on its own routes alone.  Returns per-token routing, the routes'
    intermediates and ref / S / A [n, H]."""
    assert cfg.fmt == "mxfp4", "NVFP4 tensor scales couple tokens; use layer_forward"
    E, k, ns = cfg.E, cfg.top_k, cfg.n_shared
    logits, lsum = router_logits(x_rows_f64, wr_f64)
    idx, w = route(logits, bias_f32, k, cfg.n_group, cfg.topk_group, cfg.routed_scaling,
                   cfg.renormalize)
    xc, xs = Q.mx_quantize(x_rows_f64)
    n, H = x_rows_f64.shape
    ref, S, A = np.zeros((n, H)), np.zeros((n, H)), np.zeros((n, H))
    routes = []
    for i in range(n):
        a = Q.mx_dequant(xc[i:i + 1], xs[i:i + 1])
        per = []
        for j, e in enumerate(list(idx[i]) + list(range(E, E + ns))):
            wt = w[i, j] if j < k else 1.0
            info = expert_rows(cfg, int(e), a, np.array([wt]), weights, gamma, with_ambiguity)
            ref[i] += wt * info["y"][0]
            S[i] += abs(wt) * info["Sy"][0]
            A[i] += abs(wt) * info["Ay"][0]
            info["expert"] = int(e)
            per.append(info)
        routes.append(per)
    margins = [decision_margins(logits[i], bias_f32, k, cfg.n_group, cfg.topk_group) for i in range(n)]
    return {"logits": logits, "lsum": lsum, "idx": idx, "w": w, "margins": margins, "xc": xc, "xs": xs,
            "routes": routes, "ref": ref, "S": S, "A": A}


def tolerance(ref: np.ndarray, S: np.ndarray, A: np.ndarray) -> np.ndarray:
    """Per-element bound |gpu - ref| may not exceed."""
    return 2.0 ** -8 * np.abs(ref) + 1e-3 * S + A
