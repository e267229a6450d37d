"""NVFP4 emulation mode of the MoE layer (FP64 oracle; test infrastructure
only).

"Serving NVFP4 models on AMD Instinct MI355 accelerators", sections "Weight
Dequantization and Activation QDQ" and "Memory Management": NVFP4 weights are
dequantised to BF16 at GEMM time (for MoE, only the dispatched experts), the
input activations pass through an NVFP4 quantise-dequantise round trip, and
both enter the matrix multiply as BF16 tensors with FP32 accumulation.

The page does not say how the dequantised value is rounded to BF16.  The
reading used here: the NVFP4 value as this library's NVFP4 reading forms it
-- d_b = fp32(E4M3(s_b) * g), v = fp32(E2M1(q) * d_b) -- rounded to BF16 by
round-to-nearest-even.  The same rule applies to the weights (their own
tensor scale per expert and weight tensor), to x (one tensor scale per
call) and to the intermediate h (one tensor scale per expert, over the
expert's fp32 h), exactly as the native NVFP4 layer quantises them.

Per route (token t, expert e, routing weight w):

    a       = bf16(qdq(x[t]))
    [g | u] = a . bf16(dq(W13[e]))^T             (fp32 accumulation on the GPU)
    h       = silu(g) * u, rounded to fp32
    h_hat   = bf16(qdq(h))
    y       = h_hat . bf16(dq(W2[e]))^T
    out[t] += w * y

Tolerance as for the native layer, with the allowance A widened by the BF16
rounding of a flipped element.
"""
from __future__ import annotations

import numpy as np

from . import quant as Q
from .formats import E2M1_TABLE, E4M3_TABLE
from .moe import EPS_EXP_PER_G, EPS_SWIGLU, GAMMA, SILU_LIP, _h_candidates_nv, silu
from .permute import permute
from .router import decision_margins, route, router_logits


def bf16_rne(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even of fp32 values to bf16, returned as float64."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32).astype(np.float64)


def nv_dequant_bf16(codes: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """BF16 values of unpacked NVFP4 codes [..., K] with E4M3 scale bytes
    [..., K/16] and tensor scale g: bf16(fp32(E2M1(q) * fp32(E4M3(s) * g)))."""
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1]
    d = (E4M3_TABLE[np.asarray(scales, dtype=np.uint8)].astype(np.float32) * np.float32(g)).astype(np.float32)
    q = E2M1_TABLE[codes].astype(np.float32).reshape(codes.shape[:-1] + (K // Q.NV_BLOCK, Q.NV_BLOCK))
    v = (q * d[..., None]).astype(np.float32).reshape(codes.shape)
    return bf16_rne(v)


def emulated_expert_rows(cfg, e: int, a: np.ndarray, wts: np.ndarray, weights, gamma: float = GAMMA,
                         with_ambiguity: bool = True) -> dict:
    """The emulated MLP of expert e for BF16 activation rows a [n, H].
    ``weights`` yields the native NVFP4 tensors (codes, scale bytes, g)."""
    E, I = cfg.E, cfg.I
    w13 = weights.get("w13", e) if e < E else weights.get("sh13", e - E)
    w2 = weights.get("w2", e) if e < E else weights.get("sh2", e - E)
    W13 = nv_dequant_bf16(*w13)
    gu = a @ W13.T
    g, u = gu[:, :I], gu[:, I:]
    h = silu(g) * u
    h32 = h.astype(np.float32).astype(np.float64)
    hq, hs, g_h = Q.nv_quantize(h32)
    hd = nv_dequant_bf16(hq, hs, g_h)
    W2 = nv_dequant_bf16(*w2)
    y = hd @ W2.T
    info = {"wt": wts, "h": h, "h32": h32, "hq": hq, "hs": hs, "g_h": g_h, "hd": hd, "y": y}
    W2a = np.abs(W2)
    info["Sy"] = np.abs(hd) @ W2a.T
    if with_ambiguity:
        gu_abs = np.abs(a) @ np.abs(W13).T
        dg = gamma * gu_abs[:, :I] + 2.0 ** -22 * np.abs(g)
        du = gamma * gu_abs[:, I:] + 2.0 ** -22 * np.abs(u)
        dh = (SILU_LIP * dg * (np.abs(u) + du) + np.abs(silu(g)) * du
              + (EPS_SWIGLU + EPS_EXP_PER_G * np.abs(g)) * np.abs(h) + 2.0 ** -140)
        dmax, srange = _h_candidates_nv(h32, dh, hq, hs, g_h)
        # a flipped element is also rounded to bf16 (at most 2**-9 of its size)
        dmax = np.where(dmax > 0, dmax * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(hd), 0.0)
        info.update({"dh": dh, "dmax": dmax, "scale_range": srange, "Ay": dmax @ W2a.T,
                     "n_ambiguous": int(np.count_nonzero(dmax))})
    else:
        info["Ay"] = np.zeros_like(y)
    return info


def emulated_layer_forward(cfg, x_bits_f64: np.ndarray, wr_f64: np.ndarray, bias_f32: np.ndarray, weights,
                           tokens=None, gamma: float = GAMMA, with_ambiguity: bool = True):
    """The emulated layer over all T tokens (the tensor scales of x and of
    each expert's h couple tokens); outputs for ``tokens`` (default all)."""
    T, H, E, k, ns = cfg.T, cfg.H, cfg.E, cfg.top_k, cfg.n_shared
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    logits, lsum = router_logits(x_bits_f64, wr_f64)
    idx, w = route(logits, bias_f32, k, cfg.n_group, cfg.topk_group, cfg.routed_scaling, cfg.renormalize)
    xc, xs, gx = Q.nv_quantize(x_bits_f64)
    a_all = nv_dequant_bf16(xc, xs, gx)
    counts, offsets, ptok, pslot = permute(idx, E, ns)
    need = sorted(set(int(e) for t in tokens for e in idx[t]) | set(range(E, E + ns)))
    pos = {int(t): i for i, t in enumerate(tokens)}
    ref, S, A = (np.zeros((len(tokens), H)) for _ in range(3))
    experts = {}
    for e in need:
        rows = np.arange(offsets[e], offsets[e + 1])
        toks, slots = ptok[rows], pslot[rows]
        wts = w[toks, np.minimum(slots, k - 1)] if e < E else np.ones(len(rows))
        info = emulated_expert_rows(cfg, e, a_all[toks], wts, weights, gamma, with_ambiguity)
        info.update({"rows": rows, "tok": toks, "slot": slots})
        for r, t in enumerate(toks):
            if int(t) in pos:
                i = pos[int(t)]
                ref[i] += wts[r] * info["y"][r]
                S[i] += abs(wts[r]) * info["Sy"][r]
                A[i] += abs(wts[r]) * info["Ay"][r]
        experts[e] = info
    margins = [decision_margins(logits[t], bias_f32, k, cfg.n_group, cfg.topk_group) for t in range(T)]
    return {"logits": logits, "lsum": lsum, "idx": idx, "w": w, "margins": margins, "xc": xc, "xs": xs, "gx": gx,
            "a": a_all, "experts": experts, "tokens": tokens, "ref": ref, "S": S, "A": A}
