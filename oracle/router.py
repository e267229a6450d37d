"""Sigmoid + correction-bias grouped top-k routing (FP64 oracle; test only).

The pages name the router ("Kimi-K2.7-Code on Gaudi 2", section "What was
built": the grouped top-k router, sigmoid scoring with correction bias) and
keep it in high precision ("Serving NVFP4 models on AMD Instinct MI355
accelerators", section "Layer Selection"; "Serve Kimi-K2.5-MXFP4 on MI355X with
ATOM", section "Checkpoint Layout and Quantization Metadata").  The steps,
in the DeepSeek-V3 form the pages refer to:

    l[t, e] = sum_h x[t, h] * Wr[e, h]          (bf16 inputs, exact products)
    s       = 1 / (1 + exp(-l))
    c       = s + bias[e]
    group score = sum of the two largest c in the group; keep the topk_group
                  groups with the largest scores (n_group = 1: keep all)
    idx     = the top_k experts by c among the kept groups
    w_j     = s[idx_j] / sum_j s[idx_j] * routed_scaling   (renormalize = 1)
              s[idx_j] * routed_scaling                     (renormalize = 0)

Ties go to the lower group index and the lower expert index.  idx is listed
in descending c.  Everything is float64.
"""
from __future__ import annotations

import numpy as np


def router_logits(x: np.ndarray, wr: np.ndarray):
    """x [T, H] and Wr [E, H] as exact float64 values.  Returns (logits [T, E],
    sum_abs [T, E] = sum_h |x * Wr|, the scale of any accumulation error)."""
    return x @ wr.T, np.abs(x) @ np.abs(wr).T


def _top_order(vals: np.ndarray) -> np.ndarray:
    """Indices sorted by descending value, ties by ascending index."""
    return np.lexsort((np.arange(len(vals)), -vals))


def route_token(logit: np.ndarray, bias: np.ndarray, top_k: int, n_group: int,
                topk_group: int, routed_scaling: float, renormalize: int):
    """Route one token.  Returns (idx [top_k] int64, w [top_k] float64, info)."""
    E = logit.shape[0]
    s = 1.0 / (1.0 + np.exp(-logit))
    c = s + bias.astype(np.float64)
    allowed = np.ones(E, dtype=bool)
    gscore = None
    if n_group > 1:
        gsz = E // n_group
        assert gsz >= 2, "a group's score sums its two largest corrected scores"
        cg = c.reshape(n_group, gsz)
        top2 = np.sort(cg, axis=1)[:, -2:]
        gscore = top2[:, 0] + top2[:, 1]
        keep = _top_order(gscore)[:topk_group]
        allowed = np.zeros(E, dtype=bool)
        for g in keep:
            allowed[g * gsz:(g + 1) * gsz] = True
    cand = np.where(allowed)[0]
    order = cand[_top_order(c[cand])]
    idx = order[:top_k]
    w = s[idx].copy()
    if renormalize:
        w = w / np.sum(w)
    w = w * routed_scaling
    info = {"s": s, "c": c, "allowed": allowed, "gscore": gscore, "order": order}
    return idx.astype(np.int64), w, info


def route(logits: np.ndarray, bias: np.ndarray, top_k: int, n_group: int = 1,
          topk_group: int = 1, routed_scaling: float = 1.0, renormalize: int = 1):
    """Route all tokens.  Returns (idx [T, k] int64, w [T, k] float64)."""
    T = logits.shape[0]
    idx = np.zeros((T, top_k), dtype=np.int64)
    w = np.zeros((T, top_k), dtype=np.float64)
    for t in range(T):
        idx[t], w[t], _ = route_token(logits[t], bias, top_k, n_group, topk_group,
                                      routed_scaling, renormalize)
    return idx, w


def decision_margins(logit: np.ndarray, bias: np.ndarray, top_k: int, n_group: int,
                     topk_group: int):
    """Gaps that decide one token's selection: the gap between the k-th and
    (k+1)-th kept expert by c and, for grouped routing, between the
    topk_group-th and next group score.  Used to tell which tokens a tiny
    change of the logits could route differently."""
    idx, _, info = route_token(logit, bias, top_k, n_group, topk_group, 1.0, 1)
    c = info["c"]
    order = info["order"]
    em = c[order[top_k - 1]] - c[order[top_k]] if len(order) > top_k else np.inf
    gm = np.inf
    if n_group > 1 and topk_group < n_group:
        gs = np.sort(info["gscore"])[::-1]
        gm = gs[topk_group - 1] - gs[topk_group]
    return em, gm


def select_fp32(s32: np.ndarray, bias32: np.ndarray, top_k: int, n_group: int, topk_group: int,
                routed_scaling: float, renormalize: int):
    """The selection step of one token taken in fp32, from fp32 sigmoid
    scores: the integer decisions of route_token (group choice, top-k) made on
    fp32 values, as a router that keeps its scores in fp32 makes them.  Each
    step is one correctly rounded fp32 operation:

        c           = fp32(s + bias)
        group score = fp32(largest c + second largest c)   (per group)
        keep the topk_group groups with the largest scores (ties: lower group)
        idx         = the top_k kept experts by descending c (ties: lower index)
        tot         = fp32 running sum of s[idx_0], s[idx_1], ... from 0
        w_j         = fp32(fp32(s[idx_j] / tot) * routed_scaling)   (renormalize)
                      fp32(s[idx_j] * routed_scaling)                (otherwise)

    Returns (idx [top_k] int64, w [top_k] float32)."""
    s = np.asarray(s32, dtype=np.float32)
    b = np.asarray(bias32, dtype=np.float32)
    E = s.shape[0]
    c = (s + b).astype(np.float32)
    allowed = np.ones(E, dtype=bool)
    if n_group > 1:
        gsz = E // n_group
        assert gsz >= 2, "a group's score sums its two largest corrected scores"
        top2 = np.sort(c.reshape(n_group, gsz), axis=1)[:, -2:]
        gscore = (top2[:, 1] + top2[:, 0]).astype(np.float32)
        allowed = np.zeros(E, dtype=bool)
        for g in _top_order(gscore.astype(np.float64))[:topk_group]:
            allowed[g * gsz:(g + 1) * gsz] = True
    cand = np.where(allowed)[0]
    idx = cand[_top_order(c[cand].astype(np.float64))][:top_k]
    tot = np.float32(0.0)
    for e in idx:
        tot = np.float32(tot + s[e])
    scal = np.float32(routed_scaling)
    if renormalize:
        w = np.array([np.float32(np.float32(s[e] / tot) * scal) for e in idx], dtype=np.float32)
    else:
        w = np.array([np.float32(s[e] * scal) for e in idx], dtype=np.float32)
    return idx.astype(np.int64), w


def sigmoid_f64(logit: np.ndarray) -> np.ndarray:
    """1 / (1 + exp(-l)) in float64 (the score the fp32 router approximates)."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-np.asarray(logit, dtype=np.float64)))
