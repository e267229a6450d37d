"""Expert histogram, prefix sum and stable token permutation (oracle; test only).

The layer groups its routes by expert before the grouped GEMMs (the two-stage
fused MoE of "Serve Kimi-K2.5-MXFP4 on MI355X with ATOM", section "Stage D:
MXFP4 Fused MoE"; expert tiles in "Inside the Kimi K3 optimization effort",
technical note on expert routing).  The pages do not fix the order inside an
expert; the reading used here is a stable counting sort: routes are visited
token by token (slot j within a token), so inside one expert tokens ascend.
Shared experts take ids E .. E+n_shared-1 and receive every token.
"""
from __future__ import annotations

import numpy as np


def permute(idx: np.ndarray, E: int, n_shared: int = 0):
    """idx [T, k] expert ids.  Returns (counts [E+ns], offsets [E+ns+1],
    perm_tok [R], perm_slot [R]) with R = T*k + T*ns: sorted position p holds
    route (perm_tok[p], perm_slot[p]); slot k+s is shared expert s."""
    T, k = idx.shape
    n_exp = E + n_shared
    counts = np.zeros(n_exp, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    counts[E:] = T
    offsets = np.zeros(n_exp + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    R = int(offsets[-1])
    perm_tok = np.zeros(R, dtype=np.int64)
    perm_slot = np.zeros(R, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            perm_tok[fill[e]] = t
            perm_slot[fill[e]] = j
            fill[e] += 1
        for s in range(n_shared):
            perm_tok[fill[E + s]] = t
            perm_slot[fill[E + s]] = k + s
            fill[E + s] += 1
    return counts, offsets, perm_tok, perm_slot
