"""Pins of the oracle's router and permutation: brute force over expert and
group subsets, planted ties, reduction to plain top-k, stable sort."""
import itertools

import numpy as np
import pytest

import synth
from oracle import router as R
from oracle.permute import permute


def _brute_topk(c, allowed, k):
    """Best k-subset by sum of c over allowed experts; among equal sums the
    lexicographically smallest index tuple wins."""
    best = None
    for sub in itertools.combinations(np.flatnonzero(allowed), k):
        val = sum(c[list(sub)])
        if best is None or val > best[0]:
            best = (val, sub)
    return set(best[1])


def _brute_grouped(c, n_group, topk_group, k):
    E = len(c)
    gsz = E // n_group
    gscore = [sum(sorted(c[g * gsz:(g + 1) * gsz])[-2:]) for g in range(n_group)]
    best = None
    for gs in itertools.combinations(range(n_group), topk_group):
        val = sum(gscore[g] for g in gs)
        if best is None or val > best[0]:
            best = (val, gs)
    allowed = np.zeros(E, dtype=bool)
    for g in best[1]:
        allowed[g * gsz:(g + 1) * gsz] = True
    return _brute_topk(c, allowed, k)


def test_tiny_config_brute_force():
    cfg = synth.configs()["tiny"]
    x = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg))
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    b = synth.gen_bias_f32(cfg)
    logits, _ = R.router_logits(x, wr)
    idx, w = R.route(logits, b, cfg.top_k)
    for t in range(cfg.T):
        s = 1 / (1 + np.exp(-logits[t]))
        c = s + b
        assert set(idx[t]) == _brute_topk(c, np.ones(cfg.E, bool), cfg.top_k)
        assert np.isclose(w[t].sum(), cfg.routed_scaling)
        np.testing.assert_allclose(w[t], s[idx[t]] / s[idx[t]].sum() * cfg.routed_scaling, rtol=0, atol=0)


def test_grouped_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(40):
        logits = rng.standard_normal(16) * 2
        bias = (rng.standard_normal(16) * 0.1).astype(np.float32)
        idx, w, info = R.route_token(logits, bias, 4, 4, 2, 2.5, 1)
        assert set(idx) == _brute_grouped(info["c"], 4, 2, 4)
        assert np.isclose(w.sum(), 2.5)


def test_planted_ties_pick_lower_index():
    logits = np.zeros(8)
    bias = np.zeros(8, dtype=np.float32)
    idx, _, _ = R.route_token(logits, bias, 3, 1, 1, 1.0, 1)
    assert idx.tolist() == [0, 1, 2]
    # identical groups: the lower group wins, then lower experts inside it
    logits = np.tile(np.array([1.0, 0.5, 0.2, 0.1]), 4)
    idx, _, _ = R.route_token(logits, bias.repeat(2), 2, 4, 1, 1.0, 1)
    assert idx.tolist() == [0, 1]
    logits = np.array([0.0, 1.0, 1.0, 0.5])
    idx, _, _ = R.route_token(logits, np.zeros(4, np.float32), 2, 1, 1, 1.0, 1)
    assert idx.tolist() == [1, 2]


def test_single_group_is_plain_topk():
    rng = np.random.default_rng(12)
    logits = rng.standard_normal((32, 64))
    bias = (rng.standard_normal(64) * 0.1).astype(np.float32)
    idx, w = R.route(logits, bias, 6, 1, 1, 1.0, 1)
    c = 1 / (1 + np.exp(-logits)) + bias
    ref = np.argsort(-c, axis=1, kind="stable")[:, :6]
    assert np.array_equal(idx, ref)


def test_no_renormalize():
    logits = np.array([2.0, 1.0, 0.0, -1.0])
    idx, w, _ = R.route_token(logits, np.zeros(4, np.float32), 2, 1, 1, 3.0, 0)
    np.testing.assert_allclose(w, 3.0 / (1 + np.exp(-logits[:2])), rtol=1e-15)


def test_logits_match_library_matmul():
    import torch
    rng = np.random.default_rng(13)
    x = rng.standard_normal((5, 64))
    wr = rng.standard_normal((7, 64))
    l, s = R.router_logits(x, wr)
    ref = (torch.tensor(x) @ torch.tensor(wr).T).numpy()
    np.testing.assert_allclose(l, ref, rtol=1e-13, atol=1e-13)
    assert np.all(s >= np.abs(l))


def test_permutation_is_stable_sort():
    rng = np.random.default_rng(14)
    T, k, E = 50, 4, 12
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    counts, offsets, ptok, pslot = permute(idx, E, n_shared=1)
    flat_e = idx.reshape(-1)
    order = np.argsort(flat_e, kind="stable")
    assert np.array_equal(ptok[:T * k], order // k)
    assert np.array_equal(pslot[:T * k], order % k)
    assert np.array_equal(counts[:E], np.bincount(flat_e, minlength=E))
    assert counts[E] == T and np.array_equal(ptok[T * k:], np.arange(T))
    assert np.all(pslot[T * k:] == k)
    assert offsets[-1] == T * (k + 1) and np.all(np.diff(offsets) >= 0)
    # bijection onto the routes
    pairs = set(zip(ptok.tolist(), pslot.tolist()))
    assert len(pairs) == T * (k + 1)


# ------------------------------------------------------------------ decision margins
def _select_from_c(c, n_group, topk_group, k, combos_cache={}):
    """Brute force on corrected scores c: the kept groups (best topk_group-
    subset by the sum of group scores) and the best k-subset of their
    experts by the sum of c.  Returns (frozenset of experts, frozenset of groups)."""
    E = len(c)
    allowed = np.ones(E, dtype=bool)
    groups = frozenset()
    if n_group > 1:
        gsz = E // n_group
        gscore = np.sort(c.reshape(n_group, gsz), axis=1)[:, -2:].sum(axis=1)
        key = ("g", n_group, topk_group)
        if key not in combos_cache:
            combos_cache[key] = np.array(list(itertools.combinations(range(n_group), topk_group)))
        gc = combos_cache[key]
        best = gc[int(np.argmax(gscore[gc].sum(axis=1)))]
        groups = frozenset(best.tolist())
        allowed = np.zeros(E, dtype=bool)
        for g in best:
            allowed[g * gsz:(g + 1) * gsz] = True
    cand = np.flatnonzero(allowed)
    key = ("e", len(cand), k)
    if key not in combos_cache:
        combos_cache[key] = np.array(list(itertools.combinations(range(len(cand)), k)))
    ec = combos_cache[key]
    best = cand[ec[int(np.argmax(c[cand][ec].sum(axis=1)))]]
    return frozenset(best.tolist()), groups


@pytest.mark.parametrize("E,n_group,topk_group,k", [(8, 1, 1, 2), (8, 1, 1, 5), (12, 3, 2, 3), (16, 8, 3, 4),
                                                    (16, 4, 1, 2)])
def test_decision_margins_against_brute_force(E, n_group, topk_group, k):
    """The margins (em, gm) decide a token's selection: every change of the
    corrected scores by less than min(em / 2, gm / 4) in each element keeps
    the selected experts (brute force over subsets on random and corner
    perturbations), and a change of just over em / 2 (two experts) or gm / 4
    (every expert of two groups) changes the experts or the kept groups."""
    rng = np.random.default_rng(100 + E + 7 * k + n_group)
    for trial in range(12):
        logits = rng.standard_normal(E) * 1.5
        bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
        idx, _, info = R.route_token(logits, bias, k, n_group, topk_group, 1.0, 1)
        c = info["c"]
        em, gm = R.decision_margins(logits, bias, k, n_group, topk_group)
        sel0, grp0 = _select_from_c(c, n_group, topk_group, k)
        assert sel0 == frozenset(idx.tolist())
        eps = min(em / 2, gm / 4)
        assert np.isfinite(eps) and eps > 0
        for p in range(300):
            d = rng.uniform(-1, 1, E) if p % 2 else rng.choice([-1.0, 1.0], E)
            sel, grp = _select_from_c(c + 0.999 * eps * d, n_group, topk_group, k)
            assert sel == sel0 and grp == grp0, (trial, p)
        # just over em / 2: the k-th kept expert and the next one swap
        order = info["order"]
        d = np.zeros(E)
        d[order[k - 1]], d[order[k]] = -1.0, 1.0
        sel, grp = _select_from_c(c + 1.001 * (em / 2) * d, n_group, topk_group, k)
        assert sel != sel0 or grp != grp0
        if n_group > 1 and topk_group < n_group:
            # just over gm / 4: the last kept group and the best dropped one swap
            gsz = E // n_group
            gorder = np.lexsort((np.arange(n_group), -info["gscore"]))
            g_in, g_out = gorder[topk_group - 1], gorder[topk_group]
            d = np.zeros(E)
            d[g_in * gsz:(g_in + 1) * gsz] = -1.0  # the whole group moves: its top two stay its top two
            d[g_out * gsz:(g_out + 1) * gsz] = 1.0
            sel, grp = _select_from_c(c + 1.001 * (gm / 4) * d, n_group, topk_group, k)
            assert grp != grp0


# ------------------------------------------------------------------ fp32 selection step
def _f32(v):
    return np.asarray(v, dtype=np.float32)


def test_select_fp32_brute_force_on_fp32_scores():
    """The fp32 selection equals the brute-force best subsets of the fp32
    corrected scores c = fp32(s + b) (plain and grouped), lists the experts in
    descending c, and forms the weights by fp32 steps."""
    rng = np.random.default_rng(21)
    for E, n_group, topk_group, k in [(8, 1, 1, 3), (16, 4, 2, 4), (12, 6, 3, 2)]:
        for trial in range(30):
            s = _f32(1 / (1 + np.exp(-rng.standard_normal(E) * 2)))
            b = _f32(rng.standard_normal(E) * 0.1)
            idx, w = R.select_fp32(s, b, k, n_group, topk_group, 2.827, 1)
            c = (s + b).astype(np.float32).astype(np.float64)
            sel, _ = _select_from_c(c, n_group, topk_group, k)
            assert set(idx.tolist()) == sel
            assert np.all(np.diff(c[idx]) <= 0)
            tot = np.float32(0)
            for e in idx:
                tot = np.float32(tot + s[e])
            assert w.dtype == np.float32
            assert np.array_equal(w, _f32([np.float32(s[e] / tot) * np.float32(2.827) for e in idx]))
            # without renormalisation: fp32(s * scaling)
            _, w0 = R.select_fp32(s, b, k, n_group, topk_group, 2.5, 0)
            assert np.array_equal(w0, (s[idx] * np.float32(2.5)).astype(np.float32))


def test_select_fp32_agrees_with_fp64_route_away_from_ties():
    """On scores rounded once from the float64 sigmoid, with every decision
    gap far above fp32 rounding, the fp32 step picks what route_token picks
    (same order) and the weights agree to fp32 rounding."""
    rng = np.random.default_rng(22)
    n = 0
    for trial in range(200):
        logits = rng.standard_normal(32) * 2
        bias = _f32(rng.standard_normal(32) * 0.1)
        em, gm = R.decision_margins(logits, bias, 6, 4, 2)
        if min(em, gm) < 1e-5:
            continue
        n += 1
        idx64, w64, _ = R.route_token(logits, bias, 6, 4, 2, 2.827, 1)
        idx32, w32 = R.select_fp32(_f32(R.sigmoid_f64(logits)), bias, 6, 4, 2, 2.827, 1)
        assert np.array_equal(idx32, idx64)
        np.testing.assert_allclose(w32, w64, rtol=4e-7)
    assert n > 150


def test_select_fp32_planted_ties():
    """Equal fp32 scores and biases: the lower expert, and the lower group."""
    s = _f32([0.5] * 8)
    b = _f32([0.0] * 8)
    idx, w = R.select_fp32(s, b, 3, 1, 1, 1.0, 1)
    assert idx.tolist() == [0, 1, 2]
    assert np.array_equal(w, _f32([np.float32(0.5) / np.float32(1.5)] * 3))
    # two identical groups at the top: the lower group is kept
    s = _f32([0.9, 0.2, 0.1, 0.9, 0.2, 0.1, 0.3, 0.3, 0.3])
    idx, _ = R.select_fp32(s, np.zeros(9, np.float32), 2, 3, 1, 1.0, 1)
    assert idx.tolist() == [0, 1]
    # a tie made by the bias: equal corrected scores from different scores
    s = _f32([0.25, 0.5, 0.75, 0.125])
    b = _f32([0.5, 0.25, 0.0, 0.0])
    idx, _ = R.select_fp32(s, b, 2, 1, 1, 1.0, 0)
    assert idx.tolist() == [0, 1]
    # fp32 rounding of s + b decides: 1 + 2^-24 rounds to 1 (ties to even),
    # a tie with expert 0 that the lower index wins, while in float64 expert
    # 1 would rank first
    s = _f32([1.0, 1.0])
    b = _f32([0.0, 2.0 ** -24])
    assert R.select_fp32(s, b, 1, 1, 1, 1.0, 1)[0].tolist() == [0]
    assert np.argmax(s.astype(np.float64) + b.astype(np.float64)) == 1
