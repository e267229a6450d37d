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
