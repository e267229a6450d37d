"""GPU parity of fp4moe_route and fp4moe_forward against the FP64 oracle.

Staged, so that a mismatch is attributed to its step:
  1. router numerics: the GPU's logits within 2^-16 sum|x * Wr| of the exact
     ones, its fp32 sigmoid scores within 2^-21 (relative) of the float64
     sigmoid of those logits;
  2. selection, bit-exact: the oracle's selection step taken in fp32 on the
     GPU's own scores gives the GPU's experts in the GPU's order and its
     routing weights bit for bit, on every token;
  3. routing against the pure oracle: equal expert lists (order included)
     wherever the oracle's decision margins clear the logit error bound;
     elsewhere the GPU's choice must be one the bound admits;
  4. permutation: counts, slot layout, ascending tokens inside each expert,
     and route <-> row consistency (unique given the routing);
  5. quantised activations: bit-exact codes and scale bytes per route;
  6. the intermediate: h before quantisation within its error bound of the
     oracle's; its quantised form bit-exact to the oracle's quantiser
     replayed on the GPU's own h (NVFP4: with the GPU's per-expert tensor
     scale, itself checked against the GPU's h); and equal to the oracle's
     own quantisation wherever no other one is admissible;
  7. the output: within 2^-8 |ref'| + 1e-3 S' of the oracle's down
     projection and combine replayed on the GPU's quantised intermediate and
     routing weights, with no allowance for flips; and within 2^-8 |ref| +
     1e-3 S + A of the pure oracle wherever the routing agrees.
Small configurations run the whole oracle; the full-size workloads, in the
launch configuration the benchmark times, check routing on every token and
the expert math on sampled tokens."""
from dataclasses import replace

import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import formats as F
from oracle import inputs as OI
from oracle import moe as M
from oracle import quant as Q
from oracle import router as R

from gpu_util import dims_of, ensure_built, katoms_padded, read_tiled_scales, torch_cuda

pytestmark = pytest.mark.gpu

LOGIT_GAMMA = 2.0 ** -16  # |logit_gpu - logit| <= LOGIT_GAMMA * sum |x * Wr|
# |s_gpu - sigmoid(l_gpu)| <= SCORE_REL * sigmoid(l_gpu) + 2^-126: the fp32
# sigmoid 1 / (1 + e^-l) with CUDA's expf (at most 2 units in the last place)
# and two correctly rounded steps is within 1.5 * 2^-22 relative
SCORE_REL = 2.0 ** -21


def _cfg(base, **kw):
    return replace(synth.configs()[base], **kw) if kw else synth.configs()[base]


SMALL = {
    "tiny": _cfg("tiny"),
    "tiny_T1": _cfg("tiny", T=1),
    "ragged_shared": _cfg("tiny", name="ragged_shared", T=37, H=512, I=256, E=16, top_k=4, n_shared=1),
    # few-token fused front end: a ragged expert group (24 = 16 + 8), three
    # 256-column pieces per split, a shared expert; then a 3-CTA cluster
    "front_T16_shared": _cfg("tiny", name="front_T16_shared", T=16, H=768, I=256, E=24, top_k=4, n_shared=1),
    "front_cluster3": _cfg("tiny", name="front_cluster3", T=9, H=2304, I=256, E=40, top_k=3),
    "wide_padK": _cfg("tiny", name="wide_padK", T=300, H=1024, I=384, E=8, top_k=2, routed_scaling=2.827),
    # >= 80 routes per expert: the down GEMM's units cover two 112-token
    # slots (full pairs and single-slot remainders)
    "paired_padK": _cfg("tiny", name="paired_padK", T=600, H=1024, I=384, E=4, top_k=2, routed_scaling=2.827),
    # paired slots on CTA pairs (256-row units) with a shared expert (paired
    # slots on single CTAs: the 128-column blocks of the column-block test)
    "pair_shared": _cfg("tiny", name="pair_shared", T=700, H=768, I=256, E=6, top_k=2, n_shared=1),
    "nv_grouped": _cfg("deepseek_nvfp4", name="nv_grouped", T=64, H=512, I=256, E=32, top_k=4, n_group=4,
                       topk_group=2),
    "nv_wide_padK": _cfg("deepseek_nvfp4", name="nv_wide_padK", T=200, H=256, I=128, E=4, top_k=2, n_group=2,
                         topk_group=1, n_shared=1),
}


class DeviceRun:
    """One forward on the GPU plus host copies of its intermediates."""

    def __init__(self, cfg, h_debug=True, packed=True, x=None, layer=None, cta_pair=False):
        torch = torch_cuda()
        ensure_built()
        from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
        self.torch = torch
        self.cfg = cfg
        layer = layer if layer is not None else MoELayer.synthetic(cfg, packed=packed)
        x = layer.synthetic_x() if x is None else x
        L = layer.layout
        self.L = L
        dbg = fm.Debug()
        dbg.down_cta_pair = 1 if cta_pair else 0
        h_pre = None
        if h_debug:
            h_pre = torch.zeros((L.rows_cap, cfg.I), dtype=torch.float32, device="cuda")
            dbg.h_pre = h_pre.data_ptr()
        logits = torch.full((cfg.T, cfg.E), float("nan"), dtype=torch.float32, device="cuda")
        scores = torch.full((cfg.T, cfg.E), float("nan"), dtype=torch.float32, device="cuda")
        dbg.logits, dbg.scores = logits.data_ptr(), scores.data_ptr()
        out = layer.forward(x, debug=dbg)
        torch.cuda.synchronize()
        self.status = fm.get_status(layer.ws.data_ptr())
        self.logits = logits.cpu().numpy()
        self.scores = scores.cpu().numpy()
        T, k, ns = cfg.T, cfg.top_k, cfg.n_shared
        rpt = k + ns
        ws = layer.ws
        self.x_bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
        self.out = synth.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        i32 = lambda off, n: ws[off:off + 4 * n].view(torch.int32).cpu().numpy()
        f32 = lambda off, n: ws[off:off + 4 * n].view(torch.float32).cpu().numpy()
        self.idx = i32(L.topk_idx, T * k).reshape(T, k)
        self.w = f32(L.topk_w, T * k).reshape(T, k)
        self.count = i32(L.expert_count, cfg.E + ns)
        self.slot = i32(L.expert_slot, cfg.E + ns)
        self.route_row = i32(L.route_row, T * rpt).reshape(T, rpt)
        self.row_tok = i32(L.row_tok, L.rows_cap)
        self.row_w = f32(L.row_w, L.rows_cap)
        self.rows = self.route_row.reshape(-1)
        nv = cfg.fmt == "nvfp4"
        self.nv = nv
        # quantised x sits in the route rows, or (few-token path) in token rows
        xrows = np.repeat(np.arange(T), rpt) if L.x_by_token else self.rows
        xq = ws[L.xq:L.xq + L.rows_cap * cfg.H // 2].view(L.rows_cap, cfg.H // 2)
        self.xq = xq[torch.from_numpy(xrows).long().cuda()].cpu().numpy().reshape(T, rpt, cfg.H // 2)
        blk = 16 if nv else 32
        slots = L.rows_cap // 128
        xsf = ws[L.xsf:L.xsf + slots * katoms_padded(cfg.H, nv) * 512].cpu().numpy()
        self.xs = read_tiled_scales(xsf, xrows, cfg.H // blk, katoms_padded(cfg.H, nv)).reshape(T, rpt, -1)
        hq = ws[L.hq:L.hq + L.rows_cap * cfg.I // 2].view(L.rows_cap, cfg.I // 2)
        self.hq = hq[torch.from_numpy(self.rows).long().cuda()].cpu().numpy().reshape(T, rpt, cfg.I // 2)
        hsf = ws[L.hsf:L.hsf + slots * katoms_padded(cfg.I, nv) * 512].cpu().numpy()
        self.hs = read_tiled_scales(hsf, self.rows, cfg.I // blk, katoms_padded(cfg.I, nv)).reshape(T, rpt, -1)
        self.h = h_pre[torch.from_numpy(self.rows).long().cuda()].cpu().numpy().reshape(T, rpt, cfg.I) \
            if h_debug else None
        g = ws[L.gscale:L.gscale + 4 * (2 + cfg.E + ns)].view(torch.float32).cpu().numpy()
        self.gx, self.gh = g[0], g[2:]
        self.layer = layer
        del out, h_pre

    def expert_of(self, t, j):
        """Expert of route (t, j): the j-th routed expert, or a shared one."""
        return int(self.idx[t, j]) if j < self.cfg.top_k else self.cfg.E + j - self.cfg.top_k


# ------------------------------------------------------------------ routing checks
def _score_bound(cfg, lsum_row):
    """Largest error of a corrected score c = s + bias the logit bound allows
    (sigmoid slope <= 1/4), plus the fp32 sigmoid's and the fp32 add's."""
    return 0.25 * LOGIT_GAMMA * np.max(lsum_row) + 2 * SCORE_REL + 2.0 ** -22


def check_router_numerics(run, cfg, exact_logits, lsum, tokens=None):
    """The GPU's logits and scores (debug outputs) against the exact logits."""
    tokens = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    gl = run.logits[tokens].astype(np.float64)
    assert np.all(np.abs(gl - exact_logits) <= LOGIT_GAMMA * lsum), "router logits outside their bound"
    sg = R.sigmoid_f64(gl)
    err = np.abs(run.scores[tokens].astype(np.float64) - sg)
    assert np.all(err <= SCORE_REL * sg + 2.0 ** -126), float(np.max(err / sg))


def check_selection_replay(run, cfg, bias, tokens=None):
    """Bit-exact selection: the oracle's fp32 selection step on the GPU's
    scores yields the GPU's experts (order included) and weights."""
    tokens = range(cfg.T) if tokens is None else tokens
    for t in tokens:
        idx, w = R.select_fp32(run.scores[t], bias, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.routed_scaling,
                               cfg.renormalize)
        assert np.array_equal(run.idx[t], idx), (t, run.idx[t], idx)
        assert np.array_equal(run.w[t], w), (t, run.w[t], w)


def _admissible(cfg, c64, sel, delta):
    """Whether experts `sel` are a selection some corrected scores within
    delta of c64 (per element) make: each chosen expert's group is within
    4 delta of the last kept group's score, and each chosen expert within
    2 delta of the best one left out (among those groups)."""
    E = cfg.E
    allowed = np.ones(E, dtype=bool)
    if cfg.n_group > 1:
        gsz = E // cfg.n_group
        gs = np.sort(c64.reshape(cfg.n_group, gsz), axis=1)[:, -2:].sum(axis=1)
        cut = np.sort(gs)[::-1][cfg.topk_group - 1]
        for e in sel:
            if gs[e // gsz] < cut - 4 * delta:
                return False
        allowed = np.repeat(gs >= cut - 4 * delta, gsz)
    out = np.setdiff1d(np.flatnonzero(allowed), sel)
    return out.size == 0 or np.min(c64[sel]) >= np.max(c64[out]) - 2 * delta


def check_routing(run, cfg, orc, tokens):
    """Routing of the chosen tokens against the pure oracle.  Returns the
    tokens whose selection the logit bound leaves open (ambiguous); their
    choice is checked for admissibility, the others for equality with the
    oracle's expert list (order included where its gaps clear the bound)."""
    amb = set()
    for i, t in enumerate(tokens):
        info = R.route_token(orc["logits"][i], orc["bias"], cfg.top_k, cfg.n_group, cfg.topk_group, 1.0, 1)[2]
        em, gm = orc["margins"][i]
        d_c = _score_bound(cfg, orc["lsum"][i])
        gsel = run.idx[t]
        assert len(set(gsel.tolist())) == cfg.top_k
        if em <= 2 * d_c or gm <= 4 * d_c:
            amb.add(int(t))
            assert _admissible(cfg, info["c"], gsel, d_c), (t, gsel)
            continue
        osel = orc["idx"][i]
        assert set(gsel.tolist()) == set(osel.tolist()), (t, sorted(gsel), sorted(osel))
        c = info["c"]
        if np.all(np.abs(np.diff(c[osel])) > 2 * d_c):
            assert np.array_equal(gsel, osel), (t, gsel, osel)
        ow = dict(zip(osel.tolist(), orc["w"][i]))
        np.testing.assert_allclose(run.w[t], [ow[e] for e in gsel], rtol=2e-5, atol=1e-7)
    return amb


def check_permutation(run, cfg):
    T, k, ns, E = cfg.T, cfg.top_k, cfg.n_shared, cfg.E
    cnt = np.bincount(run.idx.reshape(-1), minlength=E)
    assert np.array_equal(run.count[:E], cnt)
    if ns:
        assert run.count[E] == T
    n_tile = run.L.n_tile
    tiles = (run.count + n_tile - 1) // n_tile
    assert np.array_equal(run.slot, np.concatenate([[0], np.cumsum(tiles)[:-1]]))
    for e in range(E + ns):
        pos = np.arange(run.count[e])
        rows = (run.slot[e] + pos // n_tile) * 128 + pos % n_tile
        toks = run.row_tok[rows]
        assert np.all(np.diff(toks) > 0), e  # ascending tokens, each once
        if e < E:
            assert set(toks.tolist()) == set(np.flatnonzero((run.idx == e).any(axis=1)).tolist())
    for t in range(T):
        for j in range(k + ns):
            r = run.route_row[t, j]
            assert run.row_tok[r] == t
            if j < k:
                assert run.row_w[r] == run.w[t, j]
            else:
                assert run.row_w[r] == 1.0


def check_x_quant(run, cfg, xc, xs, tokens):
    for i, t in enumerate(tokens):
        want_c = F.pack_nibbles(xc[i])
        for j in range(cfg.top_k + cfg.n_shared):
            assert np.array_equal(run.xq[t, j], want_c), (t, j)
            assert np.array_equal(run.xs[t, j], xs[i]), (t, j)


# ------------------------------------------------------------------ intermediate checks
def gpu_h_hat(run, cfg, t, j):
    """The GPU's dequantised intermediate of route (t, j)."""
    codes = F.unpack_nibbles(run.hq[t, j][None])
    if cfg.fmt == "mxfp4":
        return Q.mx_dequant(codes, run.hs[t, j][None])[0]
    return Q.nv_dequant(codes, run.hs[t, j][None], run.gh[run.expert_of(t, j)])[0]


def check_h_replay(run, cfg, tokens, stats):
    """The oracle's quantiser replayed on the GPU's own h gives the GPU's
    codes and scale bytes bit for bit (NVFP4: with the GPU's per-expert
    tensor scale, which must be fp32(amax / 2688) over that expert's rows of
    the GPU's h).  NVFP4 tensor scales are checked over all tokens."""
    rpt = cfg.top_k + cfg.n_shared
    if cfg.fmt == "nvfp4":
        amax = {}
        for t in range(cfg.T):
            for j in range(rpt):
                e = run.expert_of(t, j)
                amax[e] = max(amax.get(e, 0.0), float(np.max(np.abs(run.h[t, j]))))
        for e, a in amax.items():
            assert run.gh[e] == Q.nv_global_scale(np.float32(a)), (e, run.gh[e], a)
    n = 0
    for t in tokens:
        for j in range(rpt):
            h = run.h[t, j].astype(np.float64)[None]
            if cfg.fmt == "mxfp4":
                c, s = Q.mx_quantize(h)
            else:
                c, s, _ = Q.nv_quantize(h, g=run.gh[run.expert_of(t, j)])
            assert np.array_equal(F.pack_nibbles(c[0]), run.hq[t, j]), (t, j)
            assert np.array_equal(s[0], run.hs[t, j]), (t, j)
            n += 1
    stats["h_replayed_routes"] = stats.get("h_replayed_routes", 0) + n


def check_h_against_oracle(run, cfg, route_infos, stats):
    """route_infos: (t, j, info, r) with info from oracle.moe.expert_rows for
    the same expert and r the route's row in it.  The GPU's h within its
    bound; its quantised form (where compare_q) equal to the oracle's
    wherever no other quantisation is admissible."""
    for t, j, info, r, compare_q in route_infos:
        if run.h is not None:
            bound = info["dh"][r]
            err = np.abs(run.h[t, j].astype(np.float64) - info["h"][r])
            ratio = np.max(err / bound)
            stats["h_err_ratio"] = max(stats.get("h_err_ratio", 0.0), float(ratio))
            assert ratio <= 1.0, (t, j, ratio)
        if not compare_q:
            continue
        gpu_hd = gpu_h_hat(run, cfg, t, j)
        ref_hd = Q.dequant(info["hq"][r:r + 1], info["hs"][r:r + 1], cfg.fmt, info["g_h"])[0]
        diff = np.abs(gpu_hd - ref_hd)
        assert np.all(diff <= info["dmax"][r] * (1 + 1e-12)), (t, j, float(np.max(diff - info["dmax"][r])))
        stats["h_flips"] = stats.get("h_flips", 0) + int(np.count_nonzero(diff))
        stats["h_ambiguous"] = stats.get("h_ambiguous", 0) + int(np.count_nonzero(info["dmax"][r]))


# ------------------------------------------------------------------ output checks
def check_output(run, ref, S, A, tokens, skip=()):
    tol = M.tolerance(ref, S, A)
    worst = 0.0
    for i, t in enumerate(tokens):
        if t in skip:
            continue
        err = np.abs(run.out[t] - ref[i])
        ratio = err / tol[i]
        worst = max(worst, float(np.max(ratio)))
        bad = np.flatnonzero(ratio > 1)
        assert bad.size == 0, (t, bad[:5], run.out[t][bad[:5]], ref[i][bad[:5]], tol[i][bad[:5]])
    return worst


def down_weights(cfg, ws, e):
    """Dequantised down-projection matrix of expert e (shared ones after E)."""
    w2 = ws.get("w2", e) if e < cfg.E else ws.get("sh2", e - cfg.E)
    return Q.dequant(w2[0], w2[1], cfg.fmt, w2[2])


def check_output_replay(run, cfg, ws, tokens):
    """The oracle's down projection and combine on the GPU's quantised
    intermediate and routing weights: the output within 2^-8 |ref'| +
    1e-3 S' with no allowance for flips."""
    H = cfg.H
    ref = np.zeros((len(tokens), H))
    S = np.zeros((len(tokens), H))
    cache = {}
    for i, t in enumerate(tokens):
        for j in range(cfg.top_k + cfg.n_shared):
            e = run.expert_of(t, j)
            if e not in cache:
                if len(cache) > 64:
                    cache.clear()
                cache[e] = down_weights(cfg, ws, e)
            W2 = cache[e]
            hd = gpu_h_hat(run, cfg, t, j)
            wt = float(run.w[t, j]) if j < cfg.top_k else 1.0
            ref[i] += wt * (W2 @ hd)
            S[i] += abs(wt) * (np.abs(W2) @ np.abs(hd))
    return check_output(run, ref, S, np.zeros_like(ref), tokens)


# ------------------------------------------------------------------ whole-layer check
def full_check(cfg, tokens=None, h_debug=True, packed=True, cta_pair=False):
    run = DeviceRun(cfg, h_debug=h_debug, packed=packed, cta_pair=cta_pair)
    assert run.status == (0, 0), run.status
    x, wr, b = OI.layer_inputs(cfg)
    assert np.array_equal(run.x_bits, synth.gen_x_bf16(cfg))
    ws = OI.oracle_weights(cfg)
    tokens = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    exact, lsum = R.router_logits(x, wr)
    check_router_numerics(run, cfg, exact, lsum)
    check_selection_replay(run, cfg, b)
    if cfg.fmt == "nvfp4" and cfg.H * cfg.I >= 1 << 22:  # large NVFP4 weights: quantise in a spawn pool
        oi, _ = R.route(exact, b, cfg.top_k, cfg.n_group, cfg.topk_group, 1.0, 1)
        need = sorted({int(e) for t in tokens for e in oi[t]} | {int(e) for t in tokens for e in run.idx[t]})
        keys = [(w, e) for e in need for w in ("w13", "w2")] + [(w, 0) for w in ("sh13", "sh2")][:2 * cfg.n_shared]
        OI.prefetch(ws, cfg, keys)
    orc = M.layer_forward(cfg, x, wr, b, ws, tokens=tokens)
    sel = {"logits": orc["logits"][tokens], "lsum": orc["lsum"][tokens], "bias": b,
           "margins": [orc["margins"][t] for t in tokens], "idx": orc["idx"][tokens], "w": orc["w"][tokens]}
    amb = check_routing(run, cfg, sel, tokens)
    check_permutation(run, cfg)
    if cfg.fmt == "nvfp4":
        assert run.gx == orc["gx"]
    check_x_quant(run, cfg, orc["xc"][tokens], orc["xs"][tokens], tokens)
    stats = {"ambiguous_tokens": len(amb)}
    if h_debug:
        check_h_replay(run, cfg, tokens, stats)
    # experts whose rows differ between the GPU and the oracle (a re-routed
    # token): with NVFP4 their tensor scale of h is over other rows
    changed = set()
    for t in range(cfg.T):
        if set(run.idx[t].tolist()) != set(orc["idx"][t].tolist()):
            changed |= set(run.idx[t].tolist()) ^ set(orc["idx"][t].tolist())
    infos = []
    for e, info in orc["experts"].items():
        for r, (t, sl) in enumerate(zip(info["tok"], info["slot"])):
            t = int(t)
            hit = np.flatnonzero(run.idx[t] == e) if e < cfg.E else [cfg.top_k + e - cfg.E]
            if t in set(tokens.tolist()) and len(hit):
                infos.append((t, int(hit[0]), info, r, cfg.fmt == "mxfp4" or e not in changed))
    check_h_against_oracle(run, cfg, infos, stats)
    stats["worst_ratio_replayed"] = check_output_replay(run, cfg, ws, tokens)
    skip = set(amb)
    if cfg.fmt == "nvfp4":  # tokens on experts whose tensor scale of h the re-routing changed
        skip |= {int(t) for t in tokens if changed & set(run.idx[t].tolist())}
    stats["pure_oracle_skipped"] = len(skip)
    stats["worst_ratio"] = check_output(run, orc["ref"], orc["S"], orc["A"], tokens, skip)
    return stats


@pytest.mark.parametrize("name", list(SMALL))
def test_small_layers_full_oracle(name):
    stats = full_check(SMALL[name])
    print(name, stats)


@pytest.mark.parametrize("name", ["paired_padK", "pair_shared"])
def test_paired_down_on_cta_pairs(name):
    """The same parity with the paired-slot down units run on CTA pairs (M =
    256 MMAs over two SMs, the fp4moe_debug::down_cta_pair opt-in): full
    pairs, single-slot remainders and a shared expert."""
    print(name, full_check(SMALL[name], cta_pair=True))


@pytest.mark.parametrize("name", ["front_T16_shared", "paired_padK", "pair_shared", "nv_wide_padK"])
def test_small_layers_gateup_paired_level(name):
    """The same parity with the down weights in the plain tiled layout
    (packed = 2; the other tests use level 3, the row-tile-paired down
    weights): the down units of two weight tiles then read two 128-row
    boxes and two scale copies per stage."""
    print(name, full_check(SMALL[name], packed=2))


@pytest.mark.parametrize("name", ["tiny", "wide_padK", "nv_grouped", "nv_wide_padK"])
def test_small_layers_row_major_weights(name):
    """The same parity with the expert payloads left row-major (packed = 0);
    the other tests use the tiled layout of fp4moe_pack_weights."""
    print(name, full_check(SMALL[name], packed=False))


# Limits of the supported shapes and degenerate routings: 512 experts with
# top-16 through the few-token front end and through the many-token path, 32
# expert groups (NVFP4), a single expert, every expert chosen by every token.
EDGE = {
    "E512_top16_front": _cfg("tiny", name="E512_top16_front", T=16, H=256, I=128, E=512, top_k=16, n_shared=1),
    "E512_top16": _cfg("tiny", name="E512_top16", T=96, H=512, I=256, E=512, top_k=16),
    "nv_group32": _cfg("deepseek_nvfp4", name="nv_group32", T=40, H=256, I=128, E=512, top_k=8, n_group=32,
                       topk_group=4, n_shared=1),
    "single_expert": _cfg("tiny", name="single_expert", T=20, H=256, I=128, E=1, top_k=1, n_shared=1),
    "topk_all": _cfg("tiny", name="topk_all", T=33, H=256, I=128, E=8, top_k=8),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_layers_full_oracle(name):
    print(name, full_check(EDGE[name]))


def test_max_tokens_sampled():
    """T = 65536, the largest supported batch: routing on every token, the
    expert math on the first and last tokens and the chunk and half
    boundaries of the permutation."""
    cfg = _cfg("tiny", name="T_max", T=65536, H=256, I=128, E=16, top_k=4)
    print(full_check(cfg, tokens=[0, 1, 31, 32, 4095, 32767, 32768, 65534, 65535]))


# ------------------------------------------------------------------ planted ties
def _tie_router(E, H, n_group, seed):
    """Router weights and bias whose corrected scores tie exactly for the
    tokens of _tie_tokens: column 0 of Wr takes values from a small set
    (each repeated); without groups the bias repeats in pairs of experts;
    with groups the last group copies the first, so equal experts and equal
    groups occur."""
    rng = np.random.default_rng(seed)
    wr = synth.bf16_bits_to_f64(synth.to_bf16_bits(rng.standard_normal((E, H)) * 0.02))
    vals = np.array([0.5, 0.25, -0.125, 0.75])
    col = vals[rng.integers(0, len(vals), E)]
    if n_group > 1:
        # zero bias: a group score is then a sum of two of four sigmoid
        # values, equal for two groups only when their top two are, so the
        # fp32 and float64 group orders agree
        bias = np.zeros(E, dtype=np.float32)
        gsz = E // n_group
        col[-gsz:] = col[:gsz]
    else:
        bias = np.repeat(rng.choice(np.array([0.0, 0.125, -0.0625], dtype=np.float32), E // 2), 2)
    wr[:, 0] = col
    return wr, bias.astype(np.float32)


def _tie_tokens(T, H, seed):
    """Tokens with one non-zero element (x[t, 0] = 1): every logit is then the
    bf16 value Wr[e, 0] exactly, whatever the summation order.  Every fourth
    token is all zeros (every logit 0, every score 1/2)."""
    x = np.zeros((T, H))
    x[:, 0] = 1.0
    x[::4, 0] = 0.0
    return x


def _expect_tie_routing(cfg, x, wr, bias, gidx, gw):
    exact, _ = R.router_logits(x, wr)
    n_ties = 0
    for t in range(cfg.T):
        oi, ow, info = R.route_token(exact[t], bias, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.routed_scaling,
                                     cfg.renormalize)
        assert np.array_equal(gidx[t], oi), (t, gidx[t], oi)  # order included: ties to the lower index
        np.testing.assert_allclose(gw[t], ow, rtol=2e-7)
        c = info["c"]
        n_ties += int(np.count_nonzero(c[oi[:-1]] == c[oi[1:]]))
    assert n_ties > 0
    return n_ties


@pytest.mark.parametrize("T,n_group,topk_group", [(8, 1, 1), (40, 1, 1), (8, 4, 2), (40, 8, 3)])
def test_route_planted_ties(T, n_group, topk_group):
    """fp4moe_route (GEMV router for T <= 16, tensor-core router above) on
    tokens whose corrected scores tie exactly: expert lists equal the
    oracle's, order included (lower expert and lower group win)."""
    torch = torch_cuda()
    ensure_built()
    cfg = _cfg("tiny", name="ties", T=T, H=512, E=64, top_k=6, n_group=n_group, topk_group=topk_group,
               routed_scaling=2.5)
    wr, bias = _tie_router(cfg.E, cfg.H, n_group, 40 + T + n_group)
    x = _tie_tokens(T, cfg.H, 0)
    d = dims_of(cfg)
    xd = torch.from_numpy(synth.to_bf16_bits(x).view(np.int16)).cuda()
    wd = torch.from_numpy(synth.to_bf16_bits(wr).view(np.int16)).cuda()
    bd = torch.from_numpy(bias).cuda()
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    n = fm.workspace_size(d)
    wsb = torch.empty(n, dtype=torch.uint8, device="cuda")
    fm.route(d, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(), idx.data_ptr(), w.data_ptr(), None, wsb.data_ptr(), n)
    torch.cuda.synchronize()
    print(_expect_tie_routing(cfg, x, wr, bias, idx.cpu().numpy(), w.cpu().numpy()), "tied neighbours")


@pytest.mark.parametrize("name,n_group", [("front_T16_shared", 1), ("nv_grouped", 4)])
def test_forward_planted_ties(name, n_group):
    """The same planted ties through fp4moe_forward: the few-token fused
    front end (MXFP4, T <= 16) and the many-token NVFP4 grouped path."""
    torch = torch_cuda()
    ensure_built()
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfg = SMALL[name]
    layer = MoELayer.synthetic(cfg)
    wr, bias = _tie_router(cfg.E, cfg.H, n_group, 7)
    layer.w_router.copy_(torch.from_numpy(synth.to_bf16_bits(wr).view(np.int16)))
    layer.bias.copy_(torch.from_numpy(bias))
    x = _tie_tokens(cfg.T, cfg.H, 0)
    xd = torch.from_numpy(synth.to_bf16_bits(x).view(np.int16)).cuda().view(torch.bfloat16)
    run = DeviceRun(cfg, layer=layer, x=xd)
    assert run.status == (0, 0)
    check_selection_replay(run, cfg, bias)
    print(_expect_tie_routing(cfg, x, wr, bias, run.idx, run.w), "tied neighbours")


# ------------------------------------------------------------------ output partition
def _column_slices(cfg, layer, x, world):
    """fp4moe_forward_cols for every rank's block of output columns, run one
    after another on this GPU (no rank waits for another); each block's
    output is zero outside its columns.  Returns their sum (exact: the
    blocks are disjoint)."""
    torch = torch_cuda()
    from block_scaled_fp4_sigmoid_gb300.layer import column_block
    total = np.zeros((cfg.T, cfg.H))
    for r in range(world):
        h0, h1 = column_block(cfg.H, r, world, layer.column_unit)
        out = layer.forward_cols(x, h0, h1)
        torch.cuda.synchronize()
        assert fm.get_status(layer.ws.data_ptr()) == (0, 0)
        o = synth.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        assert not np.any(o[:, :h0]) and not np.any(o[:, h1:]), (r, h0, h1)
        total += o
    return total


def _ambiguous_tokens(cfg, orc, tokens, bias):
    amb = set()
    for i, t in enumerate(tokens):
        em, gm = orc["margins"][i]
        d_c = _score_bound(cfg, orc["lsum"][i])
        if em <= 2 * d_c or gm <= 4 * d_c:
            amb.add(int(t))
    return amb


@pytest.mark.parametrize("name,world", [("ragged_shared", 2), ("ragged_shared", 4), ("front_cluster3", 3),
                                        ("nv_grouped", 2), ("wide_padK", 8), ("paired_padK", 2),
                                        ("paired_padK", 8)])
def test_output_column_blocks_sum_to_the_layer(name, world):
    """Output-partitioned layer: the ranks' column blocks, summed, meet the
    layer tolerance against the whole oracle (the few-token front end, the
    many-token path, a shared expert, NVFP4, K padding; down units of two
    weight tiles on row-tile-paired weights in 512-column blocks, paired-slot
    units in 128-column blocks).  Blocks of whole 256-row slabs use the
    row-tile-paired down weights (packed level 3), 128-column blocks level 2."""
    from types import SimpleNamespace
    torch_cuda()
    ensure_built()
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfg = SMALL[name]
    layer = MoELayer.synthetic(cfg, packed=3 if cfg.H % (256 * world) == 0 else 2)
    total = _column_slices(cfg, layer, layer.synthetic_x(), world)
    x, wr, b = OI.layer_inputs(cfg)
    tokens = np.arange(cfg.T)
    orc = M.layer_forward(cfg, x, wr, b, OI.oracle_weights(cfg), tokens=tokens)
    amb = _ambiguous_tokens(cfg, orc, tokens, b)
    print(name, world, check_output(SimpleNamespace(out=total), orc["ref"], orc["S"], orc["A"], tokens, amb))


def test_kimi_decode_output_column_blocks_full_size():
    """The Kimi decode layer as two ranks' column blocks (3584 columns
    each), sampled tokens against the oracle."""
    from types import SimpleNamespace
    torch_cuda()
    ensure_built()
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfg = synth.configs()["kimi_decode"]
    layer = MoELayer.synthetic(cfg)
    total = _column_slices(cfg, layer, layer.synthetic_x(), 2)
    del layer
    tokens = np.array([0, 5])
    xr = np.concatenate([synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg, int(t), int(t) + 1)) for t in tokens])
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    b = synth.gen_bias_f32(cfg)
    orc = M.token_forward(cfg, xr, wr, b, OI.oracle_weights(cfg))
    amb = _ambiguous_tokens(cfg, orc, tokens, b)
    out = np.zeros((cfg.T, cfg.H))
    out[tokens] = total[tokens]
    print(check_output(SimpleNamespace(out=out), orc["ref"], orc["S"], orc["A"], tokens, amb))


def test_route_entry_point_matches_forward_routing():
    """fp4moe_route's logits within their bound, its experts and weights the
    fp32 selection replayed on the scores its logits give."""
    torch = torch_cuda()
    ensure_built()
    cfg = SMALL["nv_grouped"]
    d = dims_of(cfg)
    x = torch.from_numpy(synth.gen_x_bf16(cfg).view(np.int16)).cuda()
    wr = torch.from_numpy(synth.gen_router_bf16(cfg).view(np.int16)).cuda()
    b = torch.from_numpy(synth.gen_bias_f32(cfg)).cuda()
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    n = fm.workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    fm.route(d, x.data_ptr(), wr.data_ptr(), b.data_ptr(), idx.data_ptr(), w.data_ptr(), logits.data_ptr(),
             ws.data_ptr(), n)
    torch.cuda.synchronize()
    xf, wrf, bias = OI.layer_inputs(cfg)
    ol, lsum = R.router_logits(xf, wrf)
    gl = logits.cpu().numpy()
    assert np.all(np.abs(gl - ol) <= LOGIT_GAMMA * lsum)
    run = DeviceRun(cfg)  # the forward's router: same kernels, scores exposed
    assert np.array_equal(run.idx, idx.cpu().numpy()) and np.array_equal(run.w, w.cpu().numpy())
    assert np.array_equal(run.logits, gl)


# ------------------------------------------------------------------ full-size workloads
def _token_check(name, tokens):
    """Routing of every token (logits, scores, fp32 selection replay,
    permutation), the expert math of the sampled tokens."""
    cfg = synth.configs()[name]
    run = DeviceRun(cfg, h_debug=True)
    assert run.status == (0, 0), run.status
    tokens = np.asarray(tokens)
    x_all = synth.bf16_bits_to_f64(run.x_bits)
    assert np.array_equal(run.x_bits, synth.gen_x_bf16(cfg))
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    b = synth.gen_bias_f32(cfg)
    for t0 in range(0, cfg.T, 2048):  # exact logits of every token, in slices
        sl = slice(t0, min(cfg.T, t0 + 2048))
        exact, lsum = R.router_logits(x_all[sl], wr)
        check_router_numerics(run, cfg, exact, lsum, np.arange(cfg.T)[sl])
    check_selection_replay(run, cfg, b)
    check_permutation(run, cfg)
    xr = x_all[tokens]
    ws = OI.oracle_weights(cfg)
    orc = M.token_forward(cfg, xr, wr, b, ws)
    orc["bias"] = b
    amb = check_routing(run, cfg, orc, tokens)
    check_x_quant(run, cfg, orc["xc"], orc["xs"], tokens)
    stats = {"ambiguous_tokens": len(amb)}
    check_h_replay(run, cfg, tokens, stats)
    infos = []
    for i, t in enumerate(tokens):
        for j, info in enumerate(orc["routes"][i]):
            hit = np.flatnonzero(run.idx[t] == info["expert"]) if j < cfg.top_k else [j]
            if len(hit):
                infos.append((int(t), int(hit[0]), info, 0, True))
    check_h_against_oracle(run, cfg, infos, stats)
    stats["worst_ratio_replayed"] = check_output_replay(run, cfg, ws, tokens)
    stats["worst_ratio"] = check_output(run, orc["ref"], orc["S"], orc["A"], tokens, amb)
    return stats, run


def test_kimi_decode_full_size():
    stats, _ = _token_check("kimi_decode", [0, 3, 7])
    print(stats)


def test_kimi_prefill_full_size():
    stats, _ = _token_check("kimi_prefill", [0, 2047, 4095])
    print(stats)


def test_skewed_shared_full_size():
    cfg = synth.configs()["skewed_shared"]
    stats, run = _token_check("skewed_shared", [0, 9000, 16383])
    share = run.count[:cfg.E].max() / (cfg.T * cfg.top_k)
    assert 0.07 <= share <= 0.09, share  # Zipf-shaped bias: the hottest expert takes ~8%
    print(stats, share)


def test_deepseek_nvfp4_full_size():
    cfg = synth.configs()["deepseek_nvfp4"]
    stats = full_check(cfg, tokens=[5, 300], h_debug=True)
    print(stats)
