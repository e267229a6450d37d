"""GPU parity of fp4moe_route and fp4moe_forward against the FP64 oracle.

Staged, so that a mismatch is attributed to its step:
  1. routing: expert sets bit-exact except tokens whose oracle decision margin
     is below the logit error bound (those are checked for validity only);
     router logits within that bound; routing weights to fp32 rounding;
  2. permutation: counts, slot layout, ascending tokens inside each expert,
     and route <-> row consistency (unique given the routing);
  3. quantised activations: bit-exact codes and scale bytes per route;
  4. the pre-quantisation intermediate h within its error bound, and its
     quantised form equal to the oracle's wherever no other quantisation is
     admissible (elsewhere one of the admissible ones);
  5. the layer output: |gpu - ref| <= 2^-8 |ref| + 1e-3 S + A per element.
Small configurations run the whole oracle; the full-size workloads, in the
launch configuration the benchmark times, check sampled tokens."""
from dataclasses import replace

import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import formats as F
from oracle import inputs as OI
from oracle import moe as M
from oracle import quant as Q

from gpu_util import dims_of, ensure_built, katoms_padded, read_tiled_scales, torch_cuda

pytestmark = pytest.mark.gpu

LOGIT_GAMMA = 2.0 ** -16  # |logit_gpu - logit| <= LOGIT_GAMMA * sum |x * Wr|


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
    "nv_grouped": _cfg("deepseek_nvfp4", name="nv_grouped", T=64, H=512, I=256, E=32, top_k=4, n_group=4,
                       topk_group=2),
    "nv_wide_padK": _cfg("deepseek_nvfp4", name="nv_wide_padK", T=200, H=256, I=128, E=4, top_k=2, n_group=2,
                         topk_group=1, n_shared=1),
}


class DeviceRun:
    """One forward on the GPU plus host copies of its intermediates."""

    def __init__(self, cfg, h_debug=True, packed=True):
        torch = torch_cuda()
        ensure_built()
        from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
        self.torch = torch
        self.cfg = cfg
        layer = MoELayer.synthetic(cfg, packed=packed)
        x = layer.synthetic_x()
        L = layer.layout
        self.L = L
        dbg = fm.Debug()
        h_pre = None
        if h_debug:
            h_pre = torch.zeros((L.rows_cap, cfg.I), dtype=torch.float32, device="cuda")
            dbg.h_pre = h_pre.data_ptr()
        out = layer.forward(x, debug=dbg)
        torch.cuda.synchronize()
        self.status = fm.get_status(layer.ws.data_ptr())
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


# ------------------------------------------------------------------ checks
def _ambiguous_tokens(cfg, logits, lsum, margins, tokens):
    """Tokens whose selection a logit error within the bound could change."""
    amb = set()
    for i, t in enumerate(tokens):
        em, gm = margins[i]
        d_logit = LOGIT_GAMMA * np.max(lsum[i])
        d_c = 0.25 * d_logit + 2.0 ** -22
        if em <= 2 * d_c or gm <= 4 * d_c:
            amb.add(int(t))
    return amb


def check_routing(run, cfg, orc, tokens):
    amb = _ambiguous_tokens(cfg, orc["logits"], orc["lsum"], orc["margins"], tokens)
    for i, t in enumerate(tokens):
        gsel, osel = set(run.idx[t].tolist()), set(orc["idx"][i].tolist())
        assert len(gsel) == cfg.top_k
        if t in amb:
            continue
        assert gsel == osel, (t, sorted(gsel), sorted(osel))
        ow = dict(zip(orc["idx"][i].tolist(), orc["w"][i]))
        gw = np.array([ow[e] for e in run.idx[t]])
        np.testing.assert_allclose(run.w[t], gw, rtol=2e-5, atol=1e-7)
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


def _route_info(cfg, orc_route, run, t, j):
    """GPU dequantised h of route (t, j) and the oracle's admissible window."""
    e_fmt = cfg.fmt
    codes = F.unpack_nibbles(run.hq[t, j][None])
    if e_fmt == "mxfp4":
        gpu_hd = Q.mx_dequant(codes, run.hs[t, j][None])[0]
    else:
        e = run.idx[t, j] if j < cfg.top_k else cfg.E + j - cfg.top_k
        gpu_hd = Q.nv_dequant(codes, run.hs[t, j][None], run.gh[e])[0]
    return gpu_hd


def check_h(run, cfg, route_infos, stats):
    """route_infos: list of (t, j, info, r) with info from oracle.moe.expert_rows and r the row in it."""
    for t, j, info, r in route_infos:
        if run.h is not None:
            bound = info["dh"][r]
            err = np.abs(run.h[t, j].astype(np.float64) - info["h"][r])
            ratio = np.max(err / bound)
            stats["h_err_ratio"] = max(stats.get("h_err_ratio", 0.0), float(ratio))
            assert ratio <= 1.0, (t, j, ratio)
        gpu_hd = _route_info(cfg, None, run, t, j)
        fmt = cfg.fmt
        ref_hd = Q.dequant(info["hq"][r:r + 1], info["hs"][r:r + 1], fmt, info["g_h"])[0]
        diff = np.abs(gpu_hd - ref_hd)
        assert np.all(diff <= info["dmax"][r] * (1 + 1e-12)), (t, j, float(np.max(diff - info["dmax"][r])))
        stats["h_flips"] = stats.get("h_flips", 0) + int(np.count_nonzero(diff))
        stats["h_ambiguous"] = stats.get("h_ambiguous", 0) + int(np.count_nonzero(info["dmax"][r]))


def check_output(run, ref, S, A, tokens, skip):
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


def full_check(cfg, tokens=None, h_debug=True, packed=True):
    run = DeviceRun(cfg, h_debug=h_debug, packed=packed)
    assert run.status == (0, 0), run.status
    x, wr, b = OI.layer_inputs(cfg)
    assert np.array_equal(run.x_bits, synth.gen_x_bf16(cfg))
    ws = OI.oracle_weights(cfg)
    tokens = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    if cfg.fmt == "nvfp4" and cfg.H * cfg.I >= 1 << 22:  # large NVFP4 weights: quantise in a spawn pool
        from oracle.router import route as oroute, router_logits
        oi, _ = oroute(router_logits(x, wr)[0], b, cfg.top_k, cfg.n_group, cfg.topk_group, 1.0, 1)
        need = sorted({int(e) for t in tokens for e in oi[t]})
        keys = [(w, e) for e in need for w in ("w13", "w2")] + [(w, 0) for w in ("sh13", "sh2")][:2 * cfg.n_shared]
        OI.prefetch(ws, cfg, keys)
    orc = M.layer_forward(cfg, x, wr, b, ws, tokens=tokens)
    sel = {"logits": orc["logits"][tokens], "lsum": orc["lsum"][tokens],
           "margins": [orc["margins"][t] for t in tokens], "idx": orc["idx"][tokens], "w": orc["w"][tokens]}
    amb = check_routing(run, cfg, sel, tokens)
    check_permutation(run, cfg)
    if cfg.fmt == "nvfp4":
        assert run.gx == orc["gx"]
    check_x_quant(run, cfg, orc["xc"][tokens], orc["xs"][tokens], tokens)
    stats = {"ambiguous_tokens": len(amb)}
    infos = []
    chosen = set(tokens.tolist()) - amb
    for e, info in orc["experts"].items():
        for r, (t, sl) in enumerate(zip(info["tok"], info["slot"])):
            if int(t) in chosen:
                infos.append((int(t), int(sl), info, r))
    if cfg.fmt == "mxfp4" or not amb:  # NVFP4: a re-routed token changes its experts' tensor scales
        check_h(run, cfg, infos, stats)
    stats["worst_ratio"] = check_output(run, orc["ref"], orc["S"], orc["A"], tokens, amb)
    return stats


@pytest.mark.parametrize("name", list(SMALL))
def test_small_layers_full_oracle(name):
    stats = full_check(SMALL[name])
    print(name, stats)


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
    """T = 65536, the largest supported batch: first and last tokens, chunk
    and half boundaries of the permutation."""
    cfg = _cfg("tiny", name="T_max", T=65536, H=256, I=128, E=16, top_k=4)
    print(full_check(cfg, tokens=[0, 1, 31, 32, 4095, 32767, 32768, 65534, 65535]))


def _column_slices(cfg, layer, x, world):
    """fp4moe_forward_cols for every rank's block of output columns, run one
    after another on this GPU (no rank waits for another); each block's
    output is zero outside its columns.  Returns their sum (exact: the
    blocks are disjoint)."""
    torch = torch_cuda()
    from block_scaled_fp4_sigmoid_gb300.layer import column_block
    total = np.zeros((cfg.T, cfg.H))
    for r in range(world):
        h0, h1 = column_block(cfg.H, r, world)
        out = layer.forward_cols(x, h0, h1)
        torch.cuda.synchronize()
        assert fm.get_status(layer.ws.data_ptr()) == (0, 0)
        o = synth.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        assert not np.any(o[:, :h0]) and not np.any(o[:, h1:]), (r, h0, h1)
        total += o
    return total


@pytest.mark.parametrize("name,world", [("ragged_shared", 2), ("ragged_shared", 4), ("front_cluster3", 3),
                                        ("nv_grouped", 2), ("wide_padK", 8)])
def test_output_column_blocks_sum_to_the_layer(name, world):
    """Output-partitioned layer: the ranks' column blocks, summed, meet the
    layer tolerance against the whole oracle (the few-token front end, the
    many-token path, a shared expert, NVFP4, K padding)."""
    from types import SimpleNamespace
    torch_cuda()
    ensure_built()
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfg = SMALL[name]
    layer = MoELayer.synthetic(cfg)
    total = _column_slices(cfg, layer, layer.synthetic_x(), world)
    x, wr, b = OI.layer_inputs(cfg)
    tokens = np.arange(cfg.T)
    orc = M.layer_forward(cfg, x, wr, b, OI.oracle_weights(cfg), tokens=tokens)
    amb = _ambiguous_tokens(cfg, orc["logits"], orc["lsum"], orc["margins"], tokens)
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
    orc = M.token_forward(cfg, xr, wr, synth.gen_bias_f32(cfg), OI.oracle_weights(cfg))
    amb = _ambiguous_tokens(cfg, orc["logits"], orc["lsum"], orc["margins"], tokens)
    print(check_output(SimpleNamespace(out=total), orc["ref"], orc["S"], orc["A"], tokens, amb))


def test_route_entry_point_matches_forward_routing():
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
    ol, lsum = xf @ wrf.T, np.abs(xf) @ np.abs(wrf).T
    assert np.all(np.abs(logits.cpu().numpy() - ol) <= LOGIT_GAMMA * lsum)
    from oracle.router import route as oroute, decision_margins
    oi, ow = oroute(ol, bias, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.routed_scaling, 1)
    for t in range(cfg.T):
        assert set(idx[t].tolist()) == set(oi[t].tolist())


# ------------------------------------------------------------------ full-size workloads
def _token_check(name, tokens):
    cfg = synth.configs()[name]
    run = DeviceRun(cfg, h_debug=True)
    assert run.status == (0, 0), run.status
    tokens = np.asarray(tokens)
    xr = np.concatenate([synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg, int(t), int(t) + 1)) for t in tokens])
    assert np.array_equal(synth.to_bf16_bits(xr), run.x_bits[tokens])
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    b = synth.gen_bias_f32(cfg)
    ws = OI.oracle_weights(cfg)
    orc = M.token_forward(cfg, xr, wr, b, ws)
    amb = check_routing(run, cfg, orc, tokens)
    check_permutation(run, cfg)
    check_x_quant(run, cfg, orc["xc"], orc["xs"], tokens)
    stats = {"ambiguous_tokens": len(amb)}
    infos = []
    for i, t in enumerate(tokens):
        if int(t) in amb:
            continue
        for j, info in enumerate(orc["routes"][i]):
            jj = j if j >= cfg.top_k else int(np.flatnonzero(run.idx[t] == info["expert"])[0])
            infos.append((int(t), jj, info, 0))
    check_h(run, cfg, infos, stats)
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
