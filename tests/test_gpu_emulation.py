"""GPU parity of fp4moe_forward_nvfp4_emulated (the NVFP4 layer in emulation
mode: BF16 dequantised experts, NVFP4 QDQ activations and intermediate, BF16
GEMMs with fp32 accumulation) against the emulation oracle:
  1. routing: logits and scores within their bounds, the fp32 selection
     replayed on the GPU's scores bit-exact on every token, agreement with
     the pure oracle where its margins clear the bound, and permutation;
  2. the BF16 activation rows bit-exact, in every route row of a token, and
     the tensor scale of x bit-exact;
  3. the intermediate h within its error bound before the round trip; the
     per-expert tensor scale of h equal to fp32(amax / 2688) over the GPU's
     own h, and the BF16 round trip of the GPU's h replayed by the oracle
     equal to the GPU's BF16 rows bit for bit; against the oracle's own h,
     the scale within the range its bound admits and the BF16 values equal
     wherever no other NVFP4 quantisation is admissible;
  4. the layer output within 2^-8 |ref'| + 1e-3 S' of the oracle's down
     projection replayed on the GPU's BF16 intermediate (no allowance), and
     within 2^-8 |ref| + 1e-3 S + A of the pure oracle where routing agrees.
Small layers check every token; the DeepSeek-shaped layer (T = 512), in the
benchmark's launch configuration, checks sampled tokens."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import emulation as EM
from oracle import inputs as OI
from oracle import quant as Q
from oracle import router as R

from gpu_util import ensure_built, torch_cuda
from test_gpu_forward import (SMALL, check_output, check_permutation, check_router_numerics, check_routing,
                              check_selection_replay)

pytestmark = pytest.mark.gpu


def _align(v):
    return (v + 255) // 256 * 256


class RunEm:
    def __init__(self, cfg, packed=True):
        torch = torch_cuda()
        ensure_built()
        from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
        layer = MoELayer.synthetic(cfg, packed=packed)
        x = layer.synthetic_x()
        L = layer.layout
        self.L = L
        h_pre = torch.zeros((L.rows_cap, cfg.I), dtype=torch.float32, device="cuda")
        dbg = fm.Debug()
        dbg.h_pre = h_pre.data_ptr()
        logits = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        scores = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        dbg.logits, dbg.scores = logits.data_ptr(), scores.data_ptr()
        out = layer.forward_emulated(x, debug=dbg)
        torch.cuda.synchronize()
        self.cfg = cfg
        self.logits, self.scores = logits.cpu().numpy(), scores.cpu().numpy()
        ws = layer.emu_ws
        self.status = fm.get_status(ws.data_ptr())
        T, k, ns = cfg.T, cfg.top_k, cfg.n_shared
        rpt = k + ns
        i32 = lambda off, n: ws[off:off + 4 * n].view(torch.int32).cpu().numpy()
        f32 = lambda off, n: ws[off:off + 4 * n].view(torch.float32).cpu().numpy()
        self.x_bits = x.view(torch.int16).cpu().numpy().view(np.uint16)
        self.out = synth.bf16_bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
        self.idx = i32(L.topk_idx, T * k).reshape(T, k)
        self.w = f32(L.topk_w, T * k).reshape(T, k)
        self.count = i32(L.expert_count, cfg.E + ns)
        self.slot = i32(L.expert_slot, cfg.E + ns)
        self.route_row = i32(L.route_row, T * rpt).reshape(T, rpt)
        self.row_tok = i32(L.row_tok, L.rows_cap)
        self.row_w = f32(L.row_w, L.rows_cap)
        g = f32(L.gscale, 2 + cfg.E + ns)
        self.gx, self.gh = g[0], g[2:]
        # bf16 rows of x and h follow the forward's layout (256-byte aligned)
        xb_off = _align(L.total_bytes)
        hb_off = _align(xb_off + L.rows_cap * cfg.H * 2)
        rows = torch.from_numpy(self.route_row.reshape(-1).astype(np.int64)).cuda()
        xb = ws[xb_off:xb_off + L.rows_cap * cfg.H * 2].view(torch.int16).view(L.rows_cap, cfg.H)
        hb = ws[hb_off:hb_off + L.rows_cap * cfg.I * 2].view(torch.int16).view(L.rows_cap, cfg.I)
        self.xb = synth.bf16_bits_to_f64(xb[rows].cpu().numpy().view(np.uint16)).reshape(T, rpt, cfg.H)
        self.hb = synth.bf16_bits_to_f64(hb[rows].cpu().numpy().view(np.uint16)).reshape(T, rpt, cfg.I)
        self.h = h_pre[rows].cpu().numpy().reshape(T, rpt, cfg.I)
        del out, h_pre, layer

    def expert_of(self, t, j):
        return int(self.idx[t, j]) if j < self.cfg.top_k else self.cfg.E + j - self.cfg.top_k


def check_em(cfg, tokens, packed=True):
    run = RunEm(cfg, packed)
    assert run.status == (0, 0), run.status
    x, wr, b = OI.layer_inputs(cfg)
    assert np.array_equal(run.x_bits, synth.gen_x_bf16(cfg))
    ws = OI.oracle_weights(cfg)
    tokens = np.asarray(tokens)
    exact, lsum = R.router_logits(x, wr)
    check_router_numerics(run, cfg, exact, lsum)
    check_selection_replay(run, cfg, b)
    if cfg.H * cfg.I >= 1 << 22:  # large weights: quantise them in a spawn pool
        oi, _ = R.route(exact, b, cfg.top_k, cfg.n_group, cfg.topk_group, 1.0, 1)
        need = sorted({int(e) for t in tokens for e in run.idx[t]} | {int(e) for t in tokens for e in oi[t]})
        keys = [(w, e) for e in need for w in ("w13", "w2")] + [(w, 0) for w in ("sh13", "sh2")][:2 * cfg.n_shared]
        OI.prefetch(ws, cfg, keys)
    orc = EM.emulated_layer_forward(cfg, x, wr, b, ws, tokens=tokens)
    sel = {"logits": orc["logits"][tokens], "lsum": orc["lsum"][tokens], "bias": b,
           "margins": [orc["margins"][t] for t in tokens], "idx": orc["idx"][tokens], "w": orc["w"][tokens]}
    amb = check_routing(run, cfg, sel, tokens)
    check_permutation(run, cfg)
    assert run.gx == orc["gx"]
    for t in tokens:
        for j in range(cfg.top_k + cfg.n_shared):
            assert np.array_equal(run.xb[t, j], orc["a"][t]), (t, j)
    rpt = cfg.top_k + cfg.n_shared
    stats = {"ambiguous_tokens": len(amb), "h_flips": 0, "h_ambiguous": 0, "h_err_ratio": 0.0}
    # replay: the GPU's per-expert tensor scale of h from its own h, and the
    # BF16 round trip of its own h, bit for bit
    amax = {}
    for t in range(cfg.T):
        for j in range(rpt):
            e = run.expert_of(t, j)
            amax[e] = max(amax.get(e, 0.0), float(np.max(np.abs(run.h[t, j]))))
    for e, a in amax.items():
        assert run.gh[e] == Q.nv_global_scale(np.float32(a)), (e, run.gh[e], a)
    for t in tokens:
        for j in range(rpt):
            c, sc, g = Q.nv_quantize(run.h[t, j].astype(np.float64)[None], g=run.gh[run.expert_of(t, j)])
            assert np.array_equal(EM.nv_dequant_bf16(c, sc, g)[0], run.hb[t, j]), (t, j)
    # experts whose rows differ from the oracle's (re-routed tokens): their
    # tensor scale of h is over other rows, so the comparison with the
    # oracle's own quantisation skips them
    changed = set()
    for t in range(cfg.T):
        if set(run.idx[t].tolist()) != set(orc["idx"][t].tolist()):
            changed |= set(run.idx[t].tolist()) ^ set(orc["idx"][t].tolist())
    chosen = set(tokens.tolist())
    for e, info in orc["experts"].items():
        if e not in changed:
            # the tensor scale of h follows the |max| of the expert's fp32 h:
            # any value its error bound admits
            g_lo = Q.nv_global_scale(float(np.max(np.maximum(np.abs(info["h32"]) - info["dh"], 0.0))))
            g_hi = Q.nv_global_scale(float(np.max(np.abs(info["h32"]) + info["dh"])))
            assert g_lo <= run.gh[e] <= g_hi, (e, run.gh[e], g_lo, g_hi)
        for r, (t, sl) in enumerate(zip(info["tok"], info["slot"])):
            t = int(t)
            if t not in chosen:
                continue
            hit = np.flatnonzero(run.idx[t] == e) if e < cfg.E else [int(sl)]
            if not len(hit):
                continue
            jj = int(hit[0])
            err = np.abs(run.h[t, jj].astype(np.float64) - info["h"][r])
            ratio = float(np.max(err / info["dh"][r]))
            stats["h_err_ratio"] = max(stats["h_err_ratio"], ratio)
            assert ratio <= 1.0, (t, e, ratio)
            if e in changed:
                continue
            diff = np.abs(run.hb[t, jj] - info["hd"][r])
            assert np.all(diff <= info["dmax"][r] * (1 + 1e-12)), (t, e, float(np.max(diff - info["dmax"][r])))
            stats["h_flips"] += int(np.count_nonzero(diff))
            stats["h_ambiguous"] += int(np.count_nonzero(info["dmax"][r]))
    # the output against the oracle's down projection on the GPU's BF16
    # intermediate and routing weights, no allowance
    ref2 = np.zeros((len(tokens), cfg.H))
    S2 = np.zeros_like(ref2)
    for i, t in enumerate(tokens):
        for j in range(rpt):
            e = run.expert_of(t, j)
            W2 = EM.nv_dequant_bf16(*(ws.get("w2", e) if e < cfg.E else ws.get("sh2", e - cfg.E)))
            wt = float(run.w[t, j]) if j < cfg.top_k else 1.0
            ref2[i] += wt * (W2 @ run.hb[t, j])
            S2[i] += abs(wt) * (np.abs(W2) @ np.abs(run.hb[t, j]))
    stats["worst_ratio_replayed"] = check_output(run, ref2, S2, np.zeros_like(ref2), tokens)
    skip = set(amb) | {int(t) for t in tokens if changed & set(run.idx[t].tolist())}
    stats["pure_oracle_skipped"] = len(skip)
    stats["worst_ratio"] = check_output(run, orc["ref"], orc["S"], orc["A"], tokens, skip)
    return stats


@pytest.mark.parametrize("name", ["nv_grouped", "nv_wide_padK"])
def test_small_layers_emulated(name):
    cfg = SMALL[name]
    print(name, check_em(cfg, np.arange(cfg.T)))


def test_emulated_row_major_weights():
    """The weight dequantisation reading row-major payloads (packed = 0)."""
    cfg = SMALL["nv_wide_padK"]
    print(check_em(cfg, np.arange(cfg.T), packed=False))


def test_deepseek_nvfp4_emulated_full_size():
    print(check_em(synth.configs()["deepseek_nvfp4"], [5, 300]))
