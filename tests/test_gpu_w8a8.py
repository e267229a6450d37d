"""GPU parity of fp4moe_forward_w8a8 against the W8A8 FP64 oracle.

The W8A8 layer runs the experts of an MXFP4 layer after the exact per-channel
FP8 conversion, with per-token dynamic E4M3 activations.  Staged like the
A4W4 parity tests:
  1. routing (logits and scores within their bounds, the fp32 selection
     replayed on the GPU's scores bit-exact on every token) and permutation
     (same kernels as the A4W4 layer);
  2. quantised activations: E4M3 codes and the fp32 row scale bit-exact in
     every route row of a token;
  3. the intermediate h within its error bound before quantisation; its codes
     equal to the oracle's wherever no other quantisation is admissible (else
     one of the admissible ones), its row scale within the admissible range,
     and codes and scale bit-exact to the oracle's quantiser replayed on the
     GPU's own h;
  4. the layer output within |gpu - ref| <= 2^-8 |ref| + 1e-3 S + A, and
     within 2^-8 |ref'| + 1e-3 S of the oracle's down projection replayed on
     the GPU's quantised intermediate.
Small layers check every token; the Kimi-shaped layers, in the benchmark's
launch configuration, check sampled tokens."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import formats as F
from oracle import w8a8 as W8

from gpu_util import ensure_built, torch_cuda
from test_gpu_forward import (SMALL, check_output, check_permutation, check_router_numerics, check_routing,
                              check_selection_replay)
from oracle import router as R

pytestmark = pytest.mark.gpu


class Run8:
    """One W8A8 forward plus host copies of its intermediates."""

    def __init__(self, cfg):
        torch = torch_cuda()
        ensure_built()
        from block_scaled_fp4_sigmoid_gb300.layer import MoELayer, W8A8Layer
        mx = MoELayer.synthetic(cfg)
        layer = W8A8Layer(mx)
        del mx.w13, mx.w2, mx.w13_t, mx.w2_t  # the W8A8 layer keeps its own converted copies
        x = layer.synthetic_x()
        L = layer.layout
        self.L = L
        h_pre = torch.zeros((L.rows_cap, cfg.I), dtype=torch.float32, device="cuda")
        dbg = fm.Debug()
        dbg.h_pre = h_pre.data_ptr()
        logits = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        scores = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        dbg.logits, dbg.scores = logits.data_ptr(), scores.data_ptr()
        out = layer.forward(x, debug=dbg)
        torch.cuda.synchronize()
        self.logits, self.scores = logits.cpu().numpy(), scores.cpu().numpy()
        self.status = fm.get_status(layer.ws.data_ptr())
        T, k, ns = cfg.T, cfg.top_k, cfg.n_shared
        rpt = k + ns
        ws = layer.ws
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
        rows = torch.from_numpy(self.route_row.reshape(-1).astype(np.int64)).cuda()
        xq = ws[L.xq:L.xq + L.rows_cap * cfg.H].view(L.rows_cap, cfg.H)
        self.xq = xq[rows].cpu().numpy().reshape(T, rpt, cfg.H)
        self.xsig = ws[L.xsf:L.xsf + 4 * L.rows_cap].view(torch.float32)[rows].cpu().numpy().reshape(T, rpt)
        hq = ws[L.hq:L.hq + L.rows_cap * cfg.I].view(L.rows_cap, cfg.I)
        self.hq = hq[rows].cpu().numpy().reshape(T, rpt, cfg.I)
        self.hsig = ws[L.hsf:L.hsf + 4 * L.rows_cap].view(torch.float32)[rows].cpu().numpy().reshape(T, rpt)
        self.h = h_pre[rows].cpu().numpy().reshape(T, rpt, cfg.I)
        del out, h_pre, layer


def _fp8_task(args):
    cfg, which, e = args
    codes, scales = synth.gen_mx_weight(cfg, which, e)
    return (which, e), W8.converted_weight(codes, scales)


def _prefetch(ws, cfg, keys):
    import multiprocessing as mp
    keys = [k for k in keys if k not in ws._cache]
    if len(keys) < 4:
        return
    with mp.get_context("spawn").Pool(min(16, len(keys))) as pool:
        for key, val in pool.imap_unordered(_fp8_task, [(cfg, w, e) for w, e in keys]):
            ws._cache[key] = val


def check8(cfg, tokens):
    run = Run8(cfg)
    assert run.status == (0, 0), run.status
    tokens = np.asarray(tokens)
    xr = np.concatenate([synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg, int(t), int(t) + 1)) for t in tokens])
    assert np.array_equal(synth.to_bf16_bits(xr), run.x_bits[tokens])
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    b = synth.gen_bias_f32(cfg)
    ws = W8.fp8_weight_source(cfg)
    need = sorted({int(e) for t in tokens for e in run.idx[t]})
    keys = [(w, e) for e in need for w in ("w13", "w2")] + [(w, 0) for w in ("sh13", "sh2")][:2 * cfg.n_shared]
    _prefetch(ws, cfg, keys)
    orc = W8.token_forward_fp8(cfg, xr, wr, b, ws)
    orc["bias"] = b
    x_all = synth.bf16_bits_to_f64(run.x_bits)
    exact, lsum = R.router_logits(x_all, wr)
    check_router_numerics(run, cfg, exact, lsum)
    check_selection_replay(run, cfg, b)
    amb = check_routing(run, cfg, orc, tokens)
    check_permutation(run, cfg)
    stats = {"ambiguous_tokens": len(amb), "h_flips": 0, "h_ambiguous": 0, "h_err_ratio": 0.0}
    for i, t in enumerate(tokens):
        # activations: the token's codes and scale in every one of its route rows
        for j in range(cfg.top_k + cfg.n_shared):
            assert np.array_equal(run.xq[t, j], orc["xc"][i]), (t, j)
            assert run.xsig[t, j] == orc["xsig"][i], (t, j, run.xsig[t, j], orc["xsig"][i])
        if int(t) in amb:
            continue
        for j, info in enumerate(orc["routes"][i]):
            jj = j if j >= cfg.top_k else int(np.flatnonzero(run.idx[t] == info["expert"])[0])
            err = np.abs(run.h[t, jj].astype(np.float64) - info["h"][0])
            ratio = float(np.max(err / info["dh"][0]))
            stats["h_err_ratio"] = max(stats["h_err_ratio"], ratio)
            assert ratio <= 1.0, (t, j, ratio)
            s_lo, s_hi = info["scale_range"]
            assert s_lo[0] <= run.hsig[t, jj] <= s_hi[0], (t, j, run.hsig[t, jj], s_lo[0], s_hi[0])
            gpu_hd = F.E4M3_TABLE[run.hq[t, jj]] * float(run.hsig[t, jj])
            ref_hd = W8.fp8_dequant(info["hq"][0], info["hsig"][0])
            diff = np.abs(gpu_hd - ref_hd)
            assert np.all(diff <= info["dmax"][0] * (1 + 1e-12)), (t, j, float(np.max(diff - info["dmax"][0])))
            stats["h_flips"] += int(np.count_nonzero(diff))
            stats["h_ambiguous"] += int(np.count_nonzero(info["dmax"][0]))
            # replay: the oracle's quantiser on the GPU's own h gives exactly
            # the GPU's codes and row scale
            rq, rsig = W8.fp8_quantize(run.h[t, jj].astype(np.float64)[None])
            assert np.array_equal(rq[0], run.hq[t, jj]) and rsig[0] == run.hsig[t, jj], (t, j)
    stats["worst_ratio"] = check_output(run, orc["ref"], orc["S"], orc["A"], tokens, amb)
    # replay: the oracle's down projection and combine on the GPU's quantised
    # intermediate meets the tolerance with no allowance for flips
    # (with the GPU's routing, so every token is checked)
    ref2 = np.zeros_like(orc["ref"])
    S2 = np.zeros_like(orc["ref"])
    for i, t in enumerate(tokens):
        for j in range(cfg.top_k + cfg.n_shared):
            e = int(run.idx[t, j]) if j < cfg.top_k else cfg.E + j - cfg.top_k
            W2 = ws.get("w2", e) if e < cfg.E else ws.get("sh2", e - cfg.E)
            hd = F.E4M3_TABLE[run.hq[t, j]] * float(run.hsig[t, j])
            wt = float(run.w[t, j]) if j < cfg.top_k else 1.0
            ref2[i] += wt * (hd @ W2.T)
            S2[i] += abs(wt) * (np.abs(hd) @ np.abs(W2).T)
    stats["worst_ratio_replayed"] = check_output(run, ref2, S2, np.zeros_like(ref2), tokens)
    return stats


@pytest.mark.parametrize("name", ["tiny", "tiny_T1", "ragged_shared", "wide_padK"])
def test_small_layers_w8a8(name):
    cfg = SMALL[name]
    print(name, check8(cfg, np.arange(cfg.T)))


def test_kimi_decode_w8a8_full_size():
    print(check8(synth.configs()["kimi_decode"], [0, 5]))


def test_kimi_prefill_w8a8_full_size():
    print(check8(synth.configs()["kimi_prefill"], [0, 4095]))
