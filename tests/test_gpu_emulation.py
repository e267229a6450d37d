"""GPU parity of fp4moe_forward_nvfp4_emulated (the NVFP4 layer in emulation
mode: BF16 dequantised experts, NVFP4 QDQ activations and intermediate, BF16
GEMMs with fp32 accumulation) against the emulation oracle:
  1. routing and permutation;
  2. the BF16 activation rows bit-exact, in every route row of a token, and
     the tensor scale of x bit-exact;
  3. the intermediate h within its error bound before the round trip, the
     per-expert tensor scale of h within the range that bound admits, and
     its BF16 values equal to the oracle's wherever no other NVFP4
     quantisation is admissible (else within the allowance);
  4. the layer output within |gpu - ref| <= 2^-8 |ref| + 1e-3 S + A.
Small layers check every token; the DeepSeek-shaped layer (T = 512), in the
benchmark's launch configuration, checks sampled tokens."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import emulation as EM
from oracle import inputs as OI
from oracle import quant as Q

from gpu_util import ensure_built, torch_cuda
from test_gpu_forward import SMALL, check_output, check_permutation, check_routing

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
        out = layer.forward_emulated(x, debug=dbg)
        torch.cuda.synchronize()
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


def check_em(cfg, tokens, packed=True):
    run = RunEm(cfg, packed)
    assert run.status == (0, 0), run.status
    x, wr, b = OI.layer_inputs(cfg)
    assert np.array_equal(run.x_bits, synth.gen_x_bf16(cfg))
    ws = OI.oracle_weights(cfg)
    tokens = np.asarray(tokens)
    if cfg.H * cfg.I >= 1 << 22:  # large weights: quantise them in a spawn pool
        need = sorted({int(e) for t in tokens for e in run.idx[t]})
        keys = [(w, e) for e in need for w in ("w13", "w2")] + [(w, 0) for w in ("sh13", "sh2")][:2 * cfg.n_shared]
        OI.prefetch(ws, cfg, keys)
    orc = EM.emulated_layer_forward(cfg, x, wr, b, ws, tokens=tokens)
    sel = {"logits": orc["logits"][tokens], "lsum": orc["lsum"][tokens],
           "margins": [orc["margins"][t] for t in tokens], "idx": orc["idx"][tokens], "w": orc["w"][tokens]}
    amb = check_routing(run, cfg, sel, tokens)
    check_permutation(run, cfg)
    assert run.gx == orc["gx"]
    for t in tokens:
        for j in range(cfg.top_k + cfg.n_shared):
            assert np.array_equal(run.xb[t, j], orc["a"][t]), (t, j)
    stats = {"ambiguous_tokens": len(amb), "h_flips": 0, "h_ambiguous": 0, "h_err_ratio": 0.0}
    if not amb:  # a re-routed token would change its experts' tensor scales of h
        for e, info in orc["experts"].items():
            # the tensor scale of h follows the |max| of the expert's fp32 h:
            # any value its error bound admits
            g_lo = Q.nv_global_scale(float(np.max(np.maximum(np.abs(info["h32"]) - info["dh"], 0.0))))
            g_hi = Q.nv_global_scale(float(np.max(np.abs(info["h32"]) + info["dh"])))
            assert g_lo <= run.gh[e] <= g_hi, (e, run.gh[e], g_lo, g_hi)
            for r, (t, sl) in enumerate(zip(info["tok"], info["slot"])):
                if int(t) not in set(tokens.tolist()):
                    continue
                # the route's column: its expert's place among the token's
                # choices, or (shared expert) its slot after them
                jj = int(np.flatnonzero(run.idx[t] == e)[0]) if e < cfg.E else int(sl)
                err = np.abs(run.h[t, jj].astype(np.float64) - info["h"][r])
                ratio = float(np.max(err / info["dh"][r]))
                stats["h_err_ratio"] = max(stats["h_err_ratio"], ratio)
                assert ratio <= 1.0, (t, e, ratio)
                diff = np.abs(run.hb[t, jj] - info["hd"][r])
                assert np.all(diff <= info["dmax"][r] * (1 + 1e-12)), (t, e, float(np.max(diff - info["dmax"][r])))
                stats["h_flips"] += int(np.count_nonzero(diff))
                stats["h_ambiguous"] += int(np.count_nonzero(info["dmax"][r]))
    stats["worst_ratio"] = check_output(run, orc["ref"], orc["S"], orc["A"], tokens, amb)
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
