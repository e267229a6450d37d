"""Pins of the NVFP4 emulation oracle: the BF16 rounding against torch's
bfloat16 conversion, the dequantised values against the native NVFP4 values
(within half a BF16 step), a loop-by-loop recomputation of a small emulated
layer, and its gate/up pre-activations against the native layer's (the
operands differ by one BF16 rounding each)."""
from dataclasses import replace
import math

import numpy as np
import torch

import synth
from oracle import emulation as EM
from oracle import inputs as OI
from oracle import moe as M
from oracle import quant as Q


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(4096) * np.exp2(rng.integers(-40, 40, 4096))).astype(np.float32)
    v[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # ties go to even
    want = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(EM.bf16_rne(v), want)


def test_dequantised_weights_are_within_half_a_bf16_step_of_native():
    cfg = replace(synth.configs()["deepseek_nvfp4"], H=256, I=128, E=4)
    c, s, g = OI.expert_weight(cfg, "w13", 1)
    native = Q.nv_dequant(c, s, g)
    em = EM.nv_dequant_bf16(c, s, g)
    assert np.all(np.abs(em - native) <= 2.0 ** -8 * np.abs(native) * (1 + 2 ** -14))
    assert np.array_equal(em == 0, native == 0)


def _small():
    return replace(synth.configs()["deepseek_nvfp4"], name="em_small", T=5, H=256, I=128, E=8, top_k=2,
                   n_group=2, topk_group=1)


def test_emulated_layer_matches_loops():
    cfg = _small()
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    out = EM.emulated_layer_forward(cfg, x, wr, b, ws)
    H, I = cfg.H, cfg.I
    a = out["a"]
    loops = np.zeros((cfg.T, H))
    for e, info in out["experts"].items():
        W13 = EM.nv_dequant_bf16(*ws.get("w13", e))
        W2 = EM.nv_dequant_bf16(*ws.get("w2", e))
        for r, t in enumerate(info["tok"]):
            gate = [math.fsum(a[t, j] * W13[n, j] for j in range(H)) for n in range(I)]
            up = [math.fsum(a[t, j] * W13[I + n, j] for j in range(H)) for n in range(I)]
            h = [float(np.float32(gv / (1 + math.exp(-gv)) * uv)) for gv, uv in zip(gate, up)]
            assert np.array_equal(np.array(h), info["h32"][r])
            hd = info["hd"][r]
            loops[t] += info["wt"][r] * np.array([math.fsum(hd[i] * W2[o, i] for i in range(I)) for o in range(H)])
    np.testing.assert_allclose(out["ref"], loops, rtol=1e-12, atol=1e-15)


def test_emulated_gate_up_is_close_to_native():
    cfg = _small()
    x, wr, b = OI.layer_inputs(cfg)
    ws = OI.oracle_weights(cfg)
    em = EM.emulated_layer_forward(cfg, x, wr, b, ws)
    nat = M.layer_forward(cfg, x, wr, b, ws)
    assert np.array_equal(em["idx"], nat["idx"])
    # each operand is the native value rounded once to bf16 (at most 2^-9
    # relative), so the gate/up pre-activations differ by at most about
    # 2^-8 of sum |a w|
    a_nat = Q.nv_dequant(nat["xc"], nat["xs"], nat["gx"])
    for e, info in em["experts"].items():
        W_em = EM.nv_dequant_bf16(*ws.get("w13", e))
        W_nat = Q.nv_dequant(*ws.get("w13", e))
        toks = info["tok"]
        d = np.abs(em["a"][toks] @ W_em.T - a_nat[toks] @ W_nat.T)
        assert np.all(d <= (2.0 ** -8 + 2.0 ** -16) * (np.abs(a_nat[toks]) @ np.abs(W_nat).T))
