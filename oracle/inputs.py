"""Oracle-side view of the synthetic layer inputs (test infrastructure only).

Draws every input from ``synth`` (no arithmetic of the method there) and, for
the NVFP4 configuration, quantises the bf16 expert weights with the oracle's
own NVFP4 quantiser: one tensor scale per (expert, weight tensor).
"""
from __future__ import annotations

import numpy as np

import synth

from . import quant as Q
from .formats import unpack_nibbles
from .moe import WeightSource


def oracle_weights(cfg) -> WeightSource:
    def fn(which, e):
        if cfg.fmt == "mxfp4":
            codes, scales = synth.gen_mx_weight(cfg, which, e)
            return unpack_nibbles(codes), scales, None
        wb = synth.bf16_bits_to_f64(synth.gen_bf16_weight(cfg, which, e))
        c, s, g = Q.nv_quantize(wb)
        return c, s, g
    return WeightSource(fn)


def layer_inputs(cfg):
    """(x values [T, H] f64, Wr values [E, H] f64, bias f32 [E])."""
    x = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg))
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    return x, wr, synth.gen_bias_f32(cfg)
