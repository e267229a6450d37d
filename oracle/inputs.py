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


def expert_weight(cfg, which, e):
    """(codes unpacked, scale bytes, tensor scale or None) of one expert tensor."""
    if cfg.fmt == "mxfp4":
        codes, scales = synth.gen_mx_weight(cfg, which, e)
        return unpack_nibbles(codes), scales, None
    wb = synth.bf16_bits_to_f64(synth.gen_bf16_weight(cfg, which, e))
    c, s, g = Q.nv_quantize(wb)
    return c, s, g


def _expert_weight_task(args):
    return args[1:], expert_weight(*args)


def oracle_weights(cfg) -> WeightSource:
    return WeightSource(lambda which, e: expert_weight(cfg, which, e))


def prefetch(ws: WeightSource, cfg, keys, processes: int = 8):
    """Fills the cache of ``ws`` for (which, e) keys in a process pool started
    with 'spawn' (safe after CUDA has been initialised in this process)."""
    import multiprocessing as mp
    keys = [k for k in keys if k not in ws._cache]
    if not keys:
        return
    with mp.get_context("spawn").Pool(min(processes, len(keys))) as pool:
        for key, val in pool.imap_unordered(_expert_weight_task, [(cfg, w, e) for w, e in keys]):
            ws._cache[tuple(key)] = val


def layer_inputs(cfg):
    """(x values [T, H] f64, Wr values [E, H] f64, bias f32 [E])."""
    x = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg))
    wr = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    return x, wr, synth.gen_bias_f32(cfg)
