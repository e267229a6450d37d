"""Helpers of the GPU parity tests (no test functions here)."""
from __future__ import annotations

import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


_BUILT = False


def ensure_built():
    global _BUILT
    if not _BUILT:
        from block_scaled_fp4_sigmoid_gb300 import build
        build.build_library()
        synth.build_device_lib()
        _BUILT = True


def dims_of(cfg):
    fmt = fm.NVFP4 if cfg.fmt == "nvfp4" else fm.MXFP4
    return fm.make_dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.n_shared,
                        cfg.routed_scaling, cfg.renormalize, fmt)


def katoms_padded(K: int, nv: bool) -> int:
    """Scale groups (of four blocks) per row group, padded to whole 256-wide K
    tiles: the tiled scale layout documented with fp4moe_pack_scales."""
    return (K + 255) // 256 * (4 if nv else 2)


def read_tiled_scales(buf: np.ndarray, rows: np.ndarray, kblocks: int, katoms: int) -> np.ndarray:
    """Scale bytes [len(rows), kblocks] of the given rows from a buffer in the
    tiled layout: row r, block kb at ((r/128)*katoms + kb/4)*512 + 16*(r%32)
    + 4*((r/32)%4) + kb%4."""
    rows = np.asarray(rows, dtype=np.int64)[:, None]
    kb = np.arange(kblocks, dtype=np.int64)[None, :]
    off = ((rows >> 7) * katoms + (kb >> 2)) * 512 + 16 * (rows & 31) + 4 * ((rows >> 5) & 3) + (kb & 3)
    return buf[off]


def to_np(t):
    return t.detach().cpu().numpy()
