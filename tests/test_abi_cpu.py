"""The C-ABI library builds, loads and exports every function the header
declares; host-side entry points (workspace sizing, layout) answer without a
GPU.  No compute entry point is called here."""
import ctypes

import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
from block_scaled_fp4_sigmoid_gb300 import build
import synth


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return fm.lib()


def test_exports_every_header_function(lib):
    names = fm.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_version(lib):
    assert fm.version() >= 100


@pytest.mark.parametrize("name", list(synth.configs()))
def test_workspace_sizes(lib, name):
    cfg = synth.configs()[name]
    fmt = fm.NVFP4 if cfg.fmt == "nvfp4" else fm.MXFP4
    d = fm.make_dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.n_shared,
                     cfg.routed_scaling, 1, fmt)
    n = fm.workspace_size(d)
    L = fm.workspace_layout(d)
    assert n == L.total_bytes > 0
    offs = [L.status, L.logits, L.topk_idx, L.topk_w, L.expert_count, L.expert_slot, L.route_row, L.row_tok,
            L.row_w, L.xq, L.xsf, L.hq, L.hsf, L.gscale, L.out_acc]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and offs[-1] + cfg.T * cfg.H * 4 <= n
    R = cfg.T * (cfg.top_k + cfg.n_shared)
    assert L.rows_cap >= 128 * (R // L.n_tile + 1)
    assert cfg.H // 256 % L.n_splits == 0
    # few-token MXFP4 forwards quantise x once per token (token rows)
    assert L.x_by_token == int(cfg.fmt == "mxfp4" and cfg.T <= 16)


@pytest.mark.parametrize("bad", [dict(T=0), dict(H=200), dict(I=100), dict(E=0), dict(top_k=0), dict(n_shared=2),
                                 dict(n_group=3), dict(fmt=5), dict(top_k=9, E=8)])
def test_invalid_dims_rejected(lib, bad):
    kw = dict(T=4, H=256, I=128, E=8, top_k=2)
    kw.update(bad)
    fmt = kw.pop("fmt", fm.MXFP4)
    d = fm.make_dims(**kw, fmt=fmt)
    assert lib.fp4moe_workspace_size(ctypes.byref(d)) == 0
    with pytest.raises(fm.Fp4MoeError):
        fm.workspace_layout(d)


def test_packed_scale_sizes(lib):
    assert fm.packed_scales_bytes(384, 4096, 224, fm.MXFP4) == 384 * 32 * 56 * 512
    assert fm.packed_scales_bytes(1, 128, 4, fm.MXFP4) == 2 * 512   # padded to a whole K tile
    assert fm.packed_scales_bytes(1, 128, 8, fm.NVFP4) == 4 * 512
    assert fm.packed_scales_bytes(1, 100, 8, fm.MXFP4) == 0


def test_packed_weight_sizes(lib):
    # rows padded to nothing (multiples of 128 required), K to whole 128-byte tiles
    assert fm.packed_weights_bytes(384, 4096, 3584) == 384 * 4096 * 3584
    assert fm.packed_weights_bytes(2, 256, 192) == 2 * 256 * 256
    assert fm.packed_weights_bytes(1, 100, 128) == 0
    assert fm.packed_weights_bytes(1, 128, 24) == 0  # rows of 16-byte multiples only
    # unsupported shapes and null pointers are refused before any device work
    assert lib.fp4moe_pack_weights(None, None, 1, 128, 128, None) == 1
    buf = ctypes.create_string_buffer(256)
    assert lib.fp4moe_pack_weights(buf, buf, 1, 100, 128, None) == 2


def test_group_of_one_expert_is_refused(lib):
    # a group's score sums its two largest corrected scores: groups of one
    # expert are outside the supported shapes, two are inside
    assert lib.fp4moe_workspace_size(ctypes.byref(fm.make_dims(4, 256, 128, 8, 2, n_group=8, topk_group=4))) == 0
    assert lib.fp4moe_workspace_size(ctypes.byref(fm.make_dims(4, 256, 128, 8, 2, n_group=4, topk_group=2))) > 0


def test_argument_errors_need_no_gpu(lib):
    d = fm.make_dims(4, 256, 128, 8, 2)
    # null pointers are refused before any device work
    assert lib.fp4moe_forward(ctypes.byref(d), None, None, None, None, None, 0, None) == 1
    assert lib.fp4moe_quantize_act(None, 0, 4, 64, 0, None, None, None, None, None, 0, None) == 1
    assert lib.fp4moe_mxfp4_to_fp8_rowscale(None, None, 1, 32, None, None, None, None, 0, None) == 1
    assert lib.fp4moe_status_string(5) == b"device wait timed out"


def test_synth_device_library_builds():
    so = synth.build_device_lib()
    lib = ctypes.CDLL(str(so))
    for n in ("synth_words", "synth_e8m0", "synth_normal_bf16"):
        assert hasattr(lib, n)


def test_tiled_payload_formula_in_the_header_matches_the_layout():
    """The byte-offset formula fp4moe.h prints for fp4moe_pack_weights equals
    the layout's definition (blocks of 128 rows x 128 bytes, K tiles
    innermost, K zero-padded), written as a numpy reshape."""
    import numpy as np
    rng = np.random.default_rng(7)
    for n_mat, rows, kbytes in ((2, 256, 192), (1, 384, 3584), (3, 128, 16)):
        kt = -(-kbytes // 128)
        src = rng.integers(0, 256, (n_mat, rows, kbytes), dtype=np.uint8)
        pad = np.zeros((n_mat, rows, kt * 128), dtype=np.uint8)
        pad[..., :kbytes] = src
        tiled = pad.reshape(n_mat, rows // 128, 128, kt, 128).transpose(0, 1, 3, 2, 4).reshape(-1)
        m, r, c = np.meshgrid(np.arange(n_mat), np.arange(rows), np.arange(kbytes), indexing="ij")
        off = m * rows * kt * 128 + ((r // 128) * kt + c // 128) * 16384 + (r % 128) * 128 + c % 128
        assert np.array_equal(tiled[off], src)
        assert tiled.size == fm.packed_weights_bytes(n_mat, rows, kbytes)
