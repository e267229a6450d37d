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


def test_gateup_paired_formulas_in_the_header_match_the_layouts():
    """The byte-offset formulas fp4moe.h prints for fp4moe_pack_gateup_weights
    and fp4moe_pack_gateup_scales equal their definitions: the blocks (and the
    scale groups) of the plain tiled layouts, reordered per matrix by (gate/up
    pair, K tile, gate before up), written as numpy reshapes."""
    import numpy as np
    rng = np.random.default_rng(11)
    for n_mat, I, kbytes in ((2, 128, 192), (1, 384, 512), (3, 256, 16)):
        P, kt = I // 128, -(-kbytes // 128)
        src = rng.integers(0, 256, (n_mat, 2 * I, kbytes), dtype=np.uint8)
        pad = np.zeros((n_mat, 2 * I, kt * 128), dtype=np.uint8)
        pad[..., :kbytes] = src
        # [m, h, p, 128 rows, kt, 128 bytes] -> [m, p, kt, h, 128, 128]
        paired = pad.reshape(n_mat, 2, P, 128, kt, 128).transpose(0, 2, 4, 1, 3, 5).reshape(-1)
        m, r, c = np.meshgrid(np.arange(n_mat), np.arange(2 * I), np.arange(kbytes), indexing="ij")
        h, p = (r // 128) // P, (r // 128) % P
        off = m * 2 * I * kt * 128 + ((p * kt + c // 128) * 2 + h) * 16384 + (r % 128) * 128 + c % 128
        assert np.array_equal(paired[off], src)
    for n_mat, I, kblocks, A in ((2, 128, 8, 2), (1, 384, 24, 2), (2, 256, 16, 4)):
        P = I // 128
        katoms = -(-kblocks // (4 * A)) * A
        kt = katoms // A
        groups = rng.integers(0, 256, (n_mat, 2 * P, katoms, 512), dtype=np.uint8)  # plain tiled groups
        # [m, h, p, kt, a, 512] -> [m, p, kt, h, a, 512]
        paired = groups.reshape(n_mat, 2, P, kt, A, 512).transpose(0, 2, 3, 1, 4, 5).reshape(-1)
        for mm in range(n_mat):
            for rt in range(2 * P):
                hh, pp = rt // P, rt % P
                for k in range(kt):
                    for a in range(A):
                        off = ((((mm * P + pp) * kt + k) * 2 + hh) * A + a) * 512
                        assert np.array_equal(paired[off:off + 512], groups[mm, rt, k * A + a])


def _noalloc_scratch_formula(d, route_splits):
    """Scratch bytes of fp4moe_route_noalloc as the header states them: a
    256-byte status word, ceil(T/32) * (E + n_shared) * 4 bytes of counts
    rounded up to 256, then n_splits * T * E * 4 bytes of partial logits, with
    the largest split count up to fp4moe_route's that divides H / 256 and fits."""
    counts = (d.T + 31) // 32 * (d.E + d.n_shared) * 4
    limit = 8 << 20
    for s in range(route_splits, 0, -1):
        if (d.H // 256) % s == 0:
            n = 256 + (counts + 255) // 256 * 256 + s * d.T * d.E * 4
            if n <= limit:
                return n
    return 0


@pytest.mark.parametrize("E,H", [(384, 7168), (512, 7168), (256, 2048)])
def test_noalloc_limit_from_header_formula(lib, E, H):
    """The accept / refuse decision of fp4moe_route_noalloc at the edge of
    its fixed scratch array follows the header's formula: the largest T that
    fits is accepted (and fails only later, for want of a device here), the
    next one is refused with FP4MOE_ERR_WORKSPACE before any device work.
    The accepted call is made only where no CUDA device is present (its
    pointers are placeholders)."""
    def dims(T):
        return fm.make_dims(T, H, 256, E, 8)

    def fits(T):
        d = dims(T)
        return _noalloc_scratch_formula(d, fm.workspace_layout(d).n_splits) > 0

    lo, hi = 1, 65536
    assert fits(lo) and not fits(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if fits(mid) else (lo, mid)
    import torch
    for T, ok in ((lo, True), (hi, False)):
        d = dims(T)
        want = _noalloc_scratch_formula(d, fm.workspace_layout(d).n_splits)
        assert fm.route_noalloc_scratch_bytes(d) == want and (want > 0) == ok
        if ok and torch.cuda.is_available():
            continue  # with a device the accepted call would launch on these placeholder pointers
        code = lib.fp4moe_route_noalloc(ctypes.byref(d), 256, 256, 256, 256, 256, None, None)
        assert code == (fm.STATUS_CODE["FP4MOE_ERR_DEVICE"] if ok else fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]), (T, code)


def test_short_workspace_refused_before_device_work(lib):
    """A workspace one byte short of fp4moe_workspace_size is refused with
    FP4MOE_ERR_WORKSPACE before anything is launched (placeholder pointers,
    never dereferenced), for every layer entry point that takes one."""
    d = fm.make_dims(4, 256, 128, 8, 2)
    n = fm.workspace_size(d)
    w = fm.Weights(*([256] * 12), 1)
    code = lib.fp4moe_forward(ctypes.byref(d), ctypes.byref(w), 256, 256, None, 256, n - 1, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]
    code = lib.fp4moe_forward_cols(ctypes.byref(d), ctypes.byref(w), 256, 256, 0, 128, None, 256, n - 1, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]
    code = lib.fp4moe_route(ctypes.byref(d), 256, 256, 256, 256, 256, None, 256, n - 1, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]
    d8 = fm.make_dims(4, 256, 128, 8, 2, fmt=fm.FP8)
    w8 = fm.Fp8Weights(*([256] * 10))
    code = lib.fp4moe_forward_w8a8(ctypes.byref(d8), ctypes.byref(w8), 256, 256, None, 256,
                                   fm.workspace_size(d8) - 1, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]
    dn = fm.make_dims(4, 256, 128, 8, 2, fmt=fm.NVFP4)
    code = lib.fp4moe_forward_nvfp4_emulated(ctypes.byref(dn), ctypes.byref(w), 256, 256, None, 256,
                                             fm.emulation_workspace_size(dn) - 1, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]
    n_lin = fm.linear_workspace_size(fm.MXFP4, 4, 256, 256)
    code = lib.fp4moe_linear(fm.MXFP4, 4, 256, 256, 256, 256, 256, None, 256, 256, n_lin - 1, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]
    code = lib.fp4moe_check_scales(256, 64, fm.MXFP4, 256, 255, None)
    assert code == fm.STATUS_CODE["FP4MOE_ERR_WORKSPACE"]


def test_check_scales_argument_errors(lib):
    assert lib.fp4moe_check_scales(None, 64, fm.MXFP4, 256, 256, None) == fm.STATUS_CODE["FP4MOE_ERR_INVALID_ARG"]
    assert lib.fp4moe_check_scales(256, 64, 7, 256, 256, None) == fm.STATUS_CODE["FP4MOE_ERR_INVALID_ARG"]
    assert lib.fp4moe_check_scales(256, -1, fm.MXFP4, 256, 256, None) == fm.STATUS_CODE["FP4MOE_ERR_INVALID_ARG"]
