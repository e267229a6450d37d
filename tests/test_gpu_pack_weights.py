"""fp4moe_pack_weights: the tiled payload layout, bit for bit against the
layout's definition (numpy reshape of the zero-padded row-major array)."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm

from gpu_util import ensure_built, torch_cuda

pytestmark = pytest.mark.gpu


def tiled_reference(src: np.ndarray, kbytes: int) -> np.ndarray:
    """Per matrix, 128-row tile and 128-byte K tile (K tile innermost), one
    block of 128 rows x 128 bytes; K padded with zero codes."""
    n_mat, rows, _ = src.shape
    kt = -(-kbytes // 128)
    pad = np.zeros((n_mat, rows, kt * 128), dtype=np.uint8)
    pad[..., :kbytes] = src
    return pad.reshape(n_mat, rows // 128, 128, kt, 128).transpose(0, 1, 3, 2, 4).reshape(-1)


@pytest.mark.parametrize("n_mat,rows,kbytes", [(1, 128, 128), (3, 256, 192), (2, 384, 3584), (5, 128, 16),
                                               (1, 7168, 1024)])
def test_pack_weights_bit_exact(n_mat, rows, kbytes):
    torch = torch_cuda()
    ensure_built()
    rng = np.random.default_rng(n_mat * 1000 + rows + kbytes)
    src = rng.integers(0, 256, (n_mat, rows, kbytes), dtype=np.uint8)
    nbytes = fm.packed_weights_bytes(n_mat, rows, kbytes)
    assert nbytes == n_mat * rows * (-(-kbytes // 128)) * 128
    d_src = torch.from_numpy(src).cuda()
    d_dst = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    fm.pack_weights(d_src.data_ptr(), d_dst.data_ptr(), n_mat, rows, kbytes)
    torch.cuda.synchronize()
    assert np.array_equal(d_dst.cpu().numpy(), tiled_reference(src, kbytes))


def paired_reference(src: np.ndarray, kbytes: int) -> np.ndarray:
    """Gate/up-paired order: the blocks of tiled_reference, per matrix ordered
    by pair p (row tiles p and p + I/128), K tile, then gate before up."""
    n_mat, rows, _ = src.shape
    P, kt = rows // 256, -(-kbytes // 128)
    pad = np.zeros((n_mat, rows, kt * 128), dtype=np.uint8)
    pad[..., :kbytes] = src
    return pad.reshape(n_mat, 2, P, 128, kt, 128).transpose(0, 2, 4, 1, 3, 5).reshape(-1)


@pytest.mark.parametrize("n_mat,I,kbytes", [(1, 128, 128), (3, 128, 192), (2, 384, 3584), (5, 256, 16)])
def test_pack_gateup_weights_bit_exact(n_mat, I, kbytes):
    torch = torch_cuda()
    ensure_built()
    rng = np.random.default_rng(n_mat * 7 + I + kbytes)
    src = rng.integers(0, 256, (n_mat, 2 * I, kbytes), dtype=np.uint8)
    nbytes = fm.packed_weights_bytes(n_mat, 2 * I, kbytes)
    d_src = torch.from_numpy(src).cuda()
    d_dst = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    fm.pack_gateup_weights(d_src.data_ptr(), d_dst.data_ptr(), n_mat, I, kbytes)
    torch.cuda.synchronize()
    assert np.array_equal(d_dst.cpu().numpy(), paired_reference(src, kbytes))


def tiled_scales_reference(raw: np.ndarray, apk: int, pad: int) -> np.ndarray:
    """The plain tiled scale layout from its definition: per matrix, 128-row
    tile and group of four blocks (padded to whole K tiles of apk groups),
    512 bytes with row r = 32*m1 + m0 and block k1 at 16*m0 + 4*m1 + k1."""
    n_mat, rows, kblocks = raw.shape
    katoms = -(-kblocks // (4 * apk)) * apk
    padded = np.full((n_mat, rows, katoms * 4), pad, dtype=np.uint8)
    padded[..., :kblocks] = raw
    # [m, rt, m1, m0, atom, k1] -> [m, rt, atom, m0, m1, k1]
    return padded.reshape(n_mat, rows // 128, 4, 32, katoms, 4).transpose(0, 1, 4, 3, 2, 5).reshape(
        n_mat, rows // 128, katoms, 512)


@pytest.mark.parametrize("fmt_name,n_mat,I,K", [("mxfp4", 1, 128, 256), ("mxfp4", 2, 384, 7168), ("mxfp4", 3, 128, 1024),
                                               ("nvfp4", 2, 256, 512), ("nvfp4", 1, 128, 768)])
def test_pack_gateup_scales_bit_exact(fmt_name, n_mat, I, K):
    torch = torch_cuda()
    ensure_built()
    fmt = fm.MXFP4 if fmt_name == "mxfp4" else fm.NVFP4
    blk, apk, pad = (32, 2, 127) if fmt_name == "mxfp4" else (16, 4, 0x38)
    kblocks = K // blk
    rng = np.random.default_rng(n_mat + I + K)
    raw = rng.integers(0, 255, (n_mat, 2 * I, kblocks), dtype=np.uint8)
    nbytes = fm.packed_scales_bytes(n_mat, 2 * I, kblocks, fmt)
    d_raw = torch.from_numpy(raw).cuda()
    d_plain = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    d_paired = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    fm.pack_scales(d_raw.data_ptr(), d_plain.data_ptr(), n_mat, 2 * I, kblocks, fmt)
    fm.pack_gateup_scales(d_raw.data_ptr(), d_paired.data_ptr(), n_mat, I, kblocks, fmt)
    torch.cuda.synchronize()
    groups = tiled_scales_reference(raw, apk, pad)
    assert np.array_equal(d_plain.cpu().numpy(), groups.reshape(-1))
    P, katoms = I // 128, groups.shape[2]
    paired = groups.reshape(n_mat, 2, P, katoms // apk, apk, 512).transpose(0, 2, 3, 1, 4, 5).reshape(-1)
    assert np.array_equal(d_paired.cpu().numpy(), paired)
