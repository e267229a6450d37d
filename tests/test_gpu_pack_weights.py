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
