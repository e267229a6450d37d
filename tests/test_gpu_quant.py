"""GPU parity of fp4moe_quantize_act (MXFP4 and NVFP4, bf16 and fp32 inputs)
and of the seeded device generator, bit for bit against the oracle / host."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import formats as F
from oracle import quant as Q

from gpu_util import ensure_built, torch_cuda

pytestmark = pytest.mark.gpu


def _edge_values(rows, cols, rng, src):
    v = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-20, 20, (rows, 1)))
    v[0] = 0.0
    v[1] = -0.0
    # exact E2M1 midpoints under a block maximum of 6 * 2^e
    mids = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, 0.1,
                     -0.1, 4, 3, 2, 1.5, 1, 0.5, 0, -0.0, 6, -6, 5.5, 4.5, 2.25, 0.3, 0.2])
    for r in (2, 3):
        v[r] = np.tile(mids, cols // 32) * 2.0 ** (r * 5 - 12)
    v[4] = 2.0 ** -133 * (1 + np.arange(cols) % 7)  # bf16 / fp32 subnormals
    v[5] = 3.0e38 * np.sign(rng.standard_normal(cols))
    v[6, :16] = 1000.0  # NVFP4 block scale saturates at 448
    if src == "bf16":
        bits = synth.to_bf16_bits(v)
        return bits, synth.bf16_bits_to_f64(bits)
    f = v.astype(np.float32)
    return f, f.astype(np.float64)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
@pytest.mark.parametrize("src", ["bf16", "fp32"])
@pytest.mark.parametrize("rows,cols", [(37, 512), (1, 32), (300, 7168)])
def test_quantize_act_bit_exact(fmt, src, rows, cols):
    torch = torch_cuda()
    ensure_built()
    rng = np.random.default_rng(rows * 7 + cols)
    rows_eff = max(rows, 8)
    host, vals = _edge_values(rows_eff, cols, rng, src)
    host, vals = host[:rows], vals[:rows]
    nv = fmt == "nvfp4"
    blk = 16 if nv else 32
    x = torch.from_numpy(host.view(np.int16) if src == "bf16" else host).cuda()
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // blk), dtype=torch.uint8, device="cuda")
    g_out = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    fm.quantize_act(x.data_ptr(), src == "fp32", rows, cols, fm.NVFP4 if nv else fm.MXFP4, None, codes.data_ptr(),
                    scales.data_ptr(), g_out.data_ptr(), ws.data_ptr(), 256)
    torch.cuda.synchronize()
    if nv:
        c, s, g = Q.nv_quantize(vals)
        assert g_out.item() == g
    else:
        c, s = Q.mx_quantize(vals)
    assert np.array_equal(codes.cpu().numpy(), F.pack_nibbles(c))
    assert np.array_equal(scales.cpu().numpy(), s)


def test_nvfp4_given_tensor_scale():
    torch = torch_cuda()
    ensure_built()
    rng = np.random.default_rng(5)
    v = rng.standard_normal((16, 256)).astype(np.float32)
    g = np.float32(0.00123)
    x = torch.from_numpy(v).cuda()
    gi = torch.tensor([g], dtype=torch.float32, device="cuda")
    codes = torch.empty((16, 128), dtype=torch.uint8, device="cuda")
    scales = torch.empty((16, 16), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    fm.quantize_act(x.data_ptr(), True, 16, 256, fm.NVFP4, gi.data_ptr(), codes.data_ptr(), scales.data_ptr(), None,
                    ws.data_ptr(), 256)
    c, s, _ = Q.nv_quantize(v.astype(np.float64), g)
    assert np.array_equal(codes.cpu().numpy(), F.pack_nibbles(c))
    assert np.array_equal(scales.cpu().numpy(), s)


def test_device_generator_matches_host():
    torch = torch_cuda()
    ensure_built()
    cfg = synth.configs()["kimi_decode"]
    n = 1 << 20
    b = torch.empty(n, dtype=torch.uint8, device="cuda")
    synth.dev_uniform_bytes(cfg.seed, synth.S_W13, 8 * 1000, b)
    assert np.array_equal(b.cpu().numpy(), synth.uniform_bytes(cfg.seed, synth.S_W13, 8 * 1000, n))
    s = torch.empty((300, 224), dtype=torch.uint8, device="cuda")
    synth.dev_e8m0_scales(cfg.seed, synth.S_W13S, 4096 * 5, 300, 224, s)
    assert np.array_equal(s.cpu().numpy(), synth.e8m0_scales(cfg.seed, synth.S_W13S, 4096 * 5, 300, 224))
    x = torch.empty((3, cfg.H), dtype=torch.int16, device="cuda")
    synth.dev_normal_bf16(cfg.seed, synth.S_X, 2 * cfg.H, x, 1.0)
    assert np.array_equal(x.cpu().numpy().view(np.uint16), synth.gen_x_bf16(cfg, 2, 5))
