"""GPU parity of fp4moe_linear (dense block-scaled FP4 linear: bf16 x
quantised on the fly, block-scaled FP4 product, bf16 out) against the FP64
oracle: |gpu - y| <= 2^-8 |y| + 1e-3 sum_k |a_k W_k| per element.  Shapes from
one token to a 4096 x 7168 x 7168 projection (sampled rows), MXFP4 and
NVFP4; seeded numpy inputs (MXFP4 weights: uniform codes with E8M0 scales of
the synthetic recipe; NVFP4: bf16 N(0, 0.02) weights quantised by the
oracle)."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
from oracle import formats as F
from oracle import linear as LIN
from oracle import quant as Q

from gpu_util import ensure_built, torch_cuda

pytestmark = pytest.mark.gpu


def _bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)


def _inputs(T, K, N, fmt, seed):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((T, K)))
    if fmt == "mxfp4":
        codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
        scales = (127 + rng.integers(-10, -5, size=(N, 1))
                  - rng.choice([0, 1, 2], size=(N, K // 32), p=[.7, .25, .05])).astype(np.uint8)
        return x, codes, scales, None
    wb = _bf16(rng.standard_normal((N, K)) * 0.02)
    c, s, g = Q.nv_quantize(wb)
    return x, c, s, g


def _run(T, K, N, fmt, seed, rows):
    torch = torch_cuda()
    ensure_built()
    x, wc, ws, gw = _inputs(T, K, N, fmt, seed)
    f = fm.NVFP4 if fmt == "nvfp4" else fm.MXFP4
    blk = 16 if fmt == "nvfp4" else 32
    xd = torch.from_numpy(x.astype(np.float32)).cuda().to(torch.bfloat16)
    wd = torch.from_numpy(F.pack_nibbles(wc)).cuda()
    raw = torch.from_numpy(np.ascontiguousarray(ws)).cuda()
    sf = torch.empty(fm.packed_scales_bytes(1, N, K // blk, f), dtype=torch.uint8, device="cuda")
    fm.pack_scales(raw.data_ptr(), sf.data_ptr(), 1, N, K // blk, f)
    g = torch.tensor([gw], dtype=torch.float32, device="cuda") if gw is not None else None
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    n = fm.linear_workspace_size(f, T, K, N)
    wsp = torch.empty(n, dtype=torch.uint8, device="cuda")
    fm.linear(f, T, K, N, xd.data_ptr(), wd.data_ptr(), sf.data_ptr(), g.data_ptr() if g is not None else None,
              out.data_ptr(), wsp.data_ptr(), n)
    torch.cuda.synchronize()
    assert fm.get_status(wsp.data_ptr()) == (0, 0)
    got = out.float().cpu().numpy().astype(np.float64)[rows]
    if fmt == "nvfp4":  # the tensor scale of x is over all rows; quantise the sampled rows with it
        gx = Q.nv_global_scale(np.max(np.abs(x)))
        xc, xs, _ = Q.nv_quantize(x[rows], gx)
        a = Q.nv_dequant(xc, xs, gx)
        W = Q.nv_dequant(wc, ws, gw)
        y, S = a @ W.T, np.abs(a) @ np.abs(W).T
    else:
        y, S, _ = LIN.linear_forward(x[rows], wc, ws, fmt)
    ratio = np.abs(got - y) / LIN.tolerance(y, S)
    assert np.all(ratio <= 1), (float(ratio.max()), np.argwhere(ratio > 1)[:5])
    return float(ratio.max())


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
@pytest.mark.parametrize("T,K,N", [(1, 256, 256), (37, 512, 768), (300, 1024, 512), (129, 2048, 1280)])
def test_linear_small(T, K, N, fmt):
    print(T, K, N, fmt, _run(T, K, N, fmt, seed=T + K + N, rows=np.arange(T)))


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_linear_projection_full_size(fmt):
    rows = np.array([0, 1, 2047, 4000, 4095])
    print(fmt, _run(4096, 7168, 7168, fmt, seed=11, rows=rows))
