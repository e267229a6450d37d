"""GPU parity of the exact MXFP4 -> FP8 per-channel conversion: bit-exact
against the oracle on adversarial and random rows, and at the full size of the
skewed workload (384 x (2*2048 + 7168) expert rows) exact on sampled rows plus
the lossless round trip checked on every row with plain torch ops."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import convert as C

from gpu_util import ensure_built, torch_cuda

pytestmark = pytest.mark.gpu


def _run(torch, codes, scales):
    R, K = codes.shape[0], codes.shape[1] * 2
    c = torch.from_numpy(codes).cuda()
    s = torch.from_numpy(scales).cuda()
    out = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    rs = torch.empty(R, dtype=torch.float32, device="cuda")
    st = torch.empty(R, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    fm.mxfp4_to_fp8_rowscale(c.data_ptr(), s.data_ptr(), R, K, out.data_ptr(), rs.data_ptr(), st.data_ptr(),
                             ws.data_ptr(), 256)
    code, count = fm.get_status(ws.data_ptr())
    return out.cpu().numpy(), rs.cpu().numpy(), st.cpu().numpy(), code, count


def _rows_with_span(rng, n, K, span):
    codes = rng.integers(0, 256, (n, K // 2), dtype=np.uint8)
    lo = rng.integers(1, 254 - span, n)
    sc = lo[:, None] + rng.integers(0, span + 1, (n, K // 32))
    return codes, sc.astype(np.uint8)


def test_adversarial_rows():
    torch = torch_cuda()
    ensure_built()
    codes, scales, names = synth.adversarial_conversion_rows(256)
    out, rs, st, code, count = _run(torch, codes, scales)
    ro, rrs, rst = C.mxfp4_to_fp8_rowscale(codes, scales)
    assert np.array_equal(out, ro)
    assert np.array_equal(rs.view(np.uint32), rrs.view(np.uint32))  # NaN rows compare by bits
    assert np.array_equal(st, rst)
    assert count == int((rst != 0).sum()) and code in (6, 7)


@pytest.mark.parametrize("span", [0, 3, 9, 10, 14, 30])
def test_random_rows(span):
    torch = torch_cuda()
    ensure_built()
    rng = np.random.default_rng(100 + span)
    codes, scales = _rows_with_span(rng, 513, 7168 if span < 10 else 2048, span)
    out, rs, st, code, count = _run(torch, codes, scales)
    ro, rrs, rst = C.mxfp4_to_fp8_rowscale(codes, scales)
    assert np.array_equal(st, rst)
    assert np.array_equal(rs.view(np.uint32), rrs.view(np.uint32))
    assert np.array_equal(out, ro)
    if span <= 9:
        assert np.all(st == 0) and count == 0


@pytest.mark.parametrize("K,n", [(32, 37), (96, 300), (480, 1001), (8192, 150), (8224, 90), (16384, 70)])
def test_row_lengths(K, n):
    """Row lengths from one block (odd scale-row widths, rows not a multiple
    of the warps per CTA) to past the 8192 codes a warp stages in shared
    memory, where the kernel switches to two passes over global memory."""
    torch = torch_cuda()
    ensure_built()
    rng = np.random.default_rng(K + n)
    codes, scales = _rows_with_span(rng, n, K, 12)
    out, rs, st, code, count = _run(torch, codes, scales)
    ro, rrs, rst = C.mxfp4_to_fp8_rowscale(codes, scales)
    assert np.array_equal(st, rst)
    assert np.array_equal(rs.view(np.uint32), rrs.view(np.uint32))
    assert np.array_equal(out, ro)
    assert count == int((rst != 0).sum())


def test_full_size_skewed_workload():
    """All routed expert rows of the skewed workload: 384 experts x (4096 gate/up
    rows of K=7168 + 7168 down rows of K=2048) = 4,325,376 rows."""
    torch = torch_cuda()
    ensure_built()
    cfg = synth.configs()["skewed_shared"]
    lut = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], dtype=torch.float32,
                       device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(7)
    for which, (sc, ss) in (("w13", (synth.S_W13, synth.S_W13S)), ("w2", (synth.S_W2, synth.S_W2S))):
        rows, K = synth.weight_shape(cfg, which)
        R = cfg.E * rows
        codes = torch.empty((R, K // 2), dtype=torch.uint8, device="cuda")
        synth.dev_uniform_bytes(cfg.seed, sc, 0, codes)
        scales = torch.empty((R, K // 32), dtype=torch.uint8, device="cuda")
        synth.dev_e8m0_scales(cfg.seed, ss, 0, R, K // 32, scales)
        out = torch.empty((R, K), dtype=torch.uint8, device="cuda")
        rs = torch.empty(R, dtype=torch.float32, device="cuda")
        st = torch.empty(R, dtype=torch.uint8, device="cuda")
        fm.mxfp4_to_fp8_rowscale(codes.data_ptr(), scales.data_ptr(), R, K, out.data_ptr(), rs.data_ptr(),
                                 st.data_ptr(), ws.data_ptr(), 256)
        torch.cuda.synchronize()
        assert int(st.max().item()) == 0
        # round trip on every row, in chunks: fp8 * 2^k == E2M1 * 2^(s - 127)
        for r0 in range(0, R, 1 << 16):
            r1 = min(R, r0 + (1 << 16))
            c = codes[r0:r1]
            v = torch.stack([lut[(c & 15).long()], lut[(c >> 4).long()]], dim=-1).reshape(r1 - r0, K)
            sc_f = torch.exp2(scales[r0:r1].float() - 127).repeat_interleave(32, dim=1)
            ref = v.double() * sc_f.double()
            got = out[r0:r1].view(torch.float8_e4m3fn).double() * rs[r0:r1].double()[:, None]
            assert torch.equal(got, ref)
            vals = out[r0:r1].view(torch.float8_e4m3fn).float().abs()
            assert float(vals.max()) <= 192.0
        # sampled rows, byte for byte against the oracle
        for r in rng.integers(0, R, 16):
            e, rr = divmod(int(r), rows)
            hc, hs = synth.gen_mx_weight(cfg, which, e)
            ro, rrs, rst = C.mxfp4_to_fp8_rowscale(hc[rr:rr + 1], hs[rr:rr + 1])
            assert np.array_equal(out[r].cpu().numpy(), ro[0])
            assert rs[r].item() == rrs[0]
        del codes, scales, out, rs, st
    code, count = fm.get_status(ws.data_ptr())
    assert count == 0
