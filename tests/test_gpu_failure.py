"""Failure paths on the GPU, in forms that fault and hang nothing.

* A device wait that runs out: the test knob of fp4moe_debug makes CTA 0 of
  the gate/up GEMM withhold its first pipeline stage, with a 1 ms limit on
  the pipeline waits.  The MMA issuer's wait for that stage runs out; the
  call must record FP4MOE_ERR_TIMEOUT, drain what it issued and return (the
  stream stays usable), and the next normal call on the same stream and
  workspace must be correct.  Both gate/up instances are covered: the
  few-token one (front end, token rows) and a many-token one.
* NaN block scales (E8M0 byte 255) in the expert weights: fp4moe_check_scales
  counts them into the status word, and the layer refuses such weights."""
from dataclasses import replace

import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth
from oracle import inputs as OI
from oracle import moe as M

from gpu_util import ensure_built, torch_cuda
from test_gpu_forward import SMALL

pytestmark = pytest.mark.gpu


def _check_against_oracle(cfg, out_bits):
    x, wr, b = OI.layer_inputs(cfg)
    orc = M.layer_forward(cfg, x, wr, b, OI.oracle_weights(cfg))
    got = synth.bf16_bits_to_f64(out_bits)
    ratio = np.abs(got - orc["ref"]) / M.tolerance(orc["ref"], orc["S"], orc["A"])
    return float(np.max(ratio))


@pytest.mark.parametrize("name", ["tiny", "wide_padK"])
def test_withheld_stage_times_out_and_recovers(name):
    torch = torch_cuda()
    ensure_built()
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfg = SMALL[name]
    layer = MoELayer.synthetic(cfg)
    x = layer.synthetic_x()
    dbg = fm.Debug()
    dbg.wait_limit_ns = 1_000_000
    dbg.withhold_first_stage = 1
    out = layer.forward(x, debug=dbg)
    torch.cuda.synchronize()  # the call returned and the stream drained: no fault, no hang
    st, n = fm.get_status(layer.ws.data_ptr())
    assert st == fm.STATUS_CODE["FP4MOE_ERR_TIMEOUT"] and n >= 1, (st, n)
    # the same stream and workspace, a normal call: clean status, correct output
    out = layer.forward(x)
    torch.cuda.synchronize()
    assert fm.get_status(layer.ws.data_ptr()) == (0, 0)
    worst = _check_against_oracle(cfg, out.view(torch.int16).cpu().numpy().view(np.uint16))
    assert worst <= 1.0, worst
    print(name, "timeouts recorded:", n, "worst |err|/tol after recovery:", worst)


def test_nan_scale_bytes_are_reported_and_refused():
    torch = torch_cuda()
    ensure_built()
    from block_scaled_fp4_sigmoid_gb300.layer import MoELayer
    cfg = SMALL["tiny"]
    layer = MoELayer.synthetic(cfg)  # clean weights pass the check
    raw = layer.raw["w2_scale"]
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    fm.check_scales(raw.data_ptr(), raw.numel(), fm.MXFP4, ws.data_ptr(), 256)
    assert fm.get_status(ws.data_ptr()) == (0, 0)
    bad = raw.clone()
    flat = bad.view(-1)
    planted = [0, 17, flat.numel() - 1]  # first, an inner and the last byte (past the 16-byte vector body)
    flat[planted] = 255
    fm.check_scales(bad.data_ptr(), bad.numel(), fm.MXFP4, ws.data_ptr(), 256)
    st, n = fm.get_status(ws.data_ptr())
    assert st == fm.STATUS_CODE["FP4MOE_ERR_NAN_SCALE"] and n == len(planted), (st, n)
    # NVFP4 scales: E4M3 NaN is 0x7F / 0xFF; 0x7E (448) is not
    nvs = torch.full((1000,), 0x7E, dtype=torch.uint8, device="cuda")
    nvs[[3, 999]] = torch.tensor([0x7F, 0xFF], dtype=torch.uint8, device="cuda")
    fm.clear_status(ws.data_ptr())
    fm.check_scales(nvs.data_ptr(), nvs.numel(), fm.NVFP4, ws.data_ptr(), 256)
    assert fm.get_status(ws.data_ptr()) == (fm.STATUS_CODE["FP4MOE_ERR_NAN_SCALE"], 2)
    with pytest.raises(ValueError):
        MoELayer(layer.dims, layer.w13, layer.raw["w13_scale"], layer.w2, bad, layer.w_router, layer.bias)
