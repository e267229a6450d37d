"""fp4moe_route_noalloc against fp4moe_route.

The no-allocation router is for callers that cannot allocate device memory
(memory-planned engines, or code that must not call cudaMalloc because it can
synchronise the device).  It must give the same routing as the workspace
version.  Two calls in a row check that the shared scratch array is reset
correctly between calls.  This file is collected last on purpose."""
import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth

from gpu_util import dims_of, ensure_built, torch_cuda

pytestmark = pytest.mark.gpu


CASES = {"kimi_decode": {}, "deepseek_nvfp4_T64": {"T": 64}}  # few-token GEMV and tensor-core router paths


@pytest.mark.parametrize("name", list(CASES))
def test_route_noalloc_matches_route(name):
    from dataclasses import replace
    torch = torch_cuda()
    ensure_built()
    cfg = replace(synth.configs()[name.replace("_T64", "")], **CASES[name])
    d = dims_of(cfg)
    x = torch.from_numpy(synth.gen_x_bf16(cfg).view(np.int16)).cuda()
    wr = torch.from_numpy(synth.gen_router_bf16(cfg).view(np.int16)).cuda()
    b = torch.from_numpy(synth.gen_bias_f32(cfg)).cuda()
    n = fm.workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    ref_l = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    fm.route(d, x.data_ptr(), wr.data_ptr(), b.data_ptr(), ref_idx.data_ptr(), ref_w.data_ptr(), ref_l.data_ptr(),
             ws.data_ptr(), n)
    for _ in range(2):
        idx = torch.full((cfg.T, cfg.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
        l = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        fm.route_noalloc(d, x.data_ptr(), wr.data_ptr(), b.data_ptr(), idx.data_ptr(), w.data_ptr(), l.data_ptr())
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        torch.testing.assert_close(w, ref_w, rtol=2e-5, atol=1e-7)
        torch.testing.assert_close(l, ref_l, rtol=0, atol=2.0 ** -16 * float(ref_l.abs().max()) + 1e-6)


def test_route_noalloc_rejects_oversized():
    torch_cuda()
    ensure_built()
    cfg = synth.configs()["skewed_shared"]  # 16384 x 384 logits exceed the fixed scratch
    d = dims_of(cfg)
    with pytest.raises(fm.Fp4MoeError) as ei:
        fm.route_noalloc(d, 16, 16, 16, 16, 16, None)
    assert ei.value.code == 3
