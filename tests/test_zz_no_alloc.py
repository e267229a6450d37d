"""fp4moe_route_noalloc against fp4moe_route.

The no-allocation router is for callers that cannot allocate device memory
(memory-planned engines, or code that must not call cudaMalloc because it can
synchronise the device).  It must give the same routing as the workspace
version.  Two calls in a row check that the shared scratch array is reset
correctly between calls; the array's status word must read clean after them.
Near the array's limit (the Kimi prefill router, 4096 tokens x 384 experts,
which fits only with fewer K splits than fp4moe_route takes) the routing must
agree wherever the logits' summation order cannot decide it; just past the
limit the call is refused.  This file is collected last on purpose."""
from dataclasses import replace

import numpy as np
import pytest

import block_scaled_fp4_sigmoid_gb300 as fm
import synth

from gpu_util import dims_of, ensure_built, torch_cuda

pytestmark = pytest.mark.gpu

LOGIT_GAMMA = 2.0 ** -16  # |logit_gpu - logit| <= LOGIT_GAMMA * sum |x * Wr| (either router)

CASES = {"kimi_decode": {}, "deepseek_nvfp4_T64": {"T": 64}}  # few-token GEMV and tensor-core router paths


def _inputs(cfg):
    torch = torch_cuda()
    x = torch.from_numpy(synth.gen_x_bf16(cfg).view(np.int16)).cuda()
    wr = torch.from_numpy(synth.gen_router_bf16(cfg).view(np.int16)).cuda()
    b = torch.from_numpy(synth.gen_bias_f32(cfg)).cuda()
    return x, wr, b


def _route_both(cfg, calls=2):
    """fp4moe_route once, then fp4moe_route_noalloc `calls` times; yields
    (ref idx, w, logits) and each no-allocation result in turn."""
    torch = torch_cuda()
    ensure_built()
    d = dims_of(cfg)
    x, wr, b = _inputs(cfg)
    n = fm.workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
    ref_l = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    fm.route(d, x.data_ptr(), wr.data_ptr(), b.data_ptr(), ref_idx.data_ptr(), ref_w.data_ptr(), ref_l.data_ptr(),
             ws.data_ptr(), n)
    out = []
    for _ in range(calls):
        idx = torch.full((cfg.T, cfg.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((cfg.T, cfg.top_k), dtype=torch.float32, device="cuda")
        l = torch.zeros((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        fm.route_noalloc(d, x.data_ptr(), wr.data_ptr(), b.data_ptr(), idx.data_ptr(), w.data_ptr(), l.data_ptr())
        torch.cuda.synchronize()
        assert fm.route_noalloc_status() == (0, 0)
        out.append((idx, w, l))
    return (ref_idx, ref_w, ref_l), out


@pytest.mark.parametrize("name", list(CASES))
def test_route_noalloc_matches_route(name):
    torch = torch_cuda()
    cfg = replace(synth.configs()[name.replace("_T64", "")], **CASES[name])
    (ref_idx, ref_w, ref_l), runs = _route_both(cfg)
    for idx, w, l in runs:
        assert torch.equal(idx, ref_idx)
        torch.testing.assert_close(w, ref_w, rtol=2e-5, atol=1e-7)
        torch.testing.assert_close(l, ref_l, rtol=0, atol=2.0 ** -16 * float(ref_l.abs().max()) + 1e-6)


def test_route_noalloc_near_its_limit():
    """4096 x 384 logits: accepted with fewer splits than fp4moe_route's.
    Both routers' logits lie within the error bound of the exact ones;
    tokens whose decision margin clears twice that bound route identically
    in both, with weights equal within what those logit errors allow."""
    from oracle.router import decision_margins
    torch = torch_cuda()
    ensure_built()
    cfg = synth.configs()["kimi_prefill"]
    d = dims_of(cfg)
    assert 0 < fm.route_noalloc_scratch_bytes(d) <= 8 << 20
    (ref_idx, ref_w, ref_l), runs = _route_both(cfg)
    xf = synth.bf16_bits_to_f64(synth.gen_x_bf16(cfg))
    wrf = synth.bf16_bits_to_f64(synth.gen_router_bf16(cfg))
    exact, lsum = xf @ wrf.T, np.abs(xf) @ np.abs(wrf).T
    bias = synth.gen_bias_f32(cfg)
    bound = LOGIT_GAMMA * lsum
    assert np.all(np.abs(ref_l.cpu().numpy() - exact) <= bound)
    ri, rw = ref_idx.cpu().numpy(), ref_w.cpu().numpy()
    for idx, w, l in runs:
        assert np.all(np.abs(l.cpu().numpy() - exact) <= bound)
        gi, gw = idx.cpu().numpy(), w.cpu().numpy()
        skipped = 0
        for t in range(cfg.T):
            em, gm = decision_margins(exact[t], bias, cfg.top_k, cfg.n_group, cfg.topk_group)
            d_c = 0.25 * 2 * np.max(bound[t]) + 2.0 ** -22  # sigmoid slope <= 1/4, two routers' errors
            if em <= 2 * d_c or gm <= 4 * d_c:
                skipped += 1
                continue
            assert set(gi[t]) == set(ri[t]), t
            # weights: each score moves by at most the two routers' logit
            # errors (relative, since d sigma / sigma <= d l), and the sum
            # that normalises them by as much again
            rtol = 2 * 2 * np.max(bound[t]) + 2.0 ** -20
            np.testing.assert_allclose(gw[t][np.argsort(gi[t])], rw[t][np.argsort(ri[t])], rtol=rtol)
        assert skipped < cfg.T // 4, skipped
        print("near-limit tokens skipped as order-dependent:", skipped)


def test_route_noalloc_rejects_oversized():
    """Dims whose scratch does not fit even with one split are refused
    before any device work (the pointers here are never used)."""
    torch_cuda()
    ensure_built()
    for cfg in (synth.configs()["skewed_shared"], replace(synth.configs()["kimi_prefill"], T=4096, E=512)):
        d = dims_of(cfg)
        assert fm.route_noalloc_scratch_bytes(d) == 0
        with pytest.raises(fm.Fp4MoeError) as ei:
            fm.route_noalloc(d, 16, 16, 16, 16, 16, None)
        assert ei.value.code == 3
