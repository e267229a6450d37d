"""A routed block-scaled FP4 MoE layer held in device memory.

``MoELayer`` owns the expert weights (packed FP4 codes, by default also
repacked into the tiled payload layout the GEMMs stream as whole tiles;
repacked block scales; NVFP4 tensor scales), the router weights and bias,
and a workspace;
``forward`` calls fp4moe_forward.  PyTorch only allocates device memory and
supplies the stream.  ``MoELayer.synthetic`` draws a layer from the seeded
generator in ``synth`` directly on the GPU (weights of the NVFP4
configuration are quantised from bf16 by fp4moe_quantize_act, one tensor scale
per expert and weight tensor).
"""
from __future__ import annotations

import ctypes

import torch

from . import (FP8, MXFP4, NVFP4, Debug, Fp8Weights, Weights, check_scales, emulation_workspace_size, forward,
               forward_cols,
               forward_nvfp4_emulated, forward_w8a8, get_status, make_dims,
               mxfp4_to_fp8_rowscale, pack_gateup_scales, pack_gateup_weights, pack_scales, pack_weights,
               packed_scales_bytes, packed_weights_bytes,
               quantize_act, workspace_layout, workspace_size)


def _ptr(t):
    return t.data_ptr() if t is not None else None


def column_block(H: int, rank: int, world: int, unit: int = 128) -> tuple[int, int]:
    """Output columns [h0, h1) of rank `rank` of `world` in an
    output-partitioned layer: whole tiles of `unit` columns (128, or 256 for
    down weights in the row-tile-paired layout), as even as possible."""
    tiles = H // unit
    if not 0 < world <= tiles or not 0 <= rank < world:
        raise ValueError(f"{world} ranks over {tiles} column tiles of {unit}")
    return unit * (tiles * rank // world), unit * (tiles * (rank + 1) // world)


def tp_forward(layer, x, group=None):
    """Output-partitioned forward over a torch.distributed group: each rank
    computes its block of output columns (zero elsewhere) and one all-reduce
    (sum) assembles the layer output on every rank ("Inside the Kimi K3
    optimization effort", section "MoE: remove duplicate work across GPUs")."""
    import torch.distributed as dist
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    h0, h1 = column_block(layer.dims.H, rank, world, layer.column_unit)
    out = layer.forward_cols(x, h0, h1)
    dist.all_reduce(out, group=group)
    return out


class MoELayer:
    def __init__(self, dims, w13, w13_scale, w2, w2_scale, w_router, bias, g13=None, g2=None,
                 sh13=None, sh13_scale=None, sh2=None, sh2_scale=None, packed: bool | int = True):
        """Tensors on one CUDA device.  Scales are the raw row-major block
        scales ([E, rows, K/32] E8M0 or [E, rows, K/16] E4M3); they are
        repacked here into the layout the GEMMs load.  packed (the
        fp4moe_weights level): 0 / False, the forward reads the row-major
        payloads themselves; 2, the tiled layout of fp4moe_pack_weights, with
        the gate/up matrices and their scales in the gate/up-paired order of
        fp4moe_pack_gateup_weights / _scales; 3, as 2 with the down matrices
        in the row-tile-paired order (each 256-row slab packed as a gate/up
        pair of I = 128; needs H % 256 == 0, and column blocks of whole
        slabs); True, 3 where H allows it, else 2.  The row-major tensors
        are kept either way (the FP8 conversion reads them)."""
        self.dims = dims
        self.fmt = dims.fmt
        self.device = w13.device
        self.raw = dict(w13_scale=w13_scale, w2_scale=w2_scale, sh13_scale=sh13_scale, sh2_scale=sh2_scale)
        blk = 16 if dims.fmt == NVFP4 else 32
        if packed is True:
            packed = 3 if dims.H % 256 == 0 else 2
        packed = int(packed)
        if packed not in (0, 2, 3) or (packed == 3 and dims.H % 256):
            raise ValueError(f"packed level {packed} (0, 2, or 3 with H % 256 == 0)")
        self.w13, self.w2 = w13.contiguous(), w2.contiguous()
        self.w13_scale = self._pack(w13_scale, dims.E, 2 * dims.I, dims.H // blk, gateup=packed >= 2)
        self.w2_scale = self._pack(w2_scale, dims.E, dims.H, dims.I // blk, slabs=packed == 3)
        self.w_router, self.bias = w_router.contiguous(), bias.contiguous()
        self.g13, self.g2 = g13, g2
        self.sh13, self.sh2 = sh13, sh2
        self.sh13_scale = (self._pack(sh13_scale, 1, 2 * dims.I, dims.H // blk, gateup=packed >= 2)
                           if sh13 is not None else None)
        self.sh2_scale = (self._pack(sh2_scale, 1, dims.H, dims.I // blk, slabs=packed == 3) if sh2 is not None
                          else None)
        self.packed = packed
        self.column_unit = 256 if packed == 3 else 128  # granularity of forward_cols' column blocks
        pw = self._pack_w if packed else (lambda t, *_, **__: t)
        self.w13_t = pw(self.w13, dims.E, 2 * dims.I, dims.H // 2, gateup=True)
        self.w2_t = pw(self.w2, dims.E, dims.H, dims.I // 2, slabs=packed == 3)
        self.sh13_t = pw(sh13, 1, 2 * dims.I, dims.H // 2, gateup=True) if sh13 is not None else None
        self.sh2_t = pw(sh2, 1, dims.H, dims.I // 2, slabs=packed == 3) if sh2 is not None else None
        self._check_scales()
        self.ws_bytes = workspace_size(dims)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.layout = workspace_layout(dims)
        self.weights = Weights(_ptr(self.w13_t), _ptr(self.w13_scale), _ptr(self.w2_t), _ptr(self.w2_scale),
                               _ptr(self.g13), _ptr(self.g2), _ptr(self.sh13_t), _ptr(self.sh13_scale),
                               _ptr(self.sh2_t), _ptr(self.sh2_scale), _ptr(self.w_router), _ptr(self.bias),
                               packed)

    def _check_scales(self):
        """Refuses weights with NaN block scales (fp4moe_check_scales): the
        layer does not test its scales on every call."""
        ws = torch.zeros(256, dtype=torch.uint8, device=self.device)
        s = torch.cuda.current_stream(self.device).cuda_stream
        for name, t in self.raw.items():
            if t is not None:
                check_scales(t.data_ptr(), t.numel(), self.fmt, ws.data_ptr(), 256, s)
        st, n = get_status(ws.data_ptr(), s)
        if st != 0:
            raise ValueError(f"{n} NaN block-scale bytes in the expert weights (status {st})")

    def _pack_w(self, codes, n_mat, rows, kbytes, gateup=False, slabs=False):
        dst = torch.empty(packed_weights_bytes(n_mat, rows, kbytes), dtype=torch.uint8, device=codes.device)
        s = torch.cuda.current_stream(codes.device).cuda_stream
        if gateup:  # rows = 2I: gate/up-paired tiles
            pack_gateup_weights(codes.data_ptr(), dst.data_ptr(), n_mat, rows // 2, kbytes, s)
        elif slabs:  # row-tile pairs: each 256-row slab as a gate/up pair of I = 128
            pack_gateup_weights(codes.data_ptr(), dst.data_ptr(), n_mat * rows // 256, 128, kbytes, s)
        else:
            pack_weights(codes.data_ptr(), dst.data_ptr(), n_mat, rows, kbytes, s)
        return dst

    def _pack(self, raw, n_mat, rows, kblocks, gateup=False, slabs=False):
        dst = torch.empty(packed_scales_bytes(n_mat, rows, kblocks, self.fmt), dtype=torch.uint8,
                          device=raw.device)
        s = torch.cuda.current_stream(raw.device).cuda_stream
        if gateup:  # rows = 2I: gate/up-paired scale groups
            pack_gateup_scales(raw.data_ptr(), dst.data_ptr(), n_mat, rows // 2, kblocks, self.fmt, s)
        elif slabs:  # row-tile pairs (see _pack_w)
            pack_gateup_scales(raw.data_ptr(), dst.data_ptr(), n_mat * rows // 256, 128, kblocks, self.fmt, s)
        else:
            pack_scales(raw.data_ptr(), dst.data_ptr(), n_mat, rows, kblocks, self.fmt, s)
        return dst

    def weight_bytes_per_expert(self) -> int:
        """Packed FP4 codes plus scales of one routed expert (w13 and w2)."""
        d = self.dims
        blk = 16 if d.fmt == NVFP4 else 32
        elems = 3 * d.H * d.I
        return elems // 2 + elems // blk

    def forward(self, x, out=None, debug: Debug | None = None, stream=None):
        d = self.dims
        if out is None:
            out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=self.device)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        forward(d, self.weights, x.data_ptr(), out.data_ptr(), self.ws.data_ptr(), self.ws_bytes, s, debug)
        return out

    def forward_cols(self, x, h_begin: int, h_end: int, out=None, debug: Debug | None = None, stream=None):
        """The layer output restricted to columns [h_begin, h_end); the other
        columns of out are zero (fp4moe_forward_cols)."""
        d = self.dims
        if out is None:
            out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=self.device)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        forward_cols(d, self.weights, x.data_ptr(), out.data_ptr(), h_begin, h_end, self.ws.data_ptr(),
                     self.ws_bytes, s, debug)
        return out

    def forward_emulated(self, x, out=None, debug: Debug | None = None, stream=None):
        """NVFP4 layers only: the same layer in emulation mode
        (fp4moe_forward_nvfp4_emulated: BF16 dequantised experts, NVFP4 QDQ
        activations, BF16 GEMMs), with a workspace of its own."""
        d = self.dims
        if d.fmt != NVFP4:
            raise ValueError("emulation mode is for NVFP4 layers")
        if getattr(self, "emu_ws", None) is None:
            self.emu_ws_bytes = emulation_workspace_size(d)
            self.emu_ws = torch.empty(self.emu_ws_bytes, dtype=torch.uint8, device=self.device)
        if out is None:
            out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=self.device)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        forward_nvfp4_emulated(d, self.weights, x.data_ptr(), out.data_ptr(), self.emu_ws.data_ptr(),
                               self.emu_ws_bytes, s, debug)
        return out

    # ------------------------------------------------------------ workspace views
    def ws_view(self, name: str, dtype, count: int):
        off = getattr(self.layout, name)
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype)

    # ------------------------------------------------------------ synthetic layers
    @classmethod
    def synthetic(cls, cfg, device="cuda", packed: bool | int = True):
        import synth
        fmt = NVFP4 if cfg.fmt == "nvfp4" else MXFP4
        dims = make_dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.n_shared,
                         cfg.routed_scaling, cfg.renormalize, fmt)
        dev = torch.device(device)
        wr = torch.from_numpy(synth.gen_router_bf16(cfg).view("int16")).to(dev)
        bias = torch.from_numpy(synth.gen_bias_f32(cfg)).to(dev)
        ws_small = torch.zeros(256, dtype=torch.uint8, device=dev)

        def mx_weight(which, n_exp):
            rows, K = synth.weight_shape(cfg, which)
            codes_s, scale_s = synth._mx_streams(which)
            codes = torch.empty((n_exp, rows, K // 2), dtype=torch.uint8, device=dev)
            synth.dev_uniform_bytes(cfg.seed, codes_s, 0, codes)
            scales = torch.empty((n_exp, rows, K // 32), dtype=torch.uint8, device=dev)
            synth.dev_e8m0_scales(cfg.seed, scale_s, 0, n_exp * rows, K // 32, scales)
            return codes, scales, None

        def nv_weight(which, n_exp):
            rows, K = synth.weight_shape(cfg, which)
            st = {"w13": synth.S_W13_BF16, "w2": synth.S_W2_BF16,
                  "sh13": synth.S_SH13_BF16, "sh2": synth.S_SH2_BF16}[which]
            codes = torch.empty((n_exp, rows, K // 2), dtype=torch.uint8, device=dev)
            scales = torch.empty((n_exp, rows, K // 16), dtype=torch.uint8, device=dev)
            g = torch.empty(n_exp, dtype=torch.float32, device=dev)
            tmp = torch.empty((rows, K), dtype=torch.int16, device=dev)
            s = torch.cuda.current_stream(dev).cuda_stream
            for e in range(n_exp):
                synth.dev_normal_bf16(cfg.seed, st, e * rows * K, tmp, cfg.w_std, s)
                quantize_act(tmp.data_ptr(), False, rows, K, NVFP4, None, codes[e].data_ptr(), scales[e].data_ptr(),
                             g[e:e + 1].data_ptr(), ws_small.data_ptr(), 256, s)
            return codes, scales, g

        make = nv_weight if fmt == NVFP4 else mx_weight
        w13, w13s, g13 = make("w13", cfg.E)
        w2, w2s, g2 = make("w2", cfg.E)
        sh = {}
        if cfg.n_shared:
            s13, s13s, sg13 = make("sh13", 1)
            s2, s2s, sg2 = make("sh2", 1)
            sh = dict(sh13=s13, sh13_scale=s13s, sh2=s2, sh2_scale=s2s)
            if fmt == NVFP4:
                g13 = torch.cat([g13, sg13])
                g2 = torch.cat([g2, sg2])
        layer = cls(dims, w13, w13s, w2, w2s, wr, bias, g13=g13, g2=g2, packed=packed, **sh)
        layer.cfg = cfg
        layer.raw_scales = (w13s, w2s)
        return layer

    def variant(self, cfg):
        """A layer over the same routed experts and router weights for another
        batch size or routing configuration of the same shape (E, H, I,
        format): its own dims, correction bias and workspace, no copy of the
        weights.  The shared expert is kept when cfg has one (this layer must
        hold it then) and dropped otherwise."""
        import copy
        import synth
        d = self.dims
        if (cfg.E, cfg.H, cfg.I) != (d.E, d.H, d.I) or (NVFP4 if cfg.fmt == "nvfp4" else MXFP4) != d.fmt:
            raise ValueError("a variant keeps the experts' shape and format")
        if cfg.n_shared and self.sh13 is None:
            raise ValueError("this layer holds no shared expert")
        v = copy.copy(self)
        v.cfg = cfg
        v.dims = make_dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.n_group, cfg.topk_group, cfg.n_shared,
                           cfg.routed_scaling, cfg.renormalize, d.fmt)
        v.bias = torch.from_numpy(synth.gen_bias_f32(cfg)).to(self.device)
        if not cfg.n_shared:
            v.sh13 = v.sh2 = v.sh13_scale = v.sh2_scale = v.sh13_t = v.sh2_t = None
        v.ws_bytes = workspace_size(v.dims)
        v.ws = torch.empty(v.ws_bytes, dtype=torch.uint8, device=self.device)
        v.layout = workspace_layout(v.dims)
        v.emu_ws = None
        v.weights = Weights(_ptr(v.w13_t), _ptr(v.w13_scale), _ptr(v.w2_t), _ptr(v.w2_scale), _ptr(v.g13),
                            _ptr(v.g2), _ptr(v.sh13_t), _ptr(v.sh13_scale), _ptr(v.sh2_t), _ptr(v.sh2_scale),
                            _ptr(v.w_router), _ptr(v.bias), v.packed)
        return v

    def synthetic_x(self, t0: int = 0, t1: int | None = None):
        """Activations of the synthetic configuration, drawn on the device."""
        import synth
        cfg = self.cfg
        t1 = cfg.T if t1 is None else t1
        x = torch.empty((t1 - t0, cfg.H), dtype=torch.int16, device=self.device)
        synth.dev_normal_bf16(cfg.seed, synth.S_X, t0 * cfg.H, x, cfg.x_std)
        return x.view(torch.bfloat16)


class W8A8Layer:
    """The W8A8 form of an MXFP4 ``MoELayer``: every expert matrix converted
    exactly to E4M3 with one fp32 power-of-two scale per row by
    fp4moe_mxfp4_to_fp8_rowscale, run by fp4moe_forward_w8a8 (per-token
    dynamic E4M3 activations).  Same routing weights, shape and device."""

    def __init__(self, mx: MoELayer):
        d = mx.dims
        if d.fmt != MXFP4:
            raise ValueError("the exact FP8 conversion starts from MXFP4 experts")
        self.mx = mx
        self.device = mx.device
        self.dims = make_dims(d.T, d.H, d.I, d.E, d.top_k, d.n_group, d.topk_group, d.n_shared, d.routed_scaling,
                              d.renormalize, FP8)
        s = torch.cuda.current_stream(self.device).cuda_stream
        ws = torch.zeros(256, dtype=torch.uint8, device=self.device)

        def conv(codes, raw, n_mat, rows, K):
            out = torch.empty((n_mat, rows, K), dtype=torch.uint8, device=self.device)
            rs = torch.empty((n_mat, rows), dtype=torch.float32, device=self.device)
            mxfp4_to_fp8_rowscale(codes.data_ptr(), raw.data_ptr(), n_mat * rows, K, out.data_ptr(), rs.data_ptr(),
                                  None, ws.data_ptr(), 256, s)
            return out, rs

        self.w13, self.w13_scale = conv(mx.w13, mx.raw["w13_scale"], d.E, 2 * d.I, d.H)
        self.w2, self.w2_scale = conv(mx.w2, mx.raw["w2_scale"], d.E, d.H, d.I)
        self.sh13 = self.sh13_scale = self.sh2 = self.sh2_scale = None
        if d.n_shared:
            self.sh13, self.sh13_scale = conv(mx.sh13, mx.raw["sh13_scale"], 1, 2 * d.I, d.H)
            self.sh2, self.sh2_scale = conv(mx.sh2, mx.raw["sh2_scale"], 1, d.H, d.I)
        st, n = get_status(ws.data_ptr(), s)
        if st != 0:
            raise ValueError(f"{n} expert rows are outside the exact conversion's contract (status {st})")
        self.ws_bytes = workspace_size(self.dims)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.layout = workspace_layout(self.dims)
        self.weights = Fp8Weights(_ptr(self.w13), _ptr(self.w13_scale), _ptr(self.w2), _ptr(self.w2_scale),
                                  _ptr(self.sh13), _ptr(self.sh13_scale), _ptr(self.sh2), _ptr(self.sh2_scale),
                                  _ptr(mx.w_router), _ptr(mx.bias))
        self.cfg = getattr(mx, "cfg", None)

    def weight_bytes_per_expert(self) -> int:
        """E4M3 bytes plus fp32 row scales of one routed expert (w13 and w2)."""
        d = self.dims
        return 3 * d.H * d.I + 4 * (2 * d.I + d.H)

    def forward(self, x, out=None, debug: Debug | None = None, stream=None):
        d = self.dims
        if out is None:
            out = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=self.device)
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        forward_w8a8(d, self.weights, x.data_ptr(), out.data_ptr(), self.ws.data_ptr(), self.ws_bytes, s, debug)
        return out

    def ws_view(self, name: str, dtype, count: int):
        off = getattr(self.layout, name)
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype)

    def synthetic_x(self, t0: int = 0, t1: int | None = None):
        return self.mx.synthetic_x(t0, t1)
