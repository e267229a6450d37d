"""Python binding of libfp4moe (include/fp4moe.h): argument marshalling only.

Every computation runs in the CUDA library; this module loads it with ctypes,
mirrors its C structs and turns non-zero status codes into exceptions.  There
is no fallback: if the library is missing or was not built, importing the
entry points raises.

Pointers are passed as integers (``tensor.data_ptr()``); streams as the raw
``cudaStream_t`` value (``torch.cuda.current_stream().cuda_stream``).
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libfp4moe.so"
HEADER = _PKG.parent / "include" / "fp4moe.h"

MXFP4 = 0
NVFP4 = 1
FP8 = 2  # W8A8 layer (fp4moe_forward_w8a8)

STATUS = {0: "FP4MOE_OK", 1: "FP4MOE_ERR_INVALID_ARG", 2: "FP4MOE_ERR_UNSUPPORTED_SHAPE",
          3: "FP4MOE_ERR_WORKSPACE", 4: "FP4MOE_ERR_CUDA", 5: "FP4MOE_ERR_TIMEOUT",
          6: "FP4MOE_ERR_NAN_SCALE", 7: "FP4MOE_ERR_INEXACT", 8: "FP4MOE_ERR_DEVICE"}
STATUS_CODE = {v: k for k, v in STATUS.items()}
STAGES = ("router", "topk", "permute", "quant", "gateup", "down", "finalize", "end")


class Fp4MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("routed_scaling", ctypes.c_float),
                ("renormalize", ctypes.c_int32), ("fmt", ctypes.c_int32)]


class Weights(ctypes.Structure):
    """fp4moe_weights; packed = 1: payloads in the tiled layout of pack_weights;
    2: as 1 with w13 / sh13 and their scales in the gate/up-paired layouts;
    3: as 2 with w2 / sh2 and their scales in the row-tile-paired layouts."""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w13", "w13_scale", "w2", "w2_scale", "g13", "g2", "sh13", "sh13_scale", "sh2",
                 "sh2_scale", "w_router", "bias")] + [("packed", ctypes.c_int32)]


class Fp8Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w13", "w13_scale", "w2", "w2_scale", "sh13", "sh13_scale", "sh2", "sh2_scale", "w_router",
                 "bias")]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("status", "logits", "topk_idx", "topk_w", "expert_count", "expert_slot", "route_row",
                 "row_tok", "row_w", "xq", "xsf", "hq", "hsf", "h32", "gscale", "out_acc", "total_bytes")] + \
               [(n, ctypes.c_int32) for n in ("n_splits", "n_tile", "rows_cap", "x_by_token")]


class Debug(ctypes.Structure):
    """fp4moe_debug: stage events, h before quantisation, router logits and
    scores, the pipeline wait limit and the timeout test knob."""
    _fields_ = [("events", ctypes.c_void_p * 8), ("h_pre", ctypes.c_void_p), ("logits", ctypes.c_void_p),
                ("scores", ctypes.c_void_p), ("wait_limit_ns", ctypes.c_int64),
                ("withhold_first_stage", ctypes.c_int32), ("down_cta_pair", ctypes.c_int32)]


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not LIB_PATH.exists():
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m block_scaled_fp4_sigmoid_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(str(LIB_PATH))
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        L.fp4moe_version.restype = i32
        L.fp4moe_status_string.argtypes = [i32]
        L.fp4moe_status_string.restype = ctypes.c_char_p
        L.fp4moe_workspace_size.argtypes = [P(Dims)]
        L.fp4moe_workspace_size.restype = sz
        L.fp4moe_workspace_layout.argtypes = [P(Dims), P(WsLayout)]
        L.fp4moe_packed_scales_bytes.argtypes = [i64, i32, i32, i32]
        L.fp4moe_packed_scales_bytes.restype = sz
        L.fp4moe_pack_scales.argtypes = [vp, vp, i64, i32, i32, i32, vp]
        L.fp4moe_packed_weights_bytes.argtypes = [i64, i32, i32]
        L.fp4moe_packed_weights_bytes.restype = sz
        L.fp4moe_pack_weights.argtypes = [vp, vp, i64, i32, i32, vp]
        L.fp4moe_pack_gateup_weights.argtypes = [vp, vp, i64, i32, i32, vp]
        L.fp4moe_pack_gateup_scales.argtypes = [vp, vp, i64, i32, i32, i32, vp]
        L.fp4moe_route.argtypes = [P(Dims), vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fp4moe_quantize_act.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.fp4moe_forward.argtypes = [P(Dims), P(Weights), vp, vp, P(Debug), vp, sz, vp]
        L.fp4moe_forward_cols.argtypes = [P(Dims), P(Weights), vp, vp, i32, i32, P(Debug), vp, sz, vp]
        L.fp4moe_forward_w8a8.argtypes = [P(Dims), P(Fp8Weights), vp, vp, P(Debug), vp, sz, vp]
        L.fp4moe_emulation_workspace_size.argtypes = [P(Dims)]
        L.fp4moe_emulation_workspace_size.restype = sz
        L.fp4moe_forward_nvfp4_emulated.argtypes = [P(Dims), P(Weights), vp, vp, P(Debug), vp, sz, vp]
        L.fp4moe_linear_workspace_size.argtypes = [i32, i32, i32, i32]
        L.fp4moe_linear_workspace_size.restype = sz
        L.fp4moe_linear.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.fp4moe_mxfp4_to_fp8_rowscale.argtypes = [vp, vp, i64, i32, vp, vp, vp, vp, sz, vp]
        L.fp4moe_clear_status.argtypes = [vp, vp]
        L.fp4moe_get_status.argtypes = [vp, vp, P(i32), P(i64)]
        L.fp4moe_route_noalloc.argtypes = [P(Dims), vp, vp, vp, vp, vp, vp, vp]
        L.fp4moe_check_scales.argtypes = [vp, i64, i32, vp, sz, vp]
        L.fp4moe_route_noalloc_scratch_bytes.argtypes = [P(Dims)]
        L.fp4moe_route_noalloc_scratch_bytes.restype = sz
        L.fp4moe_route_noalloc_status.argtypes = [vp, P(i32), P(i64)]
        for name in ("fp4moe_workspace_layout", "fp4moe_pack_scales", "fp4moe_pack_weights", "fp4moe_pack_gateup_weights",
                     "fp4moe_pack_gateup_scales", "fp4moe_route", "fp4moe_quantize_act",
                     "fp4moe_forward", "fp4moe_forward_cols", "fp4moe_forward_w8a8", "fp4moe_forward_nvfp4_emulated", "fp4moe_linear",
                     "fp4moe_mxfp4_to_fp8_rowscale",
                     "fp4moe_clear_status",
                     "fp4moe_get_status", "fp4moe_route_noalloc", "fp4moe_route_noalloc_status",
                     "fp4moe_check_scales"):
            getattr(L, name).restype = i32
        _LIB = L
    return _LIB


def header_functions() -> list[str]:
    """Names of the functions include/fp4moe.h declares."""
    text = HEADER.read_text()
    return sorted(set(re.findall(r"\b(fp4moe_\w+)\s*\(", text)))


def _ok(code: int, where: str) -> None:
    if code != 0:
        raise Fp4MoeError(code, where)


def make_dims(T, H, I, E, top_k, n_group=1, topk_group=1, n_shared=0, routed_scaling=1.0, renormalize=1,
              fmt=MXFP4) -> Dims:
    return Dims(T, H, I, E, top_k, n_group, topk_group, n_shared, routed_scaling, renormalize, fmt)


def version() -> int:
    return lib().fp4moe_version()


def workspace_size(dims: Dims) -> int:
    n = lib().fp4moe_workspace_size(ctypes.byref(dims))
    if n == 0:
        raise Fp4MoeError(2, "fp4moe_workspace_size")
    return n


def workspace_layout(dims: Dims) -> WsLayout:
    out = WsLayout()
    _ok(lib().fp4moe_workspace_layout(ctypes.byref(dims), ctypes.byref(out)), "fp4moe_workspace_layout")
    return out


def packed_scales_bytes(n_mat: int, rows: int, kblocks: int, fmt: int) -> int:
    return lib().fp4moe_packed_scales_bytes(n_mat, rows, kblocks, fmt)


def pack_scales(src: int, dst: int, n_mat: int, rows: int, kblocks: int, fmt: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_pack_scales(src, dst, n_mat, rows, kblocks, fmt, stream), "fp4moe_pack_scales")


def packed_weights_bytes(n_mat: int, rows: int, kbytes: int) -> int:
    return lib().fp4moe_packed_weights_bytes(n_mat, rows, kbytes)


def pack_weights(src: int, dst: int, n_mat: int, rows: int, kbytes: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_pack_weights(src, dst, n_mat, rows, kbytes, stream), "fp4moe_pack_weights")


def pack_gateup_weights(src: int, dst: int, n_mat: int, I: int, kbytes: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_pack_gateup_weights(src, dst, n_mat, I, kbytes, stream), "fp4moe_pack_gateup_weights")


def pack_gateup_scales(src: int, dst: int, n_mat: int, I: int, kblocks: int, fmt: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_pack_gateup_scales(src, dst, n_mat, I, kblocks, fmt, stream), "fp4moe_pack_gateup_scales")


def route(dims: Dims, x: int, w_router: int, bias: int, topk_idx: int, topk_w: int, logits_out: int | None,
          ws: int, ws_bytes: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_route(ctypes.byref(dims), x, w_router, bias, topk_idx, topk_w, logits_out, ws, ws_bytes,
                           stream), "fp4moe_route")


def quantize_act(x: int, x_is_fp32: bool, rows: int, cols: int, fmt: int, global_in: int | None, codes: int,
                 scales: int, global_out: int | None, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_quantize_act(x, int(x_is_fp32), rows, cols, fmt, global_in, codes, scales, global_out, ws,
                                  ws_bytes, stream), "fp4moe_quantize_act")


def forward(dims: Dims, weights: Weights, x: int, out: int, ws: int, ws_bytes: int, stream: int = 0,
            debug: Debug | None = None) -> None:
    dbg = ctypes.byref(debug) if debug is not None else None
    _ok(lib().fp4moe_forward(ctypes.byref(dims), ctypes.byref(weights), x, out, dbg, ws, ws_bytes, stream),
        "fp4moe_forward")


def forward_cols(dims: Dims, weights: Weights, x: int, out: int, h_begin: int, h_end: int, ws: int, ws_bytes: int,
                 stream: int = 0, debug: Debug | None = None) -> None:
    dbg = ctypes.byref(debug) if debug is not None else None
    _ok(lib().fp4moe_forward_cols(ctypes.byref(dims), ctypes.byref(weights), x, out, h_begin, h_end, dbg, ws,
                                  ws_bytes, stream), "fp4moe_forward_cols")


def forward_w8a8(dims: Dims, weights: Fp8Weights, x: int, out: int, ws: int, ws_bytes: int, stream: int = 0,
                 debug: Debug | None = None) -> None:
    dbg = ctypes.byref(debug) if debug is not None else None
    _ok(lib().fp4moe_forward_w8a8(ctypes.byref(dims), ctypes.byref(weights), x, out, dbg, ws, ws_bytes, stream),
        "fp4moe_forward_w8a8")


def emulation_workspace_size(dims: Dims) -> int:
    n = lib().fp4moe_emulation_workspace_size(ctypes.byref(dims))
    if n == 0:
        raise Fp4MoeError(2, "fp4moe_emulation_workspace_size")
    return n


def forward_nvfp4_emulated(dims: Dims, weights: Weights, x: int, out: int, ws: int, ws_bytes: int, stream: int = 0,
                           debug: Debug | None = None) -> None:
    dbg = ctypes.byref(debug) if debug is not None else None
    _ok(lib().fp4moe_forward_nvfp4_emulated(ctypes.byref(dims), ctypes.byref(weights), x, out, dbg, ws, ws_bytes,
                                            stream), "fp4moe_forward_nvfp4_emulated")


def linear_workspace_size(fmt: int, T: int, K: int, N: int) -> int:
    n = lib().fp4moe_linear_workspace_size(fmt, T, K, N)
    if n == 0:
        raise Fp4MoeError(2, "fp4moe_linear_workspace_size")
    return n


def linear(fmt: int, T: int, K: int, N: int, x: int, w: int, w_scale: int, g_w: int | None, out: int, ws: int,
           ws_bytes: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_linear(fmt, T, K, N, x, w, w_scale, g_w, out, ws, ws_bytes, stream), "fp4moe_linear")


def mxfp4_to_fp8_rowscale(codes: int, scales: int, rows: int, K: int, fp8_out: int, row_scale: int,
                          row_status: int | None, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_mxfp4_to_fp8_rowscale(codes, scales, rows, K, fp8_out, row_scale, row_status, ws, ws_bytes,
                                           stream), "fp4moe_mxfp4_to_fp8_rowscale")


def check_scales(scales: int, n: int, fmt: int, ws: int, ws_bytes: int, stream: int = 0) -> None:
    """Records the NaN scale bytes among n bytes in the status word of ws (fp4moe_check_scales)."""
    _ok(lib().fp4moe_check_scales(scales, n, fmt, ws, ws_bytes, stream), "fp4moe_check_scales")


def clear_status(ws: int, stream: int = 0) -> None:
    _ok(lib().fp4moe_clear_status(ws, stream), "fp4moe_clear_status")


def get_status(ws: int, stream: int = 0) -> tuple[int, int]:
    st, n = ctypes.c_int32(0), ctypes.c_int64(0)
    _ok(lib().fp4moe_get_status(ws, stream, ctypes.byref(st), ctypes.byref(n)), "fp4moe_get_status")
    return st.value, n.value


def route_noalloc(dims: Dims, x: int, w_router: int, bias: int, topk_idx: int, topk_w: int,
                  logits_out: int | None, stream: int = 0) -> None:
    """fp4moe_route without a workspace: the library's fixed scratch array is used."""
    _ok(lib().fp4moe_route_noalloc(ctypes.byref(dims), x, w_router, bias, topk_idx, topk_w, logits_out, stream),
        "fp4moe_route_noalloc")


def route_noalloc_scratch_bytes(dims: Dims) -> int:
    """Bytes of the fixed scratch array a route_noalloc call with these dims uses (0: does not fit)."""
    return lib().fp4moe_route_noalloc_scratch_bytes(ctypes.byref(dims))


def route_noalloc_status(stream: int = 0) -> tuple[int, int]:
    """Status word of the last route_noalloc call on the current device."""
    st, n = ctypes.c_int32(0), ctypes.c_int64(0)
    _ok(lib().fp4moe_route_noalloc_status(stream, ctypes.byref(st), ctypes.byref(n)), "fp4moe_route_noalloc_status")
    return st.value, n.value
