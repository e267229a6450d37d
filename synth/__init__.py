"""Seeded synthetic inputs for the routed block-scaled FP4 MoE layer.

This module draws random numbers only: it holds none of the layer's arithmetic
(no quantisation, routing, GEMM or conversion).  Both the FP64 oracle and the
CUDA path take their inputs from here, so the two see the same bytes.

Every value is a pure function of (seed, stream, flat index), built on the
SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  The device generator in ``synth_gen.cu``
implements the same definition, so a 9 GB weight set can be drawn on the GPU
while the oracle regenerates any single expert on the host.

Recipes (one per tensor kind):

* ``uniform_bytes``  - byte i is byte (i % 8) (little endian) of word i // 8.
* ``e8m0_scales``    - per row a base exponent uniform on {lo..hi}; per block an
  offset of 0 / -1 / -2 with probability 0.70 / 0.25 / 0.05; the stored byte is
  127 + base + offset.
* ``normal``         - Irwin-Hall sum of the four 16-bit lanes of a word,
  centred and scaled to the requested standard deviation in float64.  This is
  integer arithmetic followed by one correctly rounded float64 product, so the
  host and the device produce identical values.
* ``to_bf16_bits``   - float64 -> float32 (RNE) -> bfloat16 (RNE) bit pattern.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
STREAM_MUL = 0xD1B54A32D192ED03
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

# Offsets of the per-block E8M0 exponent: 0 / -1 / -2 with p = .70 / .25 / .05,
# decided on the top 32 bits of a word against these integer thresholds.
OFF_T0 = 3006477107  # floor(0.70 * 2**32)
OFF_T1 = 4080218931  # floor(0.95 * 2**32)

# Standard deviation of the Irwin-Hall sum of four uniform 16-bit integers.
IH4_SIGMA = math.sqrt((65536.0 * 65536.0 - 1.0) / 3.0)
IH4_MEAN = 131070


def _mix_scalar(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of one (seed, stream) pair."""
    return _mix_scalar(_mix_scalar(seed) ^ ((stream * STREAM_MUL) & M64))


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, in place."""
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(MIX1)
        z ^= z >> np.uint64(27)
        z *= np.uint64(MIX2)
        z ^= z >> np.uint64(31)
    return z


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of one stream, as uint64."""
    key = np.uint64(stream_key(seed, stream))
    with np.errstate(over="ignore"):
        z = np.arange(start, start + count, dtype=np.uint64)
        z *= np.uint64(GOLDEN)
        z += key
    return _mix(z)


def uniform_bytes(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Bytes ``start .. start+count-1`` of a uniform byte stream (uint8)."""
    w0 = start // 8
    w1 = (start + count + 7) // 8
    b = words(seed, stream, w0, w1 - w0).astype("<u8").view(np.uint8)
    off = start - 8 * w0
    return b[off:off + count].copy()


def e8m0_scales(seed: int, stream: int, row0: int, rows: int, nblk: int,
                lo: int = -10, hi: int = -6) -> np.ndarray:
    """E8M0 scale bytes for ``rows`` rows (starting at global row ``row0``) of
    ``nblk`` blocks each.  Row bases come from stream ``stream + 1``."""
    span = hi - lo + 1
    with np.errstate(over="ignore"):
        base = (words(seed, stream + 1, row0, rows) >> np.uint64(32)) % np.uint64(span)
        base = base.astype(np.int64) + lo
        top = words(seed, stream, row0 * nblk, rows * nblk) >> np.uint64(32)
    off = np.where(top < OFF_T0, 0, np.where(top < OFF_T1, -1, -2)).astype(np.int64)
    b = 127 + base[:, None] + off.reshape(rows, nblk)
    return b.astype(np.uint8)


def normal(seed: int, stream: int, start: int, count: int, std: float) -> np.ndarray:
    """Approximately normal float64 values with the given standard deviation."""
    w = words(seed, stream, start, count)
    s = w & np.uint64(0xFFFF)
    for lane in range(1, 4):
        w >>= np.uint64(16)
        s += w & np.uint64(0xFFFF)
    out = s.view(np.int64).astype(np.float64)
    out -= IH4_MEAN
    out *= float(std) / IH4_SIGMA
    return out


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE); returns uint16 bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).copy()
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        u += np.uint32(0x7FFF)
        u += lsb
    u >>= np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns, as float64."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Stream ids: one per tensor kind.  Weight tensors use one flat counter over
# [E, rows, ...], so expert e's slice is a contiguous counter range.
S_X = 1
S_WR = 2
S_BIAS = 3
S_W13 = 10       # codes; scales use 11 (+12 for row bases)
S_W13S = 11
S_W2 = 20
S_W2S = 21
S_SH13 = 30
S_SH13S = 31
S_SH2 = 40
S_SH2S = 41
S_W13_BF16 = 50  # NVFP4 configuration: bf16 weights before quantisation
S_W2_BF16 = 51
S_SH13_BF16 = 52
S_SH2_BF16 = 53
S_ZIPF_RANK = 60


@dataclass(frozen=True)
class LayerConfig:
    """Shape and routing parameters of one synthetic MoE layer."""
    name: str
    T: int
    H: int
    I: int
    E: int
    top_k: int
    n_group: int = 1
    topk_group: int = 1
    n_shared: int = 0
    routed_scaling: float = 1.0
    renormalize: int = 1
    fmt: str = "mxfp4"          # "mxfp4" or "nvfp4"
    seed: int = 0
    bias_std: float = 0.1
    zipf_s: float = 0.0         # >0: Zipf-shaped correction bias
    zipf_beta: float = 0.0
    x_std: float = 1.0
    wr_std: float = 0.02
    w_std: float = 0.02         # NVFP4: std of the bf16 weights before quantisation
    extra: dict = field(default_factory=dict, compare=False)


def configs() -> dict:
    """The five workloads: tiny, Kimi decode, Kimi prefill, DeepSeek NVFP4,
    skewed routing with a shared expert."""
    from pathlib import Path
    import json
    beta_file = Path(__file__).resolve().parent / "zipf_bias_beta.json"  # written by tests/golden/make_zipf_beta.py
    beta = json.loads(beta_file.read_text())["beta"] if beta_file.exists() else 0.0
    return {
        "tiny": LayerConfig("tiny", T=4, H=256, I=128, E=8, top_k=2),
        "kimi_decode": LayerConfig("kimi_decode", T=8, H=7168, I=2048, E=384, top_k=8,
                                   routed_scaling=2.827),
        "kimi_prefill": LayerConfig("kimi_prefill", T=4096, H=7168, I=2048, E=384, top_k=8,
                                    routed_scaling=2.827),
        "deepseek_nvfp4": LayerConfig("deepseek_nvfp4", T=512, H=7168, I=2048, E=256, top_k=8,
                                      n_group=8, topk_group=4, routed_scaling=2.5, fmt="nvfp4"),
        "skewed_shared": LayerConfig("skewed_shared", T=16384, H=7168, I=2048, E=384, top_k=8,
                                     n_shared=1, routed_scaling=2.827, zipf_s=1.1, zipf_beta=beta),
    }


# --------------------------------------------------------------------------
# Host-side draws of each input tensor.

def gen_x_bf16(cfg: LayerConfig, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Activations x[t0:t1, :] as bf16 bits [rows, H]."""
    t1 = cfg.T if t1 is None else t1
    v = normal(cfg.seed, S_X, t0 * cfg.H, (t1 - t0) * cfg.H, cfg.x_std)
    return to_bf16_bits(v).reshape(t1 - t0, cfg.H)


def gen_router_bf16(cfg: LayerConfig) -> np.ndarray:
    v = normal(cfg.seed, S_WR, 0, cfg.E * cfg.H, cfg.wr_std)
    return to_bf16_bits(v).reshape(cfg.E, cfg.H)


def zipf_ranks(cfg: LayerConfig) -> np.ndarray:
    """A seeded permutation of expert ids: rank[e] in 1..E."""
    keys = words(cfg.seed, S_ZIPF_RANK, 0, cfg.E)
    order = np.argsort(keys, kind="stable")
    rank = np.empty(cfg.E, dtype=np.int64)
    rank[order] = np.arange(1, cfg.E + 1)
    return rank


def gen_bias_f32(cfg: LayerConfig, beta: float | None = None) -> np.ndarray:
    """Correction bias [E] as float32.  Zipf configs: beta * (-s * ln rank)."""
    if cfg.zipf_s > 0:
        b = cfg.zipf_beta if beta is None else beta
        return (b * (-cfg.zipf_s * np.log(zipf_ranks(cfg).astype(np.float64)))).astype(np.float32)
    return normal(cfg.seed, S_BIAS, 0, cfg.E, cfg.bias_std).astype(np.float32)


def _mx_streams(which: str):
    return {"w13": (S_W13, S_W13S), "w2": (S_W2, S_W2S),
            "sh13": (S_SH13, S_SH13S), "sh2": (S_SH2, S_SH2S)}[which]


def weight_shape(cfg: LayerConfig, which: str):
    """(rows per expert, K) of one weight tensor."""
    if which in ("w13", "sh13"):
        return 2 * cfg.I, cfg.H
    return cfg.H, cfg.I


def gen_mx_weight(cfg: LayerConfig, which: str, e: int):
    """MXFP4 weight of expert e: (codes uint8 [rows, K/2], scales uint8 [rows, K/32])."""
    rows, K = weight_shape(cfg, which)
    sc, ss = _mx_streams(which)
    codes = uniform_bytes(cfg.seed, sc, e * rows * (K // 2), rows * (K // 2)).reshape(rows, K // 2)
    scales = e8m0_scales(cfg.seed, ss, e * rows, rows, K // 32)
    return codes, scales


def gen_bf16_weight(cfg: LayerConfig, which: str, e: int) -> np.ndarray:
    """bf16 weight of expert e (NVFP4 configuration) as bits [rows, K]."""
    rows, K = weight_shape(cfg, which)
    st = {"w13": S_W13_BF16, "w2": S_W2_BF16, "sh13": S_SH13_BF16, "sh2": S_SH2_BF16}[which]
    v = normal(cfg.seed, st, e * rows * K, rows * K, cfg.w_std)
    return to_bf16_bits(v).reshape(rows, K)


def adversarial_conversion_rows(K: int = 256) -> tuple[np.ndarray, np.ndarray, list[str]]:
    """Hand-built MXFP4 rows for the FP8 conversion: scale spans of exactly 9
    and 10 binades, E8M0 bytes 0 / 254 / 255, an all-zero row, negative zeros.
    Returns (codes [n, K/2], scales [n, K/32], names)."""
    nb = K // 32
    rows_c, rows_s, names = [], [], []

    def add(name, code_bytes, scales):
        cb = np.asarray(code_bytes, dtype=np.uint8)
        rows_c.append(np.broadcast_to(cb, (K // 2,)).copy() if cb.ndim == 0 else cb)
        rows_s.append(np.asarray(scales, dtype=np.uint8))
        names.append(name)

    # Byte 0x77 holds two 6.0 codes (largest exponent of a block), 0x11 two
    # 0.5 codes (smallest).  Block 0 carries the largest scale.
    edge = np.full(K // 2, 0x11, dtype=np.uint8)
    edge[:16] = 0x77
    add("span9", edge, [127 + 9] + [127] * (nb - 1))
    add("span10", edge, [127 + 10] + [127] * (nb - 1))
    add("span9_low", edge, [0 + 9] + [0] * (nb - 1))
    add("span12_mild", 0x11, [127 + 12] + [127] * (nb - 1))
    add("e8m0_0", 0x77, [0] * nb)
    add("e8m0_254", 0x77, [254] * nb)
    add("e8m0_255", 0x77, [127] * (nb - 1) + [255])
    add("all_zero", 0x00, [127] * nb)
    add("neg_zero", 0x88, [127] * nb)
    add("neg_half", 0x99, [120 + (b % 3) for b in range(nb)])
    mixed = (np.arange(K // 2, dtype=np.int64) * 37) % 256
    rows_c.append(mixed.astype(np.uint8))
    rows_s.append(np.asarray([127 - (b % 4) for b in range(nb)], dtype=np.uint8))
    names.append("mixed_codes")
    return np.stack(rows_c), np.stack(rows_s), names


# --------------------------------------------------------------------------
# Device-side draws (same definitions), through synth/libfp4moe_synth.so.

_DEV = None


def _device_lib():
    global _DEV
    if _DEV is None:
        import ctypes
        from pathlib import Path
        so = Path(__file__).resolve().parent / "libfp4moe_synth.so"
        if not so.exists():
            build_device_lib()
        lib = ctypes.CDLL(str(so))
        u64, vp, i32, f64 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.synth_words.argtypes = [u64, u64, u64, vp, vp]
        lib.synth_e8m0.argtypes = [u64, u64, u64, u64, i32, i32, i32, vp, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, f64, vp, vp]
        for f in (lib.synth_words, lib.synth_e8m0, lib.synth_normal_bf16):
            f.restype = i32
        _DEV = lib
    return _DEV


def build_device_lib(force: bool = False):
    """Compiles synth_gen.cu into synth/libfp4moe_synth.so (sm_103a)."""
    import subprocess
    from pathlib import Path
    here = Path(__file__).resolve().parent
    src, out = here / "synth_gen.cu", here / "libfp4moe_synth.so"
    if out.exists() and not force and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-Xcompiler", "-fPIC", "-shared",
           str(src), "-o", str(out)]
    subprocess.run(cmd, check=True)
    return out


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"synth device kernel failed: cuda error {rc}")


def dev_uniform_bytes(seed, stream, start_byte, out_tensor, cuda_stream=0):
    """Fills a uint8 CUDA tensor (size multiple of 8, start_byte % 8 == 0) with
    bytes start_byte.. of the stream."""
    n = out_tensor.numel()
    assert n % 8 == 0 and start_byte % 8 == 0
    _check(_device_lib().synth_words(stream_key(seed, stream), start_byte // 8, n // 8,
                                     out_tensor.data_ptr(), cuda_stream))


def dev_e8m0_scales(seed, stream, row0, rows, nblk, out_tensor, lo=-10, hi=-6, cuda_stream=0):
    _check(_device_lib().synth_e8m0(stream_key(seed, stream), stream_key(seed, stream + 1), row0, rows, nblk,
                                    lo, hi, out_tensor.data_ptr(), cuda_stream))


def dev_normal_bf16(seed, stream, start, out_tensor, std, cuda_stream=0):
    _check(_device_lib().synth_normal_bf16(stream_key(seed, stream), start, out_tensor.numel(),
                                           float(std) / IH4_SIGMA, out_tensor.data_ptr(), cuda_stream))
