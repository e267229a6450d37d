#include <cuda_bf16.h>
// Activation quantisation (MXFP4 / NVFP4), scale repacking, the fused
// gather-and-quantise step of the forward, NVFP4 requantisation of the
// intermediate, the combine finaliser, and the exact MXFP4 -> FP8 conversion.
#include <algorithm>
#include <array>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

namespace {

// Loads 32 consecutive values (bf16 or fp32) starting at element i.
__device__ __forceinline__ void load32(const void* x, int x_is_fp32, int64_t i, float* v) {
  if (x_is_fp32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(x) + i);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4 w = __ldg(p + q);
      v[4 * q + 0] = __uint_as_float(w.x);
      v[4 * q + 1] = __uint_as_float(w.y);
      v[4 * q + 2] = __uint_as_float(w.z);
      v[4 * q + 3] = __uint_as_float(w.w);
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + i);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w = __ldg(p + q);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * q + 2 * j] = __uint_as_float(u[j] << 16);
        v[8 * q + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
      }
    }
  }
}

// ---------------------------------------------------------------- amax
__global__ void amax_kernel(const void* x, int x_is_fp32, int64_t n, uint32_t* amax_bits) {
  float m = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = x_is_fp32 ? static_cast<const float*>(x)[i] : bf16_to_f32(static_cast<const uint16_t*>(x)[i]);
    m = fmaxf(m, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(m));  // non-negative floats order as ints
  }
}

// ---------------------------------------------------------------- row-major quantisation
// One thread per 32 values.  MXFP4: one block; NVFP4: two blocks.
__global__ void quantize_rows_kernel(const void* x, int x_is_fp32, int64_t rows, int cols, int nv,
                                     const float* global_in, const uint32_t* amax_bits, uint8_t* codes,
                                     uint8_t* scales, float* global_out) {
  const int per_row = cols >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= rows * per_row) return;
  const int64_t r = tid / per_row;
  const int b = (int)(tid - r * per_row);
  float v[32];
  load32(x, x_is_fp32, r * cols + 32 * b, v);
  uint32_t p[4];
  uint4* dst = reinterpret_cast<uint4*>(codes + r * (cols >> 1) + 16 * b);
  if (!nv) {
    uint32_t s;
    mx_quant32(v, p, &s);
    *dst = make_uint4(p[0], p[1], p[2], p[3]);
    scales[r * per_row + b] = (uint8_t)s;
  } else {
    const float g = global_in ? *global_in : nv_global(__uint_as_float(*amax_bits));
    if (tid == 0 && global_out) *global_out = g;
    uint32_t s0, s1;
    nv_quant16(v, g, p, &s0);
    nv_quant16(v + 16, g, p + 2, &s1);
    *dst = make_uint4(p[0], p[1], p[2], p[3]);
    scales[r * (cols >> 4) + 2 * b] = (uint8_t)s0;
    scales[r * (cols >> 4) + 2 * b + 1] = (uint8_t)s1;
  }
}

// ---------------------------------------------------------------- forward: gather + quantise x
// One thread per (token, 32 values of H): quantises the block once and
// stores it into the padded row of each of the token's routes, with the
// scales in the tiled layout.
__global__ void gather_quant_kernel(const uint16_t* x, int T, int H, int routes_per_tok,
                                    const int32_t* route_row, uint8_t* xq, uint8_t* xsf, int nv,
                                    const uint32_t* amax_x, float* g_out) {
  pdl_wait();  // route_row (and the NVFP4 amax) come from the previous kernels
  pdl_trigger();
  const int per_row = H >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= (int64_t)T * per_row) return;
  const int64_t t = tid / per_row;
  const int b = (int)(tid - t * per_row);
  float v[32];
  load32(x, 0, t * H + 32 * b, v);
  uint32_t p[4], s0, s1 = 0;
  const int64_t katoms = katoms_padded(H, nv != 0);
  if (!nv) {
    mx_quant32(v, p, &s0);
  } else {
    const float g = nv_global(__uint_as_float(*amax_x));
    if (tid == 0 && g_out) *g_out = g;
    nv_quant16(v, g, p, &s0);
    nv_quant16(v + 16, g, p + 2, &s1);
  }
  const uint4 q = make_uint4(p[0], p[1], p[2], p[3]);
  for (int j = 0; j < routes_per_tok; ++j) {
    const int64_t row = route_row[t * routes_per_tok + j];
    *reinterpret_cast<uint4*>(xq + row * (H >> 1) + 16 * b) = q;
    if (!nv) {
      xsf[sf_tiled_offset(row, b, katoms)] = (uint8_t)s0;
    } else {
      xsf[sf_tiled_offset(row, 2 * b, katoms)] = (uint8_t)s0;
      xsf[sf_tiled_offset(row, 2 * b + 1, katoms)] = (uint8_t)s1;
    }
  }
}

// ---------------------------------------------------------------- forward: NVFP4 requantisation of h
// One thread per (route, 32 values of I).  The tensor scale of h is one per
// expert: g_h[e] = amax_h[e] / 2688.
__global__ void h_quant_nv_kernel(const float* h32, int I, int64_t n_routes, const int32_t* route_row,
                                  const int32_t* row_e, const uint32_t* amax_h, float* gh_out, uint8_t* hq,
                                  uint8_t* hsf, int n_exp) {
  const int per_row = I >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid < n_exp && gh_out) gh_out[tid] = nv_global(__uint_as_float(amax_h[tid]));
  if (tid >= n_routes * per_row) return;
  const int64_t rt = tid / per_row;
  const int b = (int)(tid - rt * per_row);
  const int64_t row = route_row[rt];
  const int e = row_e[row];
  const float g = nv_global(__uint_as_float(amax_h[e]));
  float v[32];
  load32(h32, 1, row * I + 32 * b, v);
  uint32_t p[4], s0, s1;
  nv_quant16(v, g, p, &s0);
  nv_quant16(v + 16, g, p + 2, &s1);
  *reinterpret_cast<uint4*>(hq + row * (I >> 1) + 16 * b) = make_uint4(p[0], p[1], p[2], p[3]);
  const int64_t katoms = katoms_padded(I, true);
  hsf[sf_tiled_offset(row, 2 * b, katoms)] = (uint8_t)s0;
  hsf[sf_tiled_offset(row, 2 * b + 1, katoms)] = (uint8_t)s1;
  // scale groups past I up to the whole K tile hold 1.0 (their codes are zero)
  const int real_blocks = I >> 4, pad_blocks = (int)(katoms * 4) - real_blocks;
  for (int pb = b; pb < pad_blocks; pb += per_row) hsf[sf_tiled_offset(row, real_blocks + pb, katoms)] = 0x38;
}

// ---------------------------------------------------------------- scale repacking
// One thread per 4-byte word of the destination: (matrix, row tile, group, m0, m1).
// ---------------------------------------------------------------- W8A8 activations
// Per-token dynamic E4M3 ("Kimi-K2.7-Code on Gaudi 2", section "Exact MXFP4
// to FP8 per-channel conversion": the converted experts run with per-channel
// weights and dynamic per-token activations).  sigma = amax / 448 and each
// code = RNE_E4M3(v / sigma), saturating, both correctly rounded fp32 steps.
constexpr int kF8Threads = 256;

__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < kF8Threads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

// Four E4M3 codes packed little-endian: value j in byte j.
__device__ __forceinline__ uint32_t fp8_pack4(float a, float b, float c, float d, float sigma) {
  return fp8_code(a, sigma) | fp8_code(b, sigma) << 8 | fp8_code(c, sigma) << 16 | fp8_code(d, sigma) << 24;
}

// One CTA per token: the codes go to every route row of the token, sigma to
// the row-scale array at those rows.
__global__ void __launch_bounds__(kF8Threads) fp8_x_quant_kernel(const uint16_t* __restrict__ x, int H, int rpt,
                                                                 const int32_t* __restrict__ route_row,
                                                                 uint8_t* __restrict__ xq, float* __restrict__ xsig) {
  __shared__ float red[kF8Threads / 32];
  const int t = blockIdx.x;
  const uint16_t* xr = x + (int64_t)t * H;
  float m = 0.f;
  for (int i = threadIdx.x * 8; i < H; i += kF8Threads * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      m = fmaxf(m, fmaxf(fabsf(bf16_to_f32((uint16_t)(w[k] & 0xFFFFu))), fabsf(bf16_to_f32((uint16_t)(w[k] >> 16)))));
  }
  const float sig = __fdiv_rn(block_max(m, red), 448.0f);
  for (int i = threadIdx.x * 8; i < H; i += kF8Threads * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = bf16_to_f32((uint16_t)(w[k] & 0xFFFFu));
      f[2 * k + 1] = bf16_to_f32((uint16_t)(w[k] >> 16));
    }
    const uint2 c = make_uint2(fp8_pack4(f[0], f[1], f[2], f[3], sig), fp8_pack4(f[4], f[5], f[6], f[7], sig));
    for (int j = 0; j < rpt; ++j) *reinterpret_cast<uint2*>(xq + (int64_t)route_row[(int64_t)t * rpt + j] * H + i) = c;
  }
  if (threadIdx.x < rpt) xsig[route_row[(int64_t)t * rpt + threadIdx.x]] = sig;
}

// One CTA per route: the intermediate row h (fp32) to E4M3 with sigma from
// the row's |max|, gathered by the gate/up epilogue.
__global__ void __launch_bounds__(kF8Threads) fp8_h_quant_kernel(const float* __restrict__ h32, int I,
                                                                 const int32_t* __restrict__ route_row,
                                                                 const uint32_t* __restrict__ amax_row,
                                                                 uint8_t* __restrict__ hq, float* __restrict__ hsig) {
  const int64_t row = route_row[blockIdx.x];
  const float sig = __fdiv_rn(__uint_as_float(amax_row[row]), 448.0f);
  const float* hr = h32 + row * I;
  for (int i = threadIdx.x * 8; i < I; i += kF8Threads * 8) {
    const float4 a = *reinterpret_cast<const float4*>(hr + i);
    const float4 b = *reinterpret_cast<const float4*>(hr + i + 4);
    *reinterpret_cast<uint2*>(hq + row * I + i) =
        make_uint2(fp8_pack4(a.x, a.y, a.z, a.w, sig), fp8_pack4(b.x, b.y, b.z, b.w, sig));
  }
  if (threadIdx.x == 0) hsig[row] = sig;
}

// ---------------------------------------------------------------- NVFP4 emulation mode
// "Serving NVFP4 models on AMD Instinct MI355 accelerators", sections "Weight
// Dequantization and Activation QDQ" and "Memory Management": weights are
// dequantised to BF16 at GEMM time (for MoE only the dispatched experts) and
// activations pass through an NVFP4 quantise-dequantise round trip.  Each
// BF16 value is bf16_rn(fp32(E2M1(q) * fp32(E4M3(s) * g))).

// fp32(E2M1(c) * d) for a 4-bit code: twice the magnitude from a nibble
// table (0, 1, 2, 3, 4, 6, 8, 12), halved exactly, times d, the sign bit of
// the code moved to bit 31.  Equal to e2m1_val(c) * d.
__device__ __forceinline__ float e2m1_times(uint32_t c, float d) {
  const float mag = (float)((0xC8643210u >> (4u * (c & 7u))) & 15u) * 0.5f;
  return __uint_as_float(__float_as_uint(__fmul_rn(mag, d)) ^ ((c & 8u) << 28));
}

// Two fp32 values to packed bf16 (round to nearest even; low half first).
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 values of one NVFP4 block (codes: value i in nibble i) to BF16, 32 bytes.
__device__ __forceinline__ void nv_block_bf16(uint64_t codes, uint32_t sbyte, float g, uint4* dst) {
  const float d = __fmul_rn(e4m3_value(sbyte), g);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = bf16x2_rn(e2m1_times((uint32_t)(codes >> (8 * i)) & 0xFu, d),
                     e2m1_times((uint32_t)(codes >> (8 * i + 4)) & 0xFu, d));
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Weights of n_mat matrices [rows, K] (codes [n_mat, rows, K/2], scales in
// the tiled layout, tensor scale g[m]) to bf16 [n_mat, rows, K]; matrices
// whose expert has no routes (count[m] == 0) are skipped.  Grid: (.., n_mat).
constexpr int kDqBlocksPerThread = 4;
__global__ void nv_weight_bf16_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                      const float* __restrict__ g, int rows, int K, bool tiled, int pairs,
                                      const int32_t* __restrict__ count, uint16_t* __restrict__ out) {
  const int m = blockIdx.y;
  if (count && count[m] == 0) return;
  const int per_row = K >> 4;
  const int64_t katoms = katoms_padded(K, true);
  const float gm = g[m];
  const int64_t n = (int64_t)rows * per_row;
  // consecutive threads take consecutive blocks, so a warp's loads and its
  // 32-byte stores are contiguous
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, j = 0; j < kDqBlocksPerThread && i < n;
       i += stride, ++j) {
    const int64_t r = (int64_t)m * rows + i / per_row;  // row over all matrices
    const int b = (int)(i % per_row);
    const int64_t off = tiled ? w_tiled_offset(r, 8 * b, (K + 255) >> 8, pairs) : r * (K >> 1) + 8 * b;
    const uint64_t c = *reinterpret_cast<const uint64_t*>(codes + off);
    const int64_t so = pairs ? sf_tiled_offset_gu(r, b, katoms, atoms_per_ktile(true), pairs) : sf_tiled_offset(r, b, katoms);
    nv_block_bf16(c, sf[so], gm, reinterpret_cast<uint4*>(out + r * K + 16 * b));
  }
}

// x through NVFP4 QDQ into every route row of its token, as bf16 [rows, H]:
// one thread per (token, 32 values); tensor scale from the amax of x.
__global__ void nv_qdq_x_bf16_kernel(const uint16_t* __restrict__ x, int T, int H, int rpt,
                                     const int32_t* __restrict__ route_row, const uint32_t* __restrict__ amax_x,
                                     float* __restrict__ g_out, uint16_t* __restrict__ xb) {
  const int per_row = H >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= (int64_t)T * per_row) return;
  const int64_t t = tid / per_row;
  const int b = (int)(tid - t * per_row);
  const float g = nv_global(__uint_as_float(*amax_x));
  if (tid == 0 && g_out) *g_out = g;
  float v[32];
  load32(x, 0, t * H + 32 * b, v);
  uint32_t q[4], s0, s1;
  nv_quant16(v, g, q, &s0);
  nv_quant16(v + 16, g, q + 2, &s1);
  uint4 o[4];
  nv_block_bf16((uint64_t)q[0] | (uint64_t)q[1] << 32, s0, g, o);
  nv_block_bf16((uint64_t)q[2] | (uint64_t)q[3] << 32, s1, g, o + 2);
  for (int j = 0; j < rpt; ++j) {
    uint4* dst = reinterpret_cast<uint4*>(xb + (int64_t)route_row[t * rpt + j] * H + 32 * b);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = o[k];
  }
}

// The intermediate h (fp32 [rows, I]) through NVFP4 QDQ per route row, with
// the tensor scale of the row's expert (amax_h[e] / 2688), as bf16 [rows, I];
// also stores the scales to gh_out.
__global__ void nv_qdq_h_bf16_kernel(const float* __restrict__ h32, int I, int64_t n_routes,
                                     const int32_t* __restrict__ route_row, const int32_t* __restrict__ row_e,
                                     const uint32_t* __restrict__ amax_h, float* __restrict__ gh_out, int n_exp,
                                     uint16_t* __restrict__ hb) {
  const int per_row = I >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid < n_exp && gh_out) gh_out[tid] = nv_global(__uint_as_float(amax_h[tid]));
  if (tid >= n_routes * per_row) return;
  const int64_t rt = tid / per_row;
  const int b = (int)(tid - rt * per_row);
  const int64_t row = route_row[rt];
  const float g = nv_global(__uint_as_float(amax_h[row_e[row]]));
  float v[32];
  load32(h32, 1, row * I + 32 * b, v);
  uint32_t q[4], s0, s1;
  nv_quant16(v, g, q, &s0);
  nv_quant16(v + 16, g, q + 2, &s1);
  uint4* dst = reinterpret_cast<uint4*>(hb + row * I + 32 * b);
  nv_block_bf16((uint64_t)q[0] | (uint64_t)q[1] << 32, s0, g, dst);
  nv_block_bf16((uint64_t)q[2] | (uint64_t)q[3] << 32, s1, g, dst + 2);
}

__global__ void pack_scales_kernel(const uint8_t* src, uint8_t* dst, int64_t n_mat, int rows, int kblocks,
                                   int64_t katoms, int apk, int pairs, uint8_t pad) {
  const int64_t words = n_mat * (rows / 128) * katoms * 128;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= words) return;
  const int64_t grp = tid >> 7;  // group of the destination: (matrix, row tile, atom) in tile-slot order
  const int w = (int)(tid & 127);
  const int m0 = w >> 2, m1 = w & 3;
  int64_t atom = grp % katoms;
  int64_t mt = grp / katoms;  // matrix * row tiles + row tile
  if (pairs) {  // gate/up-paired slots: slot = ((m * P + p) * KT + kt) * 2 + h, apk groups each
    const int64_t kts = katoms / apk;
    const int64_t slot = grp / apk, a = grp - slot * apk;
    const int64_t h = slot & 1, t = slot >> 1, kt = t % kts, mp = t / kts;
    const int64_t m = mp / pairs, pp = mp - m * pairs;
    mt = m * 2 * pairs + h * pairs + pp;
    atom = kt * apk + a;
  }
  const int64_t row = mt * 128 + 32 * m1 + m0;  // global row over all matrices
  uint32_t word = 0;
#pragma unroll
  for (int k1 = 0; k1 < 4; ++k1) {
    const int64_t kb = atom * 4 + k1;
    const uint32_t byte = kb < kblocks ? src[row * kblocks + kb] : pad;
    word |= byte << (8 * k1);
  }
  reinterpret_cast<uint32_t*>(dst)[grp * 128 + 4 * m0 + m1] = word;
}

// ---------------------------------------------------------------- combine finaliser
__global__ void finalize_kernel(const float* acc, uint16_t* out, int64_t n) {
  pdl_wait();
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    const float4 v = *reinterpret_cast<const float4*>(acc + i);
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_rn(v.x) | ((uint32_t)f32_to_bf16_rn(v.y) << 16);
    o.y = (uint32_t)f32_to_bf16_rn(v.z) | ((uint32_t)f32_to_bf16_rn(v.w) << 16);
    *reinterpret_cast<uint2*>(out + i) = o;
  } else {
    for (int64_t j = i; j < n; ++j) out[j] = f32_to_bf16_rn(acc[j]);
  }
}

// ---------------------------------------------------------------- MXFP4 -> FP8 conversion
// E4M3 byte of one E2M1 code with block exponent sb (scale byte - 127) under
// channel shift k.  *low is set when a non-zero element lands below 2^-5.
__device__ __forceinline__ uint32_t conv_nibble(uint32_t c, int sb, int k, bool* low) {
  const uint32_t mag = c & 7u, sign = (c & 8u) << 4;
  if (mag == 0) return sign;
  const int x = (int)(mag >> 1) - 1 + sb - k;  // element exponent after the shift
  const uint32_t m = (mag > 1u) ? (mag & 1u) : 0u;  // significand 1.0 or 1.5
  if (x < -5) *low = true;
  if (x >= -6) return sign | ((uint32_t)(x + 7) << 3) | (m << 2);
  // E4M3 subnormal: value (2 + m) * 2^(x - 1) in units of 2^-9 is (2 + m) * 2^(x + 8)
  const uint32_t q = 2u + m;
  const int sh = -(x + 8);
  uint32_t r;
  if (sh < 0) r = q << 1;
  else if (sh == 0) r = q;
  else if (sh >= 3) r = 0;
  else {
    const uint32_t half = 1u << (sh - 1), rem = q & ((1u << sh) - 1u);
    r = (q >> sh) + ((rem > half || (rem == half && ((q >> sh) & 1u))) ? 1u : 0u);
  }
  return sign | r;
}

// Exponent class of the largest magnitude among 16 codes (two words): 0 when
// every magnitude is zero, else 1, 2, 3, 4 for a largest magnitude of 1,
// 2-3, 4-5, 6-7, whose element exponents floor(log2 v) are -1, 0, 1, 2.
__device__ __forceinline__ int half_class(uint32_t x, uint32_t y) {
  const uint32_t om = (x | y) & 0x77777777u;
  const uint32_t b21 = ((x & (x << 1)) | (y & (y << 1))) & 0x44444444u;  // a magnitude 6 or 7
  return (om != 0u) + ((om & 0x66666666u) != 0u) + ((om & 0x44444444u) != 0u) + (b21 != 0u);
}

// Eight codes -> eight E4M3 bytes (two words).  Magnitude by table lookup:
// each code's low three bits select a byte of the block table (tlo, thi).
// Sign: bit 3 of even codes moves to bit 7 of a byte after a 4-bit shift,
// bit 3 of odd codes already sits at bit 7 of a byte; a byte permute
// interleaves them into code order.
__device__ __forceinline__ void conv8(uint32_t w, uint32_t tlo, uint32_t thi, uint32_t& o0, uint32_t& o1) {
  const uint32_t m = w & 0x77777777u, e = w << 4;
  o0 = __byte_perm(tlo, thi, m) | (__byte_perm(e, w, 0x5140) & 0x80808080u);
  o1 = __byte_perm(tlo, thi, m >> 16) | (__byte_perm(e, w, 0x7362) & 0x80808080u);
}

// Nonzero when some code of w has magnitude in [1, j], where c = (7 - j) in
// every nibble: adding 7 to a 3-bit magnitude carries into the nibble's top
// bit iff it is at least 1, adding 7 - j iff it exceeds j.  c = 0x77777777
// (j = 0) gives zero.
__device__ __forceinline__ uint32_t small_codes(uint32_t w, uint32_t c) {
  const uint32_t m = w & 0x77777777u;
  return (m + 0x77777777u) & ~(m + c) & 0x88888888u;
}

// The E4M3 byte of magnitude m under a block depends only on the block's
// exponent relative to the row shift, delta = (scale - 127) - k.  A block
// holding a nonzero code has delta <= 8 (its largest element is at most the
// row's largest, exponent k + 7); at delta <= -13 every nonzero magnitude is
// below half the smallest E4M3 subnormal, so all deltas under the table's
// range give the same bytes as its first entry, and deltas above it only
// occur for blocks whose codes are all zero.  The magnitudes that land below
// the normal range are always 1..j for some j (the exponent grows with the
// magnitude); the table keeps (7 - j) in every nibble.
constexpr int kDeltaLo = -16, kDeltaN = 32;

// Rows are spread over a persistent grid, one warp per row at a time.  Lane
// l handles the 16-code halves l, l + 32, ... of the row (NPER of them).
// Each warp double-buffers code rows in shared memory with cp.async: the
// next row's codes (and, into registers, its scale bytes) are in flight while
// the current row is encoded.  Rows longer than 8192 codes go to a plain
// two-pass kernel over global memory.
constexpr int kConvWarps = 8;
constexpr int kConvRowBytes = 4096;
constexpr int kConvSmem = kConvWarps * 2 * kConvRowBytes;
constexpr int kConvMaxPer = kConvRowBytes / (8 * 32);  // 16 halves per lane

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct ConvTables {
  uint2 mag[kDeltaN];      // E4M3 bytes of magnitudes 0..3 (x) and 4..7 (y)
  uint32_t small[kDeltaN];  // (7 - j) per nibble, magnitudes 1..j below the normal range
};

__device__ __forceinline__ void build_tables(ConvTables& t) {
  if (threadIdx.x < kDeltaN) {
    uint32_t l = 0, h = 0, j = 0;
    const int delta = kDeltaLo + (int)threadIdx.x;
    for (uint32_t m = 0; m < 8; ++m) {
      bool f = false;
      const uint32_t byte = conv_nibble(m, delta, 0, &f);
      if (m < 4) l |= byte << (8 * m);
      else h |= byte << (8 * (m - 4));
      if (f) j = m;
    }
    t.mag[threadIdx.x] = make_uint2(l, h);
    t.small[threadIdx.x] = (7u - j) * 0x11111111u;
  }
  __syncthreads();
}

// Row results: per-row status byte, power-of-two scale, global status word.
__device__ __forceinline__ void finish_row(int64_t row, bool nan, bool low, int k, float* row_scale,
                                           uint8_t* row_status, int32_t* status) {
  const uint32_t st = nan ? 2u : (low ? 1u : 0u);
  if (row_status) row_status[row] = (uint8_t)st;
  float sc;
  if (nan) sc = __uint_as_float(0x7FC00000u);
  else if (k >= -126) sc = __uint_as_float((uint32_t)(k + 127) << 23);
  else sc = __uint_as_float(1u << (k + 149));  // fp32 subnormal, exact
  row_scale[row] = sc;
  if (st == 2u) record_status(status, FP4MOE_ERR_NAN_SCALE, ST_NAN);
  if (st == 1u) record_status(status, FP4MOE_ERR_INEXACT, ST_INEXACT);
}

// Row-wide reductions of pass 1.  top = max over halves of (class + scale)
// for nonzero halves (0 when the row is all zero): the row's largest element
// exponent is top - 129.  smin = least scale of a nonzero half (255 if none),
// smax = largest scale byte (255 marks a NaN scale).
struct RowStats {
  uint32_t top = 0, smin = 255, smax = 0;
  __device__ __forceinline__ void add(uint2 w, uint32_t sc) {
    const uint32_t c = (uint32_t)half_class(w.x, w.y);
    top = max(top, c ? c + sc : 0u);
    smin = min(smin, c ? sc : 255u);
    smax = max(smax, sc);
  }
  __device__ __forceinline__ void reduce() {
    top = __reduce_max_sync(0xffffffffu, top);
    smin = __reduce_min_sync(0xffffffffu, smin);
    smax = __reduce_max_sync(0xffffffffu, smax);
  }
  // shift k = (largest element exponent) - 7
  __device__ __forceinline__ int shift() const { return top ? (int)top - 136 : 0; }
  // A nonzero code lands below the normal range only if its element exponent
  // (at least smin - 128) is under k - 5.
  __device__ __forceinline__ bool maybe_low() const { return top && (int)smin - 128 < shift() - 5; }
};

template <int NPER>
__global__ void __launch_bounds__(32 * kConvWarps, 3) convert_kernel(const uint8_t* codes, const uint8_t* scales,
                                                                     int64_t rows, int K, uint8_t* out,
                                                                     float* row_scale, uint8_t* row_status,
                                                                     int32_t* status) {
  extern __shared__ __align__(16) uint8_t conv_smem[];
  __shared__ ConvTables tab;
  build_tables(tab);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * kConvWarps;
  const int nhalf = K >> 4, nchunk = K >> 5;  // 8-byte halves and 16-byte chunks of a code row
  const bool last_ok = lane + 32 * (NPER - 1) < nhalf;  // only the last half per lane can be past the row
  int64_t row = (int64_t)blockIdx.x * kConvWarps + warp;

  uint8_t* wbuf = conv_smem + warp * 2 * kConvRowBytes;
  uint32_t cs[NPER], ns[NPER];
  auto stage = [&](int64_t r, int b, uint32_t* sdst) {
    const uint8_t* src = codes + r * (K >> 1);
    const uint32_t dst = smem_u32(wbuf + b * kConvRowBytes);
    for (int c = lane; c < nchunk; c += 32) cp_async16(dst + 16 * c, src + 16 * c);
    const uint8_t* srow = scales + r * (K >> 5) + (lane >> 1);
#pragma unroll
    for (int i = 0; i < NPER; ++i)
      if (i < NPER - 1 || last_ok) sdst[i] = __ldg(srow + 16 * i);
  };
  if (row < rows) stage(row, 0, cs);
  cp_async_commit();
  int buf = 0;
  for (; row < rows; row += nwarps) {
    const int64_t next = row + nwarps;
    if (next < rows) stage(next, buf ^ 1, ns);
    cp_async_commit();
    cp_async_wait<1>();  // this row's group has landed (the next row's may still fly)
    __syncwarp();
    const uint2* cur = reinterpret_cast<const uint2*>(wbuf + buf * kConvRowBytes) + lane;
    RowStats rs;
#pragma unroll
    for (int i = 0; i < NPER; ++i)
      if (i < NPER - 1 || last_ok) rs.add(cur[32 * i], cs[i]);
    rs.reduce();
    const bool nan = rs.smax == 255u;
    const int k = rs.shift();
    uint4* orow = reinterpret_cast<uint4*>(out + row * K) + lane;
    const int base = 127 + k + kDeltaLo;
    uint32_t lowacc = 0;
    if (nan) {
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (i < NPER - 1 || last_ok) orow[32 * i] = make_uint4(0u, 0u, 0u, 0u);
    } else if (!rs.maybe_low()) {
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (i < NPER - 1 || last_ok) {
          const uint2 w = cur[32 * i];
          const uint2 t = tab.mag[min(max((int)cs[i] - base, 0), kDeltaN - 1)];
          uint4 o;
          conv8(w.x, t.x, t.y, o.x, o.y);
          conv8(w.y, t.x, t.y, o.z, o.w);
          orow[32 * i] = o;
        }
    } else {
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (i < NPER - 1 || last_ok) {
          const uint2 w = cur[32 * i];
          const int idx = min(max((int)cs[i] - base, 0), kDeltaN - 1);
          const uint2 t = tab.mag[idx];
          const uint32_t c = tab.small[idx];
          lowacc |= small_codes(w.x, c) | small_codes(w.y, c);
          uint4 o;
          conv8(w.x, t.x, t.y, o.x, o.y);
          conv8(w.y, t.x, t.y, o.z, o.w);
          orow[32 * i] = o;
        }
    }
    const bool low = __any_sync(0xffffffffu, lowacc != 0u);
    if (lane == 0) finish_row(row, nan, low, k, row_scale, row_status, status);
#pragma unroll
    for (int i = 0; i < NPER; ++i) cs[i] = ns[i];
    buf ^= 1;
    __syncwarp();  // every lane is done with this buffer before it is refilled
  }
  cp_async_wait<0>();
}

// Rows longer than the staging buffer: pass 1 and pass 2 both read global
// memory.
__global__ void __launch_bounds__(32 * kConvWarps) convert_long_kernel(const uint8_t* codes, const uint8_t* scales,
                                                                       int64_t rows, int K, uint8_t* out,
                                                                       float* row_scale, uint8_t* row_status,
                                                                       int32_t* status) {
  __shared__ ConvTables tab;
  build_tables(tab);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * kConvWarps;
  const int nhalf = K >> 4;
  for (int64_t row = (int64_t)blockIdx.x * kConvWarps + (threadIdx.x >> 5); row < rows; row += nwarps) {
    const uint2* crow = reinterpret_cast<const uint2*>(codes + row * (K >> 1));
    const uint8_t* srow = scales + row * (K >> 5);
    RowStats rs;
    for (int h = lane; h < nhalf; h += 32) rs.add(__ldg(crow + h), __ldg(srow + (h >> 1)));
    rs.reduce();
    const bool nan = rs.smax == 255u;
    const int k = rs.shift();
    const int base = 127 + k + kDeltaLo;
    uint4* orow = reinterpret_cast<uint4*>(out + row * K);
    uint32_t lowacc = 0;
    for (int h = lane; h < nhalf; h += 32) {
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (!nan) {
        const uint2 w = __ldg(crow + h);
        const int idx = min(max((int)__ldg(srow + (h >> 1)) - base, 0), kDeltaN - 1);
        const uint2 t = tab.mag[idx];
        lowacc |= small_codes(w.x, tab.small[idx]) | small_codes(w.y, tab.small[idx]);
        conv8(w.x, t.x, t.y, o.x, o.y);
        conv8(w.y, t.x, t.y, o.z, o.w);
      }
      orow[h] = o;
    }
    const bool low = __any_sync(0xffffffffu, lowacc != 0u);
    if (lane == 0) finish_row(row, nan, low, k, row_scale, row_status, status);
  }
}

using ConvKernel = void (*)(const uint8_t*, const uint8_t*, int64_t, int, uint8_t*, float*, uint8_t*, int32_t*);

template <int... P>
constexpr std::array<ConvKernel, sizeof...(P)> conv_kernels(std::integer_sequence<int, P...>) {
  return {convert_kernel<P + 1>...};
}

inline unsigned blocks_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_amax(const void* x, int x_is_fp32, int64_t n, uint32_t* amax_bits, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (n == 0) return cudaSuccess;
  int blocks = (int)std::min<int64_t>(blocks_for(n, 256), 4 * 152);
  amax_kernel<<<blocks, 256, 0, s>>>(x, x_is_fp32, n, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void* x, int x_is_fp32, int64_t rows, int cols, bool nv,
                                 const float* global_in, const uint32_t* amax_bits, uint8_t* codes,
                                 uint8_t* scales, float* global_out, cudaStream_t s) {
  const int64_t n = rows * (cols >> 5);
  if (n == 0) return cudaSuccess;
  quantize_rows_kernel<<<blocks_for(n, 256), 256, 0, s>>>(x, x_is_fp32, rows, cols, nv ? 1 : 0, global_in,
                                                           amax_bits, codes, scales, global_out);
  return cudaGetLastError();
}

cudaError_t launch_gather_quant(const fp4moe_dims& d, const uint16_t* x, const int32_t* route_row, uint8_t* xq,
                                uint8_t* xsf, const uint32_t* amax_x, float* g_out, cudaStream_t s) {
  const int rpt = d.top_k + d.n_shared;
  const int64_t n = (int64_t)d.T * (d.H >> 5);
  if (n == 0) return cudaSuccess;
  return launch_pdl(gather_quant_kernel, dim3(blocks_for(n, 256)), dim3(256), 0, s, x, d.T, d.H, rpt, route_row,
                    xq, xsf, (int)(d.fmt == FP4MOE_NVFP4), amax_x, g_out);
}

cudaError_t launch_h_quant_nv_routes(const fp4moe_dims& d, const float* h32, const int32_t* route_row,
                                     const int32_t* row_e, const uint32_t* amax_h, float* gh_out, uint8_t* hq,
                                     uint8_t* hsf, cudaStream_t s) {
  const int rpt = d.top_k + d.n_shared;
  const int64_t n_routes = (int64_t)d.T * rpt;
  const int64_t n = std::max<int64_t>(n_routes * (d.I >> 5), d.E + d.n_shared);
  h_quant_nv_kernel<<<blocks_for(n, 256), 256, 0, s>>>(h32, d.I, n_routes, route_row, row_e, amax_h, gh_out, hq,
                                                        hsf, d.E + d.n_shared);
  return cudaGetLastError();
}

cudaError_t launch_fp8_x_quant(const fp4moe_dims& d, const uint16_t* x, const int32_t* route_row, uint8_t* xq,
                               float* xsig, cudaStream_t s) {
  if (d.T <= 0) return cudaSuccess;
  fp8_x_quant_kernel<<<(unsigned)d.T, kF8Threads, 0, s>>>(x, d.H, d.top_k + d.n_shared, route_row, xq, xsig);
  return cudaGetLastError();
}

cudaError_t launch_fp8_h_quant(const fp4moe_dims& d, const float* h32, const int32_t* route_row,
                               const uint32_t* amax_row, uint8_t* hq, float* hsig, cudaStream_t s) {
  const int64_t n_routes = (int64_t)d.T * (d.top_k + d.n_shared);
  if (n_routes <= 0) return cudaSuccess;
  fp8_h_quant_kernel<<<(unsigned)n_routes, kF8Threads, 0, s>>>(h32, d.I, route_row, amax_row, hq, hsig);
  return cudaGetLastError();
}

cudaError_t launch_nv_weight_bf16(const uint8_t* codes, bool tiled, int pairs, const uint8_t* sf, const float* g,
                                  int n_mat, int rows, int K, const int32_t* count, uint16_t* out, cudaStream_t s) {
  if (n_mat <= 0) return cudaSuccess;
  const int64_t n = (int64_t)rows * (K >> 4);
  const dim3 grid((unsigned)blocks_for((n + kDqBlocksPerThread - 1) / kDqBlocksPerThread, 256), (unsigned)n_mat);
  nv_weight_bf16_kernel<<<grid, 256, 0, s>>>(codes, sf, g, rows, K, tiled, pairs, count, out);
  return cudaGetLastError();
}

cudaError_t launch_nv_qdq_x_bf16(const fp4moe_dims& d, const uint16_t* x, const int32_t* route_row,
                                 const uint32_t* amax_x, float* g_out, uint16_t* xb, cudaStream_t s) {
  const int64_t n = (int64_t)d.T * (d.H >> 5);
  if (n == 0) return cudaSuccess;
  nv_qdq_x_bf16_kernel<<<blocks_for(n, 256), 256, 0, s>>>(x, d.T, d.H, d.top_k + d.n_shared, route_row, amax_x,
                                                          g_out, xb);
  return cudaGetLastError();
}

cudaError_t launch_nv_qdq_h_bf16(const fp4moe_dims& d, const float* h32, const int32_t* route_row,
                                 const int32_t* row_e, const uint32_t* amax_h, float* gh_out, uint16_t* hb,
                                 cudaStream_t s) {
  const int64_t n_routes = (int64_t)d.T * (d.top_k + d.n_shared);
  const int n_exp = d.E + d.n_shared;
  const int64_t n = std::max<int64_t>(n_routes * (d.I >> 5), n_exp);
  nv_qdq_h_bf16_kernel<<<blocks_for(n, 256), 256, 0, s>>>(h32, d.I, n_routes, route_row, row_e, amax_h, gh_out,
                                                          n_exp, hb);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(finalize_kernel, dim3(blocks_for((n + 3) / 4, 256)), dim3(256), 0, s, acc, out, n);
}

// Row-major FP4 payloads [rows_total, kbytes] -> the tiled layout (see
// w_tiled_offset): one thread per 16 bytes of the output, so a warp writes
// 512 contiguous bytes and reads four 128-byte row pieces; bytes past
// kbytes (K padded to whole K tiles) are zero codes.
__global__ void pack_weights_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t n16,
                                    int kbytes, int ktb, int pairs) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = i >> 10;          // 1024 pieces of 16 bytes per 128 x 128-byte block (tile slot)
    int64_t rt = blk / ktb, kt = blk % ktb;
    if (pairs) {  // gate/up-paired slots: slot = ((m * P + p) * KT + kt) * 2 + h
      const int64_t h = blk & 1, t = blk >> 1, mp = t / ktb, m = mp / pairs, pp = mp - m * pairs;
      kt = t - mp * ktb;
      rt = m * 2 * pairs + h * pairs + pp;
    }
    const int64_t r = rt * 128 + ((i >> 3) & 127);
    const int cb = (int)kt * 128 + (int)(i & 7) * 16;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (cb < kbytes) v = *reinterpret_cast<const uint4*>(src + r * kbytes + cb);
    reinterpret_cast<uint4*>(dst)[i] = v;
  }
}

cudaError_t launch_pack_weights(const uint8_t* src, uint8_t* dst, int64_t rows_total, int kbytes, int pairs,
                                cudaStream_t s) {
  const int ktb = (kbytes + 127) / 128;
  const int64_t n16 = rows_total * ktb * 8;
  if (n16 == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>(blocks_for(n16, 256), 1 << 20);
  pack_weights_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, dst, n16, kbytes, ktb, pairs);
  return cudaGetLastError();
}

// Counts the NaN scale bytes of n bytes (E8M0: 255; E4M3: magnitude bits
// 0x7F) and records them in the status word as FP4MOE_ERR_NAN_SCALE.
__global__ void nan_scales_kernel(const uint8_t* __restrict__ src, int64_t n, int nv, int32_t* status) {
  __shared__ int s_cnt;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  int cnt = 0;
  const int64_t n16 = n / 16, stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (w[j] >> (8 * b)) & 0xFFu;
        cnt += nv ? ((byte & 0x7Fu) == 0x7Fu) : (byte == 0xFFu);
      }
  }
  for (int64_t i = n16 * 16 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint32_t byte = src[i];
    cnt += nv ? ((byte & 0x7Fu) == 0x7Fu) : (byte == 0xFFu);
  }
  if (cnt) atomicAdd(&s_cnt, cnt);
  __syncthreads();
  if (threadIdx.x == 0 && s_cnt) record_status(status, FP4MOE_ERR_NAN_SCALE, ST_NAN, s_cnt);
}

cudaError_t launch_nan_scales(const uint8_t* src, int64_t n, bool nv, int32_t* status, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t want = (n / 16 + 255) / 256;
  const unsigned blocks = (unsigned)(want < 4 * 152 ? (want > 0 ? want : 1) : 4 * 152);
  nan_scales_kernel<<<blocks, 256, 0, s>>>(src, n, nv ? 1 : 0, status);
  return cudaGetLastError();
}

cudaError_t launch_pack_scales(const uint8_t* src, uint8_t* dst, int64_t n_mat, int rows, int kblocks, bool nv,
                               int pairs, cudaStream_t s) {
  const int64_t katoms = katoms_padded((int64_t)kblocks * (nv ? 16 : 32), nv);
  const int64_t words = n_mat * (rows / 128) * katoms * 128;
  if (words == 0) return cudaSuccess;
  pack_scales_kernel<<<blocks_for(words, 256), 256, 0, s>>>(src, dst, n_mat, rows, kblocks, katoms,
                                                            atoms_per_ktile(nv), pairs, nv ? 0x38 : 127);
  return cudaGetLastError();
}

cudaError_t launch_convert(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, uint8_t* out,
                           float* row_scale, uint8_t* row_status, int32_t* status, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  static const auto kernels = conv_kernels(std::make_integer_sequence<int, kConvMaxPer>{});
  static int resident[64][kConvMaxPer + 1] = {};  // CTAs per SM, per device and kernel
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int nper = ((K >> 4) + 31) / 32;
  const bool staged = nper <= kConvMaxPer;
  const ConvKernel kern = staged ? kernels[nper - 1] : convert_long_kernel;
  const int slot = staged ? nper : 0;
  const int smem = staged ? kConvSmem : 0;
  if (!resident[dev][slot]) {
    int n = 0;
    cudaError_t e = staged ? cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                           : cudaSuccess;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * kConvWarps, smem);
    if (e != cudaSuccess) return e;
    resident[dev][slot] = n > 0 ? n : 1;
  }
  const int64_t grid =
      std::min<int64_t>(blocks_for(rows, kConvWarps), (int64_t)device_sm_count() * resident[dev][slot]);
  kern<<<(unsigned)grid, 32 * kConvWarps, smem, s>>>(codes, scales, rows, K, out, row_scale, row_status, status);
  return cudaGetLastError();
}

}  // namespace fp4moe
