// Activation quantisation (MXFP4 / NVFP4), scale repacking, the fused
// gather-and-quantise step of the forward, NVFP4 requantisation of the
// intermediate, the combine finaliser, and the exact MXFP4 -> FP8 conversion.
#include <algorithm>

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
// One thread per (route, 32 values of H): quantises x[token] into the route's
// padded row of xq, with the scales in the tiled layout.
__global__ void gather_quant_kernel(const uint16_t* x, int T, int H, int routes_per_tok,
                                    const int32_t* route_row, uint8_t* xq, uint8_t* xsf, int nv,
                                    const uint32_t* amax_x, float* g_out) {
  pdl_wait();  // route_row (and the NVFP4 amax) come from the previous kernels
  pdl_trigger();
  const int per_row = H >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n_routes = (int64_t)T * routes_per_tok;
  if (tid >= n_routes * per_row) return;
  const int64_t rt = tid / per_row;
  const int b = (int)(tid - rt * per_row);
  const int64_t t = rt / routes_per_tok;
  const int64_t row = route_row[rt];
  float v[32];
  load32(x, 0, t * H + 32 * b, v);
  uint32_t p[4];
  uint4* dst = reinterpret_cast<uint4*>(xq + row * (H >> 1) + 16 * b);
  const int64_t katoms = katoms_padded(H, nv != 0);
  if (!nv) {
    uint32_t s;
    mx_quant32(v, p, &s);
    *dst = make_uint4(p[0], p[1], p[2], p[3]);
    xsf[sf_tiled_offset(row, b, katoms)] = (uint8_t)s;
  } else {
    const float g = nv_global(__uint_as_float(*amax_x));
    if (tid == 0 && g_out) *g_out = g;
    uint32_t s0, s1;
    nv_quant16(v, g, p, &s0);
    nv_quant16(v + 16, g, p + 2, &s1);
    *dst = make_uint4(p[0], p[1], p[2], p[3]);
    xsf[sf_tiled_offset(row, 2 * b, katoms)] = (uint8_t)s0;
    xsf[sf_tiled_offset(row, 2 * b + 1, katoms)] = (uint8_t)s1;
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
__global__ void pack_scales_kernel(const uint8_t* src, uint8_t* dst, int64_t n_mat, int rows, int kblocks,
                                   int64_t katoms, uint8_t pad) {
  const int64_t words = n_mat * (rows / 128) * katoms * 128;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= words) return;
  const int64_t grp = tid >> 7;  // (matrix, row tile, atom)
  const int w = (int)(tid & 127);
  const int m0 = w >> 2, m1 = w & 3;
  const int64_t atom = grp % katoms;
  const int64_t mt = grp / katoms;  // matrix * row tiles + row tile
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
// Exponent of the largest magnitude code among 8 nibbles of a word: codes
// 1..7 have exponents -1, 0, 0, 1, 1, 2, 2 (code >> 1) - 1; -100 if all zero.
__device__ __forceinline__ uint32_t max_mag_nibble(uint32_t w) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = max(m, (w >> (4 * j)) & 7u);
  return m;
}

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

// One warp per row.  Lane l handles 32-element blocks l, l + 32, ...
__global__ void convert_kernel(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, uint8_t* out,
                               float* row_scale, uint8_t* row_status, int32_t* status) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int nblk = K >> 5;
  const uint4* crow = reinterpret_cast<const uint4*>(codes + row * (K >> 1));
  const uint8_t* srow = scales + row * nblk;
  int emax = -1000;
  bool nan = false;
  for (int b = lane; b < nblk; b += 32) {
    const uint4 w = __ldg(crow + b);
    const uint32_t s = __ldg(srow + b);
    nan |= (s == 255u);
    const uint32_t m = max(max(max_mag_nibble(w.x), max_mag_nibble(w.y)), max(max_mag_nibble(w.z), max_mag_nibble(w.w)));
    if (m) emax = max(emax, (int)(m >> 1) - 1 + (int)s - 127);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
  nan = __any_sync(0xffffffffu, nan);
  const int k = emax == -1000 ? 0 : emax - 7;
  uint4* orow = reinterpret_cast<uint4*>(out + row * K);
  bool low = false;
  for (int b = lane; b < nblk; b += 32) {
    uint32_t o[8];
    if (nan) {
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = 0;
    } else {
      const uint4 w = __ldg(crow + b);
      const int sb = (int)__ldg(srow + b) - 127;
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) lo |= conv_nibble((ws[q] >> (4 * j)) & 15u, sb, k, &low) << (8 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) hi |= conv_nibble((ws[q] >> (16 + 4 * j)) & 15u, sb, k, &low) << (8 * j);
        o[2 * q] = lo;
        o[2 * q + 1] = hi;
      }
    }
    orow[2 * b] = make_uint4(o[0], o[1], o[2], o[3]);
    orow[2 * b + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  low = __any_sync(0xffffffffu, low);
  if (lane == 0) {
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
  const int64_t n = (int64_t)d.T * rpt * (d.H >> 5);
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

cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(finalize_kernel, dim3(blocks_for((n + 3) / 4, 256)), dim3(256), 0, s, acc, out, n);
}

cudaError_t launch_pack_scales(const uint8_t* src, uint8_t* dst, int64_t n_mat, int rows, int kblocks, bool nv,
                               cudaStream_t s) {
  const int64_t katoms = katoms_padded((int64_t)kblocks * (nv ? 16 : 32), nv);
  const int64_t words = n_mat * (rows / 128) * katoms * 128;
  if (words == 0) return cudaSuccess;
  pack_scales_kernel<<<blocks_for(words, 256), 256, 0, s>>>(src, dst, n_mat, rows, kblocks, katoms,
                                                            nv ? 0x38 : 127);
  return cudaGetLastError();
}

cudaError_t launch_convert(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, uint8_t* out,
                           float* row_scale, uint8_t* row_status, int32_t* status, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int warps = 8;
  convert_kernel<<<blocks_for(rows, warps), 32 * warps, 0, s>>>(codes, scales, rows, K, out, row_scale, row_status,
                                                                status);
  return cudaGetLastError();
}

}  // namespace fp4moe
