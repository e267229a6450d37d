// Host side of the grouped GEMMs: tensor maps, parameter block and the
// choice of template instance.
#pragma once

#include "gemm.cuh"

namespace fp4moe {

// L2 bytes the down GEMM's combine rows of one unit group may take (of the
// 126 MB): the group's G weight tiles x their rows x T tokens x fp32.
constexpr int64_t kCombineL2Bytes = 48ll << 20;
// Combine buffers up to this size keep the expert-major order: measured, a
// 4096-token layer (117 MB) gained nothing from groups, a 16384-token layer
// (470 MB) 19% of its down GEMM.
constexpr int64_t kCombineGroupAbove = 256ll << 20;

// Weight tiles (of tile_rows rows) per group of the down GEMM's unit order:
// the largest divisor of M whose combine rows fit kCombineL2Bytes; M
// (expert-major) when the whole buffer is small, or when each token has one
// route, so that no row is added twice.
inline int combine_group(int M, int64_t T, int routes_per_token, int tile_rows) {
  const int64_t row_bytes = (int64_t)tile_rows * 4;  // fp32 combine row slice of one tile
  if (routes_per_token <= 1 || T * M * row_bytes <= kCombineGroupAbove) return M;
  int g = 1;
  for (int c = 1; c <= M; ++c)
    if (M % c == 0 && T * c * row_bytes <= kCombineL2Bytes) g = c;
  return g;
}

// The block-scaled FP4 instances (MXFP4 / NVFP4); DPW: down weights in the
// row-tile-paired order.
template <bool GATEUP, bool DPW>
cudaError_t launch_fp4(const GemmArgs& a, KParams& p, int vis, int grid, cudaStream_t s) {
  if constexpr (!GATEUP) {
    if (a.dn_w2) {  // MXFP4, 112-token tiles: two weight tiles per unit
      if (a.n_tile != 112 || a.nv || a.dn_pair != 1 || a.dn_cta_pair || vis % 256 != 0) return cudaErrorInvalidValue;
      if (p.m_group < p.unit_mtiles) return launch_gemm_t<112, false, false, kOpFp4, false, true, true, DPW>(p, grid, s);
      return launch_gemm_t<112, false, false, kOpFp4, false, false, true, DPW>(p, grid, s);
    }
    if (a.dn_pair == 2) {  // MXFP4, 112-token tiles: two slots per unit
      if (a.n_tile != 112 || a.nv || a.f8 || a.bf) return cudaErrorInvalidValue;
      if (a.dn_cta_pair) {
        if (vis % 256 != 0) return cudaErrorInvalidValue;
        p.m_group = p.unit_mtiles;  // (expert-major order only)
        return launch_gemm_t<240, false, false, kOpFp4, true, false, false, DPW>(p, grid, s);
      }
      if (p.m_group < p.unit_mtiles) return launch_gemm_t<240, false, false, kOpFp4, false, true, false, DPW>(p, grid, s);
      return launch_gemm_t<240, false, false, kOpFp4, false, false, false, DPW>(p, grid, s);
    }
  }
  switch (a.n_tile * 2 + (a.nv ? 1 : 0)) {
    case 32: return launch_gemm_t<16, GATEUP, false, kOpFp4, false, false, false, DPW>(p, grid, s);  // few tokens (MXFP4)
    case 64: return launch_gemm_t<32, GATEUP, false, kOpFp4, false, false, false, DPW>(p, grid, s);
    case 65: return launch_gemm_t<32, GATEUP, true, kOpFp4, false, false, false, DPW>(p, grid, s);
    case 128: return launch_gemm_t<64, GATEUP, false, kOpFp4, false, false, false, DPW>(p, grid, s);
    case 129: return launch_gemm_t<64, GATEUP, true, kOpFp4, false, false, false, DPW>(p, grid, s);
    case 224: return launch_gemm_t<112, GATEUP, false, kOpFp4, false, false, false, DPW>(p, grid, s);
    case 225: return launch_gemm_t<112, GATEUP, true, kOpFp4, false, false, false, DPW>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

template <bool GATEUP>
cudaError_t launch_grouped(const GemmArgs& a, cudaStream_t s) {
  const fp4moe_dims& d = *a.d;
  KParams p;
  memset(&p, 0, sizeof(p));
  const int K = GATEUP ? d.H : d.I;
  const int rows = GATEUP ? 2 * d.I : d.H;
  // bytes of one K row: E4M3 1, BF16 2, FP4 1/2 per value
  const uint64_t Kb = a.f8 ? (uint64_t)K : a.bf ? 2 * (uint64_t)K : (uint64_t)K / 2;
  // Weights: row-major [n_mat, rows, Kb], or the tiled layout (per matrix,
  // 128-row tile and 128-byte K tile, one contiguous 16 KB block: a view of
  // 128-byte rows in which the block of (row tile rt, K tile kt) starts at
  // view row (rt * KTb + kt) * 128)
  const uint64_t KTb = (Kb + 127) / 128;
  // Down over an output-column slice: weight rows [r0, r0 + vis) of every
  // expert matrix (the maps start at row r0 and see vis rows; the matrix
  // stride stays that of all rows), and the same columns of the combine
  // buffer.  A row's bytes in memory: Kb, or whole K tiles when tiled.
  const int r0 = GATEUP ? 0 : a.row_begin;
  const int vis = (GATEUP || a.row_count <= 0) ? rows : a.row_count;
  const uint64_t a_row = a.w_tiled ? KTb * 128 : Kb;
  const uint64_t a_dim0 = a.w_tiled ? 128 : Kb, a_dim1 = a.w_tiled ? (uint64_t)vis * KTb : (uint64_t)vis;
  const uint64_t a_mat = (uint64_t)rows * a_row;
  // gate/up-paired tiles (gu_pairs): one box of 256 view rows holds the gate
  // and the up block of a (pair, K tile); likewise, for the down GEMM's
  // units of two weight tiles (W2), the two blocks of a row-tile pair
  const bool gu_paired = GATEUP && a.w_tiled && a.gu_pairs > 0;
  const bool w2 = !GATEUP && a.dn_w2;
  const bool dn_paired = !GATEUP && a.w_tiled && a.dn_paired;
  if (dn_paired && (r0 % 256 != 0 || rows % 256 != 0)) return cudaErrorInvalidValue;  // whole slabs only
  const uint32_t box_rows = (gu_paired || (w2 && dn_paired)) ? 256 : 128;
  {
    const uint64_t dims[3] = {a_dim0, a_dim1, (uint64_t)d.E};
    const uint64_t strides[2] = {a_dim0, a_mat};
    const uint32_t box[3] = {128, box_rows, 1};
    if (!encode_tmap_u8(&p.tmA, a.w + (uint64_t)r0 * a_row, 3, dims, strides, box, true)) return cudaErrorInvalidValue;
  }
  if (a.sh) {
    const uint64_t dims[3] = {a_dim0, a_dim1, 1};
    const uint64_t strides[2] = {a_dim0, a_mat};
    const uint32_t box[3] = {128, box_rows, 1};
    if (!encode_tmap_u8(&p.tmA_sh, a.sh + (uint64_t)r0 * a_row, 3, dims, strides, box, true))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {Kb, (uint64_t)a.rows_cap};
    const uint64_t strides[1] = {Kb};
    const uint32_t box[2] = {128, (uint32_t)a.n_tile};
    if (!encode_tmap_u8(&p.tmB, a.b, 2, dims, strides, box, true)) return cudaErrorInvalidValue;
  }
  // scale groups of the slice: 128-row tiles r0 / 128 on (tiled scale layout)
  const int64_t sf_r0 = (int64_t)(r0 / 128) * katoms_padded(K, a.nv) * 512;
  p.wsf = a.wsf ? a.wsf + sf_r0 : nullptr;
  p.shsf = a.shsf ? a.shsf + sf_r0 : nullptr;
  p.bsf = a.bsf;
  p.gw = a.gw;
  p.gb = a.g_b;
  p.expert_count = a.expert_count;
  p.expert_slot = a.expert_slot;
  p.unit_start = a.unit_start;
  p.total_units = GATEUP ? &a.plan->gu_units : &a.plan->dn_units;
  p.row_tok = a.row_tok;
  p.tok_mask = GATEUP ? a.tok_mask : nullptr;
  p.plan_early = a.plan_from_prev ? 0 : 1;
  p.T = d.T;
  p.row_w = a.row_w;
  p.hq = a.hq;
  p.hsf = a.hsf;
  p.h32 = a.h32;
  p.h_dbg = a.h_dbg;
  p.out_acc = a.out_acc ? a.out_acc + r0 : nullptr;  // row stride stays H
  if (GATEUP && a.zero_acc) {
    p.zero_buf = reinterpret_cast<float4*>(a.out_acc);
    p.zero_n4 = (int64_t)d.T * d.H / 4;
  }
  p.amax_h = a.amax_h;
  p.status = a.status;
  p.E = d.E;
  p.n_exp = d.E + d.n_shared;
  p.H = d.H;
  p.I = d.I;
  p.K = K;
  p.rows_per_expert = rows;
  p.m_tiles = GATEUP ? d.I / 128 : vis / 128;
  p.unit_mtiles = GATEUP ? d.I / 128 : vis / ((a.dn_cta_pair || w2) ? 256 : 128);
  // grouped unit order: the paired-slot and two-weight-tile down instances
  // only (the other instances take units expert-major)
  p.m_group = (GATEUP || (a.dn_pair != 2 && !w2))
                  ? p.unit_mtiles
                  : combine_group(p.unit_mtiles, d.T, d.top_k + d.n_shared, w2 ? 256 : 128);
  p.katoms_a = (int)katoms_padded(K, a.nv);
  p.katoms_b = (int)katoms_padded(K, a.nv);
  p.katoms_h = (int)katoms_padded(d.I, a.nv);
  p.has_shared = a.sh != nullptr;
  p.w_tiled = a.w_tiled ? 1 : 0;
  p.gu_pairs = gu_paired ? a.gu_pairs : 0;
  p.wait_ns = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  p.withhold = (GATEUP && a.withhold) ? 1 : 0;
  p.wrs = a.wrs ? a.wrs + r0 : nullptr;
  p.shrs = a.shrs ? a.shrs + r0 : nullptr;
  p.brs = a.brs;
  const int grid = a.num_sms > 0 ? a.num_sms : 1;
  if (a.f8 || a.bf) {
    if (a.nv || (a.f8 && a.bf)) return cudaErrorInvalidValue;
    if (a.f8) switch (a.n_tile) {
        case 32: return launch_gemm_t<32, GATEUP, false, kOpE4M3>(p, grid, s);
        case 64: return launch_gemm_t<64, GATEUP, false, kOpE4M3>(p, grid, s);
        case 112: return launch_gemm_t<112, GATEUP, false, kOpE4M3>(p, grid, s);
        default: return cudaErrorInvalidValue;
      }
    switch (a.n_tile) {
      case 32: return launch_gemm_t<32, GATEUP, false, kOpBf16>(p, grid, s);
      case 64: return launch_gemm_t<64, GATEUP, false, kOpBf16>(p, grid, s);
      case 112: return launch_gemm_t<112, GATEUP, false, kOpBf16>(p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if constexpr (!GATEUP)
    if (dn_paired) return launch_fp4<false, true>(a, p, vis, grid, s);
  return launch_fp4<GATEUP, false>(a, p, vis, grid, s);
}

}  // namespace fp4moe
