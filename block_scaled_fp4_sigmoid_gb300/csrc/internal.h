// Host-side interfaces between the translation units of libfp4moe.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fp4moe.h"

namespace fp4moe {

constexpr int kSlotRows = 128;    // rows of one slot of the permuted layout
constexpr int kChunkTokens = 32;  // tokens per chunk of the stable scatter (one warp each)

// Device-side plan of one forward call, written by the plan kernel.
struct Plan {
  int32_t n_exp;         // E + n_shared
  int32_t gu_units;      // gate/up work units
  int32_t dn_units;      // down work units
  int32_t slots;         // 128-row slots in use
};

// Everything the kernels of one forward call need to know about the workspace.
struct Layout {
  fp4moe_ws_layout ws;
  int64_t chunk_counts;  // int32 [n_chunks, n_exp]
  int64_t plan;          // Plan
  int64_t gu_start;      // int32 [n_exp + 1] prefix of gate/up units
  int64_t dn_start;      // int32 [n_exp + 1] prefix of down units
  int64_t row_e;         // int32 [rows_cap] expert of each row
  int64_t amax;          // uint32 [2 + n_exp] amax bits (x, spare, h per expert)
  bool front;            // few-token MXFP4 forward uses the fused front end
  int front_splits;      // K splits of the front end's router GEMV (cluster size)
  int n_exp, n_chunks, n_route_per_tok;
};

bool make_layout(const fp4moe_dims& d, Layout* L);

// FP4MOE_OK for cudaSuccess, else FP4MOE_ERR_CUDA.
fp4moe_status cuda_status(cudaError_t e);
// FP4MOE_OK when the current device is sm_103 (the kernels use sm_103a
// instructions), else FP4MOE_ERR_DEVICE; every attribute query checked.
fp4moe_status check_device();

// ------------------------------------------------------------- launchers
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* wr, float* partial, int T, int H, int E,
                                 int n_splits, int32_t* status, cudaStream_t s);
// tcgen05 bf16 router GEMM (T > 16): tiles of 128 tokens x router_tc_n(E) experts
cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* wr, float* partial, int T, int H, int E, int n_splits,
                             int32_t* status, cudaStream_t s);
int router_tc_n(int E);
// logits_out / scores_out (nullable): fp32 [T, E] summed logits and sigmoid scores
cudaError_t launch_topk(const fp4moe_dims& d, const float* partial, int n_splits, const float* bias,
                        int32_t* idx, float* w, float* logits_out, float* scores_out, int32_t* chunk_counts,
                        int n_exp, cudaStream_t s);
// dn_mtiles: 128-column tiles of the layer output the down GEMM computes
// (H / 128 for the whole output); dn_pair: tiles (slots) per down unit
cudaError_t launch_plan(const fp4moe_dims& d, int32_t* chunk_counts, int n_chunks, int n_exp, int n_tile, int dn_pair,
                        int dn_mtiles, int32_t* expert_count, int32_t* expert_slot, int32_t* gu_start,
                        int32_t* dn_start, Plan* plan, int32_t* ticket, cudaStream_t s);
// Dense linear: one expert holding every token in order, weight 1; zeroes acc
// (acc_n floats, a multiple of 4)
cudaError_t launch_linear_plan(int T, int n_tile, int dn_pair, int m_tiles, int32_t* count, int32_t* slot,
                               int32_t* dn_start,
                               Plan* plan, int32_t* route_row, int32_t* row_tok, float* row_w, float* acc,
                               int64_t acc_n, cudaStream_t s);
cudaError_t launch_scatter(const fp4moe_dims& d, const int32_t* idx, const float* w, const int32_t* chunk_counts,
                           int n_chunks, int n_exp, int n_tile, const int32_t* expert_slot, int32_t* route_row,
                           int32_t* row_tok, float* row_w, int32_t* row_e, cudaStream_t s);
// Fused router + top-k + plan + scatter for few tokens (MXFP4, T <= 16):
// one launch instead of four.
struct FrontArgs {
  fp4moe_dims d;  // by value: the kernel reads it
  const uint16_t *x, *wr;
  const float* bias;
  float* partial;
  int n_splits, n_tile, n_exp;  // n_splits: K splits (cluster size, <= 8), H / n_splits <= kFrontMaxKc
  int dn_mtiles;                 // 128-column tiles of the output the down GEMM computes
  float* out_acc;                // zeroed here
  int32_t* idx;
  float* w;
  int32_t *expert_count, *expert_slot, *gu_start, *dn_start;
  Plan* plan;
  int32_t *route_row, *row_tok, *row_e;
  float* row_w;
  int32_t* ticket;  // zero on entry
  uint8_t *xq, *xsf;     // quantised x: token rows (slot 0 of the permuted layout)
  uint32_t* tok_mask;    // [n_exp] bit t: token t routes to the expert
  float *logits_dbg, *scores_dbg;  // nullable: fp32 [T, E] logits and sigmoid scores
  // weights that do not depend on routing (the shared expert's), pulled
  // into L2 by the helper CTAs while the last CTA routes; nullable
  const uint8_t* l2_pf[4];
  int64_t l2_pf_bytes[4];
};
constexpr int kFrontMaxT = 16;
constexpr int kFrontMaxKc = 2048;  // router columns per split of the front end
cudaError_t launch_decode_front(const FrontArgs& a, cudaStream_t s);

cudaError_t launch_amax(const void* x, int x_is_fp32, int64_t n, uint32_t* amax_bits, cudaStream_t s);
cudaError_t launch_gather_quant(const fp4moe_dims& d, const uint16_t* x, const int32_t* route_row, uint8_t* xq,
                                uint8_t* xsf, const uint32_t* amax_x, float* g_out, cudaStream_t s);
cudaError_t launch_h_quant_nv_routes(const fp4moe_dims& d, const float* h32, const int32_t* route_row,
                                     const int32_t* row_e, const uint32_t* amax_h, float* gh_out, uint8_t* hq,
                                     uint8_t* hsf, cudaStream_t s);
cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t n, cudaStream_t s);
// NVFP4 emulation: weights of touched experts to bf16 (count nullable: all
// n_mat matrices; tiled: payloads in the layout of fp4moe_pack_weights); x and h through NVFP4 QDQ into bf16 rows
// pairs > 0: gate/up-paired tiled payloads and scales (P = I / 128 pairs per
// matrix); 0: the plain tiled (or, tiled = false, row-major) payloads
cudaError_t launch_nv_weight_bf16(const uint8_t* codes, bool tiled, int pairs, const uint8_t* sf, const float* g,
                                  int n_mat, int rows, int K, const int32_t* count, uint16_t* out, cudaStream_t s);
cudaError_t launch_nv_qdq_x_bf16(const fp4moe_dims& d, const uint16_t* x, const int32_t* route_row,
                                 const uint32_t* amax_x, float* g_out, uint16_t* xb, cudaStream_t s);
cudaError_t launch_nv_qdq_h_bf16(const fp4moe_dims& d, const float* h32, const int32_t* route_row,
                                 const int32_t* row_e, const uint32_t* amax_h, float* gh_out, uint16_t* hb,
                                 cudaStream_t s);
// W8A8: x per token to E4M3 into its route rows (+ sigma per row); h per route
// row to E4M3 with sigma from amax_row
cudaError_t launch_fp8_x_quant(const fp4moe_dims& d, const uint16_t* x, const int32_t* route_row, uint8_t* xq,
                               float* xsig, cudaStream_t s);
cudaError_t launch_fp8_h_quant(const fp4moe_dims& d, const float* h32, const int32_t* route_row,
                               const uint32_t* amax_row, uint8_t* hq, float* hsig, cudaStream_t s);
cudaError_t launch_quantize_rows(const void* x, int x_is_fp32, int64_t rows, int cols, bool nv,
                                 const float* global_in, const uint32_t* amax_bits, uint8_t* codes,
                                 uint8_t* scales, float* global_out, cudaStream_t s);
cudaError_t launch_pack_weights(const uint8_t* src, uint8_t* dst, int64_t rows_total, int kbytes, int pairs,
                                cudaStream_t s);
// NaN scale bytes (E8M0 255, E4M3 0x7F / 0xFF) of src[n] into the status word
cudaError_t launch_nan_scales(const uint8_t* src, int64_t n, bool nv, int32_t* status, cudaStream_t s);
cudaError_t launch_pack_scales(const uint8_t* src, uint8_t* dst, int64_t n_mat, int rows, int kblocks, bool nv,
                               int pairs, cudaStream_t s);
cudaError_t launch_convert(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K, uint8_t* out,
                           float* row_scale, uint8_t* row_status, int32_t* status, cudaStream_t s);

// ------------------------------------------------------------- grouped GEMMs
struct GemmArgs {
  const fp4moe_dims* d;
  bool nv;
  bool f8;                         // W8A8: E4M3 operands with per-row fp32 scales (below)
  bool bf;                         // NVFP4 emulation: BF16 operands (dequantised), no scales
  int n_tile;
  int num_sms;
  // weights
  const uint8_t *w, *wsf;          // routed experts
  bool w_tiled;                    // w and sh in the tiled layout of fp4moe_pack_weights
  int row_begin, row_count;        // down: weight rows (= output columns) [row_begin, +row_count);
                                   // row_count 0: all H rows
  const uint8_t *sh, *shsf;        // shared expert (nullable)
  const float *gw;                 // NVFP4 tensor scales [E + n_shared]
  // activations (B operand)
  const uint8_t *b, *bsf;
  int rows_cap;
  // plan
  const int32_t *expert_count, *expert_slot, *unit_start;
  const Plan* plan;
  const int32_t *row_tok;
  const float *row_w;
  const uint32_t *tok_mask;        // gate/up, few tokens: B = token rows, column t kept per mask bit
  bool plan_from_prev;             // the kernel launched just before wrote the plan
  const float *g_b;                // NVFP4: tensor scale of B (x: one; h: per expert)
  // outputs
  uint8_t *hq, *hsf;               // gate/up, MXFP4
  float *h32;                      // gate/up, NVFP4 (pre-quantisation h)
  uint32_t *amax_h;                // gate/up, NVFP4
  float *h_dbg;                    // optional copy of h
  float *out_acc;                  // down; gate/up: zeroed there when zero_acc
  bool zero_acc;                   // gate/up zeroes out_acc ([T, H] fp32) for the down GEMM
  int32_t *status;
  uint64_t wait_ns;                // pipeline wait limit; 0: kWaitLimitNs
  bool withhold;                   // gate/up test knob (fp4moe_debug.withhold_first_stage)
  int dn_pair;                     // down, 112-token tiles: 2 = one unit covers two slots (224 tokens)
  int gu_pairs;                    // gate/up: weights and scales in the gate/up-paired tiled order (I / 128), or 0
  bool dn_cta_pair;                // down, dn_pair 2: run on CTA pairs (units of 256 weight rows)
  bool dn_w2;                      // down, 112-token tiles, dn_pair 1: units of two weight tiles (256 rows)
  bool dn_paired;                  // down: w / sh and their scales in the row-tile-paired tiled order
  // W8A8: channel scales of the weights (routed [E, rows], shared [rows]),
  // scales of the B rows (per permuted row); amax_h is then per permuted row
  const float *wrs, *shrs, *brs;
};

cudaError_t launch_gateup(const GemmArgs& a, cudaStream_t s);
cudaError_t launch_down(const GemmArgs& a, cudaStream_t s);

int device_sm_count();

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialisation: it may begin while the previous kernel on s drains; the
// kernel waits (griddepcontrol.wait) before reading that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As launch_pdl, with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Encodes a uint8 tensor map: dims[0] innermost (bytes), strides[i] the byte
// stride of dimension i + 1, box in elements, optional 128-byte swizzle.
bool encode_tmap_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box, bool swizzle128);

}  // namespace fp4moe
