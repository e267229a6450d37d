// C-ABI entry points of libfp4moe: argument checks, workspace layout and the
// launch sequence of the forward.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

namespace {

constexpr int64_t kAlign = 256;
inline int64_t align_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(const fp4moe_dims& d) {
  if (d.T < 1 || d.T > 65536) return false;
  if (d.H < 256 || d.H % 256 != 0 || d.H > 65536) return false;
  if (d.I < 128 || d.I % 128 != 0 || d.I > 65536) return false;
  if (d.E < 1 || d.E > 512) return false;
  if (d.top_k < 1 || d.top_k > 16 || d.top_k > d.E) return false;
  if (d.n_group < 1 || d.n_group > 32 || d.E % d.n_group != 0) return false;
  if (d.topk_group < 1 || d.topk_group > d.n_group) return false;
  // grouped routing scores a group by its two largest corrected scores, so
  // a group holds at least two experts
  if (d.n_group > 1 && (d.E / d.n_group < 2 || d.E / d.n_group > 64 || d.topk_group * (d.E / d.n_group) < d.top_k))
    return false;
  if (d.n_shared < 0 || d.n_shared > 1) return false;
  if (d.fmt != FP4MOE_MXFP4 && d.fmt != FP4MOE_NVFP4 && d.fmt != FP4MOE_FP8) return false;
  if (!(d.routed_scaling == d.routed_scaling)) return false;
  return true;
}

// Down GEMM of the MXFP4 layers with 112-token tiles: one unit covers two
// slots (up to 224 tokens, N = 240 MMAs), twice the work per pipeline step,
// with one MMA issuer (two accumulator sets of 240 columns fill tensor
// memory).  A unit that stays within one slot then runs at half the issue
// rate of the unpaired kernel's two issuers, so pairing pays only when
// enough units fill both slots: at >= 80 routes per expert on average
// (measured with the register-transpose epilogue: skewed 16k-token layer
// down -6%, 4k-token prefill at 85 routes per expert -11%; with the earlier
// shared-memory epilogue prefill had been +6%).  NVFP4's larger scale
// groups leave no room for two such accumulator sets.
int fp4_down_pair(int n_tile, bool nv, double routes_per_expert) {
  return (n_tile == 112 && !nv && routes_per_expert >= 80.0) ? 2 : 1;
}

// Paired-slot down units over an output range of a multiple of 256 rows can
// run on CTA pairs (M = 256 MMAs issued by one CTA for two SMs, half the
// tcgen05 instructions per FLOP); their units then count 256-row tiles.  An
// opt-in (fp4moe_debug::down_cta_pair): measured on GB300, the pair's MMAs
// and scale copies each hold the issuing thread ~90 cycles against ~60 for
// one CTA's, so the pair's K tile (1444 cycles) is slower than two single
// CTAs' (1046): skewed 16k-token down 1.75 -> 2.16 ms.
bool fp4_down_cta_pair(int dn_pair, int out_rows, const fp4moe_debug* dbg) {
  return dbg && dbg->down_cta_pair && dn_pair == 2 && out_rows % 256 == 0;
}

// Where paired slots would be chosen and the output range is a multiple of
// 256 rows, a down unit instead covers two adjacent weight tiles of one
// 112-token tile: the gate/up GEMM's mainloop (two A operands, one issuer
// each, one shared B tile), with the same operand bytes per FLOP as the
// paired slots.  (The CTA-pair opt-in keeps the paired slots.)
bool fp4_down_w2(int dn_pair, int out_rows, const fp4moe_debug* dbg) {
  return dn_pair == 2 && out_rows % 256 == 0 && !(dbg && dbg->down_cta_pair);
}

int pick_n_tile(const fp4moe_dims& d) {
  const double avg = (double)d.T * d.top_k / d.E;
  // Every size keeps two accumulator sets in tensor memory (the epilogue of
  // one unit overlaps the next unit's MMAs): 2 x (gate + up) x 112 columns
  // plus one K tile's scale factors is the most that fits in 512.  Wider
  // tiles do more work per MMA, which wins once experts see 64 tokens on
  // average.
  if (avg <= 24.0) return 32;
  if (avg < 64.0) return 64;
  return 112;
}

// Router split-K factor: a divisor of H / 256 that gives the logits kernel
// enough CTAs (or warps) to cover the GPU.
int pick_splits(const fp4moe_dims& d) {
  const int kt = d.H / 256;
  int64_t units, want;
  if (d.T <= 16) {
    units = d.E;             // warps; each should issue all its weight loads in one batch
    want = 16 * 152;
  } else {  // tensor-core router: one CTA per (128 tokens, expert tile, split), at most 8 splits
    units = (int64_t)((d.T + 127) / 128) * ((d.E + 255) / 256);
    want = 152;
    int best = 1;
    for (int s = 1; s <= kt && s <= 8; ++s)
      if (kt % s == 0) {
        best = s;
        if (units * s >= want) return s;
      }
    return best;
  }
  for (int s = 1; s <= kt; ++s)
    if (kt % s == 0 && units * s >= want) return s;
  return kt;
}

}  // namespace

fp4moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4MOE_OK : FP4MOE_ERR_CUDA; }

fp4moe_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4MOE_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FP4MOE_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FP4MOE_ERR_DEVICE;
  return (major == 10 && minor == 3) ? FP4MOE_OK : FP4MOE_ERR_DEVICE;
}

bool make_layout(const fp4moe_dims& d, Layout* L) {
  if (!dims_ok(d)) return false;
  memset(L, 0, sizeof(*L));
  const bool nv = d.fmt == FP4MOE_NVFP4;
  const bool f8 = d.fmt == FP4MOE_FP8;  // W8A8: E4M3 rows with one fp32 scale each
  L->n_exp = d.E + d.n_shared;
  L->n_chunks = (d.T + kChunkTokens - 1) / kChunkTokens;
  L->n_route_per_tok = d.top_k + d.n_shared;
  const int64_t R = (int64_t)d.T * L->n_route_per_tok;
  fp4moe_ws_layout& w = L->ws;
  w.n_tile = pick_n_tile(d);
  w.n_splits = pick_splits(d);
  // the fused front end: K splits of at most 1024 router columns when that
  // takes no more than 8 (one cluster per expert group), else of at most
  // kFrontMaxKc; rows too long for 8 splits use the separate kernels
  L->front_splits = 0;
  for (int cap : {1024, kFrontMaxKc}) {
    for (int s = 1; s <= 8 && !L->front_splits; ++s)
      if ((d.H / 256) % s == 0 && d.H / s <= cap) L->front_splits = s;
    if (L->front_splits) break;
  }
  L->front = !nv && !f8 && d.T <= kFrontMaxT && L->front_splits > 0;
  w.x_by_token = L->front ? 1 : 0;
  // few tokens: one 16-token tile holds every token (the gate/up B operand)
  // and every expert's routes; half the B bytes and MMA columns of 32
  if (L->front) w.n_tile = 16;
  const int planes = w.n_splits;  // the front end keeps one plane of scores
  const int64_t slots_cap = R / w.n_tile + L->n_exp + 1;
  if (slots_cap * kSlotRows > INT32_MAX / 2) return false;
  w.rows_cap = (int32_t)(slots_cap * kSlotRows);
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  // status and the per-chunk counters are adjacent: one memset clears both
  w.status = take(kStatusInts * 4);
  L->chunk_counts = take((int64_t)L->n_chunks * L->n_exp * 4);
  w.logits = take((int64_t)planes * d.T * d.E * 4);
  w.topk_idx = take((int64_t)d.T * d.top_k * 4);
  w.topk_w = take((int64_t)d.T * d.top_k * 4);
  L->plan = take(sizeof(Plan));
  w.expert_count = take((int64_t)L->n_exp * 4);
  w.expert_slot = take((int64_t)L->n_exp * 4);
  L->gu_start = take((int64_t)(L->n_exp + 1) * 4);
  L->dn_start = take((int64_t)(L->n_exp + 1) * 4);
  w.route_row = take(R * 4);
  w.row_tok = take((int64_t)w.rows_cap * 4);
  w.row_w = take((int64_t)w.rows_cap * 4);
  L->row_e = take((int64_t)w.rows_cap * 4);
  w.xq = take((int64_t)w.rows_cap * (f8 ? d.H : d.H / 2));
  w.xsf = f8 ? take((int64_t)w.rows_cap * 4) : take((int64_t)slots_cap * katoms_padded(d.H, nv) * 512);
  w.hq = take((int64_t)w.rows_cap * (f8 ? d.I : d.I / 2));
  w.hsf = f8 ? take((int64_t)w.rows_cap * 4) : take((int64_t)slots_cap * katoms_padded(d.I, nv) * 512);
  w.h32 = (nv || f8) ? take((int64_t)w.rows_cap * d.I * 4) : take(0);
  w.gscale = take((int64_t)(2 + L->n_exp) * 4);
  // amax bits: NVFP4 x, spare, h per expert; W8A8 h per permuted row
  L->amax = take(f8 ? (int64_t)w.rows_cap * 4 : (int64_t)(2 + L->n_exp) * 4);
  w.out_acc = take((int64_t)d.T * d.H * 4);
  w.total_bytes = off;
  return true;
}

// NVFP4 emulation mode: the NVFP4 forward's workspace followed by bf16 rows of
// x and h and bf16 copies of the expert weights (touched experts written).
struct EmuLayout {
  Layout L;
  int64_t xb, hb, w13b, w2b, sh13b, sh2b, total;
};

bool emulation_layout(const fp4moe_dims& d, EmuLayout* M) {
  if (d.fmt != FP4MOE_NVFP4 || !make_layout(d, &M->L)) return false;
  int64_t off = (M->L.ws.total_bytes + 255) / 256 * 256;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off = (off + bytes + 255) / 256 * 256;
    return o;
  };
  const int64_t rc = M->L.ws.rows_cap;
  M->xb = take(rc * d.H * 2);
  M->hb = take(rc * d.I * 2);
  M->w13b = take((int64_t)d.E * 2 * d.I * d.H * 2);
  M->w2b = take((int64_t)d.E * d.H * d.I * 2);
  M->sh13b = take(d.n_shared ? (int64_t)2 * d.I * d.H * 2 : 0);
  M->sh2b = take(d.n_shared ? (int64_t)d.H * d.I * 2 : 0);
  M->total = off;
  return true;
}

// Dense linear as a one-expert MoE layer: the down GEMM's view (H = N output
// rows, I = K), top-1, one token per route.
fp4moe_dims linear_dims(int32_t fmt, int32_t T, int32_t K, int32_t N) {
  fp4moe_dims d;
  memset(&d, 0, sizeof(d));
  d.T = T;
  d.H = N;
  d.I = K;
  d.E = 1;
  d.top_k = 1;
  d.n_group = 1;
  d.topk_group = 1;
  d.n_shared = 0;
  d.routed_scaling = 1.0f;
  d.renormalize = 0;
  d.fmt = fmt;
  return d;
}

bool linear_layout(int32_t fmt, int32_t T, int32_t K, int32_t N, Layout* L) {
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return false;
  if (K < 256 || K % 256 != 0 || N < 256 || N % 256 != 0) return false;
  return make_layout(linear_dims(fmt, T, K, N), L);
}

}  // namespace fp4moe

using namespace fp4moe;

extern "C" {

int32_t fp4moe_version(void) { return 100; }

const char* fp4moe_status_string(int32_t s) {
  switch (s) {
    case FP4MOE_OK: return "ok";
    case FP4MOE_ERR_INVALID_ARG: return "invalid argument";
    case FP4MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FP4MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case FP4MOE_ERR_CUDA: return "CUDA error";
    case FP4MOE_ERR_TIMEOUT: return "device wait timed out";
    case FP4MOE_ERR_NAN_SCALE: return "NaN scale byte";
    case FP4MOE_ERR_INEXACT: return "conversion row below the exponent floor";
    case FP4MOE_ERR_DEVICE: return "no sm_103 device";
    default: return "unknown status";
  }
}

size_t fp4moe_workspace_size(const fp4moe_dims* dims) {
  if (!dims) return 0;
  Layout L;
  if (!make_layout(*dims, &L)) return 0;
  return (size_t)L.ws.total_bytes;
}

fp4moe_status fp4moe_workspace_layout(const fp4moe_dims* dims, fp4moe_ws_layout* out) {
  if (!dims || !out) return FP4MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(*dims, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  *out = L.ws;
  return FP4MOE_OK;
}

size_t fp4moe_packed_scales_bytes(int64_t n_mat, int32_t rows, int32_t kblocks, int32_t fmt) {
  if (n_mat < 0 || rows <= 0 || rows % 128 != 0 || kblocks <= 0 || kblocks % 4 != 0) return 0;
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return 0;
  const bool nv = fmt == FP4MOE_NVFP4;
  const int64_t katoms = katoms_padded((int64_t)kblocks * (nv ? 16 : 32), nv);
  return (size_t)(n_mat * (rows / 128) * katoms * 512);
}

fp4moe_status fp4moe_pack_scales(const uint8_t* src, uint8_t* dst, int64_t n_mat, int32_t rows, int32_t kblocks,
                                 int32_t fmt, void* stream) {
  if (!src || !dst) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_packed_scales_bytes(n_mat, rows, kblocks, fmt) == 0 && n_mat != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  return cuda_status(launch_pack_scales(src, dst, n_mat, rows, kblocks, fmt == FP4MOE_NVFP4, 0,
                                        static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_pack_gateup_scales(const uint8_t* src, uint8_t* dst, int64_t n_mat, int32_t I, int32_t kblocks,
                                        int32_t fmt, void* stream) {
  if (!src || !dst) return FP4MOE_ERR_INVALID_ARG;
  if (I <= 0 || I % 128 != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fp4moe_packed_scales_bytes(n_mat, 2 * I, kblocks, fmt) == 0 && n_mat != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  return cuda_status(launch_pack_scales(src, dst, n_mat, 2 * I, kblocks, fmt == FP4MOE_NVFP4, I / 128,
                                        static_cast<cudaStream_t>(stream)));
}

size_t fp4moe_packed_weights_bytes(int64_t n_mat, int32_t rows, int32_t kbytes) {
  if (n_mat < 0 || rows <= 0 || rows % 128 != 0 || kbytes <= 0 || kbytes % 16 != 0) return 0;
  return (size_t)(n_mat * rows * (int64_t)((kbytes + 127) / 128) * 128);
}

fp4moe_status fp4moe_pack_weights(const uint8_t* src, uint8_t* dst, int64_t n_mat, int32_t rows, int32_t kbytes,
                                  void* stream) {
  if (!src || !dst) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_packed_weights_bytes(n_mat, rows, kbytes) == 0 && n_mat != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fp4moe_status st = check_device()) return st;
  return cuda_status(launch_pack_weights(src, dst, n_mat * rows, kbytes, 0, static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_pack_gateup_weights(const uint8_t* src, uint8_t* dst, int64_t n_mat, int32_t I, int32_t kbytes,
                                         void* stream) {
  if (!src || !dst) return FP4MOE_ERR_INVALID_ARG;
  if (I <= 0 || I % 128 != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fp4moe_packed_weights_bytes(n_mat, 2 * I, kbytes) == 0 && n_mat != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fp4moe_status st = check_device()) return st;
  return cuda_status(launch_pack_weights(src, dst, n_mat * 2 * I, kbytes, I / 128, static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_route(const fp4moe_dims* dims, const uint16_t* x, const uint16_t* w_router, const float* bias,
                           int32_t* topk_idx, float* topk_w, float* logits_out, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!dims || !x || !w_router || !bias || !topk_idx || !topk_w || !ws) return FP4MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(*dims, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < (size_t)L.ws.total_bytes) return FP4MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(w_router)) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const fp4moe_dims& d = *dims;
  float* partial = reinterpret_cast<float*>(base + L.ws.logits);
  int32_t* cc = reinterpret_cast<int32_t*>(base + L.chunk_counts);
  cudaError_t e = cudaMemsetAsync(cc, 0, (size_t)L.n_chunks * L.n_exp * 4, s);
  if (e == cudaSuccess)
    e = launch_router_logits(x, w_router, partial, d.T, d.H, d.E, L.ws.n_splits,
                             reinterpret_cast<int32_t*>(base + L.ws.status), s);
  if (e == cudaSuccess)
    e = launch_topk(d, partial, L.ws.n_splits, bias, topk_idx, topk_w, logits_out, nullptr, cc, L.n_exp, s);
  return cuda_status(e);
}

fp4moe_status fp4moe_quantize_act(const void* x, int32_t x_is_fp32, int64_t rows, int32_t cols, int32_t fmt,
                                  const float* global_in, uint8_t* codes, uint8_t* scales, float* global_out,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (!x || !codes || !scales || !ws) return FP4MOE_ERR_INVALID_ARG;
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return FP4MOE_ERR_INVALID_ARG;
  if (ws_bytes < 256) return FP4MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(codes)) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* amax = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + 64);
  const bool nv = fmt == FP4MOE_NVFP4;
  cudaError_t e = cudaSuccess;
  if (nv && !global_in) e = launch_amax(x, x_is_fp32 ? 1 : 0, rows * (int64_t)cols, amax, s);
  if (e == cudaSuccess)
    e = launch_quantize_rows(x, x_is_fp32 ? 1 : 0, rows, cols, nv, global_in, amax, codes, scales, global_out, s);
  return cuda_status(e);
}

// The layer over output columns [h_begin, h_end): everything up to the
// intermediate is computed in full; the down GEMM reads the weight rows of
// those columns only and the other columns of out come out zero.
static fp4moe_status forward_cols(const fp4moe_dims* dims, const fp4moe_weights* w, const uint16_t* x,
                                  uint16_t* out, int32_t h_begin, int32_t h_end, const fp4moe_debug* dbg, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!dims || !w || !x || !out || !ws) return FP4MOE_ERR_INVALID_ARG;
  const fp4moe_dims& d = *dims;
  Layout L;
  if (!make_layout(d, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (h_begin < 0 || h_end > d.H || h_begin >= h_end || h_begin % 128 != 0 || h_end % 128 != 0)
    return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.fmt == FP4MOE_FP8) return FP4MOE_ERR_INVALID_ARG;  // fp4moe_forward_w8a8
  if (ws_bytes < (size_t)L.ws.total_bytes) return FP4MOE_ERR_WORKSPACE;
  const bool nv = d.fmt == FP4MOE_NVFP4;
  int dn_pair = fp4_down_pair(L.ws.n_tile, nv, (double)d.T * d.top_k / d.E);
  const bool dn_w2 = fp4_down_w2(dn_pair, h_end - h_begin, dbg);
  if (dn_w2) dn_pair = 1;
  const bool dn_cta = fp4_down_cta_pair(dn_pair, h_end - h_begin, dbg);
  const int dn_mtiles = (h_end - h_begin) / ((dn_cta || dn_w2) ? 256 : 128);  // weight-row tiles per down unit row
  if (!w->w13 || !w->w13_scale || !w->w2 || !w->w2_scale || !w->w_router || !w->bias) return FP4MOE_ERR_INVALID_ARG;
  if (nv && (!w->g13 || !w->g2)) return FP4MOE_ERR_INVALID_ARG;
  if (w->packed < 0 || w->packed > 3) return FP4MOE_ERR_INVALID_ARG;
  // row-tile-paired down weights: whole 256-row slabs of the output
  if (w->packed == 3 && (d.H % 256 != 0 || h_begin % 256 != 0 || h_end % 256 != 0))
    return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.n_shared && (!w->sh13 || !w->sh13_scale || !w->sh2 || !w->sh2_scale)) return FP4MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w->w13) || !aligned16(w->w2) || !aligned16(w->w13_scale) ||
      !aligned16(w->w2_scale) || !aligned16(w->w_router) || !aligned16(ws) || !aligned16(out))
    return FP4MOE_ERR_INVALID_ARG;
  if (d.n_shared && (!aligned16(w->sh13) || !aligned16(w->sh2) || !aligned16(w->sh13_scale) ||
                     !aligned16(w->sh2_scale)))
    return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return FP4MOE_ERR_DEVICE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto P = [&](int64_t off) { return base + off; };
  int32_t* status = reinterpret_cast<int32_t*>(P(L.ws.status));
  float* partial = reinterpret_cast<float*>(P(L.ws.logits));
  int32_t* idx = reinterpret_cast<int32_t*>(P(L.ws.topk_idx));
  float* tw = reinterpret_cast<float*>(P(L.ws.topk_w));
  int32_t* cc = reinterpret_cast<int32_t*>(P(L.chunk_counts));
  Plan* plan = reinterpret_cast<Plan*>(P(L.plan));
  int32_t* ecount = reinterpret_cast<int32_t*>(P(L.ws.expert_count));
  int32_t* eslot = reinterpret_cast<int32_t*>(P(L.ws.expert_slot));
  int32_t* gu_start = reinterpret_cast<int32_t*>(P(L.gu_start));
  int32_t* dn_start = reinterpret_cast<int32_t*>(P(L.dn_start));
  int32_t* route_row = reinterpret_cast<int32_t*>(P(L.ws.route_row));
  int32_t* row_tok = reinterpret_cast<int32_t*>(P(L.ws.row_tok));
  float* row_w = reinterpret_cast<float*>(P(L.ws.row_w));
  int32_t* row_e = reinterpret_cast<int32_t*>(P(L.row_e));
  uint8_t* xq = P(L.ws.xq);
  uint8_t* xsf = P(L.ws.xsf);
  uint8_t* hq = P(L.ws.hq);
  uint8_t* hsf = P(L.ws.hsf);
  float* h32 = nv ? reinterpret_cast<float*>(P(L.ws.h32)) : nullptr;
  float* gscale = reinterpret_cast<float*>(P(L.ws.gscale));
  uint32_t* amax = reinterpret_cast<uint32_t*>(P(L.amax));
  float* acc = reinterpret_cast<float*>(P(L.ws.out_acc));
  const int n_tile = L.ws.n_tile;

  auto rec = [&](int i) -> cudaError_t {
    if (dbg && dbg->events[i]) return cudaEventRecord(static_cast<cudaEvent_t>(dbg->events[i]), s);
    return cudaSuccess;
  };

  cudaError_t e = rec(0);
  // status word (with the last-CTA tickets) and the per-chunk expert counters
  const size_t clear_bytes = (size_t)(L.chunk_counts - L.ws.status) + (size_t)L.n_chunks * L.n_exp * 4;
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, clear_bytes, s);
  if (L.front) {
    // few tokens: router, top-k, plan, scatter and x quantisation in one launch
    FrontArgs f;
    memset(&f, 0, sizeof(f));
    f.d = d;
    f.x = x;
    f.wr = w->w_router;
    f.bias = w->bias;
    f.partial = partial;
    f.n_splits = L.front_splits;
    f.n_tile = n_tile;
    f.n_exp = L.n_exp;
    f.dn_mtiles = dn_mtiles;
    f.out_acc = acc;
    f.idx = idx;
    f.w = tw;
    f.expert_count = ecount;
    f.expert_slot = eslot;
    f.gu_start = gu_start;
    f.dn_start = dn_start;
    f.plan = plan;
    f.route_row = route_row;
    f.row_tok = row_tok;
    f.row_e = row_e;
    f.row_w = row_w;
    f.ticket = status + ST_TICKET_FRONT;
    f.xq = xq;
    f.xsf = xsf;
    f.tok_mask = reinterpret_cast<uint32_t*>(cc);  // the per-chunk counters are not used here
    f.logits_dbg = dbg ? dbg->logits : nullptr;
    f.scores_dbg = dbg ? dbg->scores : nullptr;
    if (d.n_shared) {  // the shared expert's weights: w13 whole, the rows of w2 this call's columns need
      const int64_t w2_row = w->packed ? (int64_t)fp4moe_packed_weights_bytes(1, d.H, d.I / 2) / d.H : d.I / 2;
      const int64_t w2_sf_tile = (int64_t)fp4moe_packed_scales_bytes(1, 128, d.I / 32, d.fmt);
      const uint8_t* r[4] = {w->sh13, w->sh13_scale, w->sh2 + h_begin * w2_row,
                             w->sh2_scale + (h_begin / 128) * w2_sf_tile};
      const int64_t n[4] = {
          w->packed ? (int64_t)fp4moe_packed_weights_bytes(1, 2 * d.I, d.H / 2) : (int64_t)d.I * d.H,
          (int64_t)fp4moe_packed_scales_bytes(1, 2 * d.I, d.H / 32, d.fmt), (h_end - h_begin) * w2_row,
          (int64_t)((h_end - h_begin) / 128) * w2_sf_tile};
      for (int i = 0; i < 4; ++i) {
        f.l2_pf[i] = r[i];
        f.l2_pf_bytes[i] = n[i];
      }
    }
    if (e == cudaSuccess) e = launch_decode_front(f, s);
    for (int i = 1; i <= 4 && e == cudaSuccess; ++i) e = rec(i);
  } else {
    if (e == cudaSuccess && nv) e = cudaMemsetAsync(amax, 0, (size_t)(2 + L.n_exp) * 4, s);
    if (e == cudaSuccess) e = launch_router_logits(x, w->w_router, partial, d.T, d.H, d.E, L.ws.n_splits, status, s);
    if (e == cudaSuccess) e = rec(1);
    if (e == cudaSuccess) e = launch_topk(d, partial, L.ws.n_splits, w->bias, idx, tw, dbg ? dbg->logits : nullptr,
                                            dbg ? dbg->scores : nullptr, cc, L.n_exp, s);
    if (e == cudaSuccess) e = rec(2);
    if (e == cudaSuccess)
      e = launch_plan(d, cc, L.n_chunks, L.n_exp, n_tile, dn_pair, dn_mtiles, ecount, eslot, gu_start, dn_start, plan,
                      status + ST_TICKET_PLAN, s);
    if (e == cudaSuccess)
      e = launch_scatter(d, idx, tw, cc, L.n_chunks, L.n_exp, n_tile, eslot, route_row, row_tok, row_w, row_e, s);
    if (e == cudaSuccess) e = rec(3);
    if (e == cudaSuccess && nv) e = launch_amax(x, 0, (int64_t)d.T * d.H, amax, s);
    if (e == cudaSuccess) e = launch_gather_quant(d, x, route_row, xq, xsf, amax, gscale, s);
    if (e == cudaSuccess) e = rec(4);
  }

  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.d = &d;
  a.nv = nv;
  a.n_tile = n_tile;
  a.num_sms = num_sms;
  a.rows_cap = L.ws.rows_cap;
  a.expert_count = ecount;
  a.expert_slot = eslot;
  a.plan = plan;
  a.row_tok = row_tok;
  a.row_w = row_w;
  a.status = status;
  a.wait_ns = (dbg && dbg->wait_limit_ns > 0) ? (uint64_t)dbg->wait_limit_ns : 0;
  if (e == cudaSuccess) {
    GemmArgs g = a;
    g.w = w->w13;
    g.w_tiled = w->packed != 0;
    g.gu_pairs = w->packed >= 2 ? d.I / 128 : 0;
    g.wsf = w->w13_scale;
    g.sh = d.n_shared ? w->sh13 : nullptr;
    g.shsf = d.n_shared ? w->sh13_scale : nullptr;
    g.gw = w->g13;
    g.b = xq;
    g.bsf = xsf;
    g.unit_start = gu_start;
    g.g_b = gscale;  // g_x
    g.hq = hq;
    g.hsf = hsf;
    g.h32 = h32;
    g.amax_h = amax + 2;
    g.h_dbg = dbg ? dbg->h_pre : nullptr;
    g.tok_mask = L.front ? reinterpret_cast<const uint32_t*>(cc) : nullptr;
    g.plan_from_prev = L.front;  // the front end, launched just before, wrote the plan
    g.out_acc = acc;
    g.zero_acc = !L.front;  // the front end zeroes it itself
    g.withhold = dbg && dbg->withhold_first_stage;
    e = launch_gateup(g, s);
  }
  if (e == cudaSuccess && nv) e = launch_h_quant_nv_routes(d, h32, route_row, row_e, amax + 2, gscale + 2, hq, hsf, s);
  if (e == cudaSuccess) e = rec(5);
  if (e == cudaSuccess) {
    GemmArgs g = a;
    g.w = w->w2;
    g.w_tiled = w->packed != 0;
    g.row_begin = h_begin;
    g.row_count = h_end - h_begin;
    g.wsf = w->w2_scale;
    g.sh = d.n_shared ? w->sh2 : nullptr;
    g.shsf = d.n_shared ? w->sh2_scale : nullptr;
    g.gw = w->g2;
    g.b = hq;
    g.bsf = hsf;
    g.unit_start = dn_start;
    g.g_b = gscale + 2;  // g_h per expert
    g.out_acc = acc;
    g.dn_pair = dn_pair;
    g.dn_cta_pair = dn_cta;
    g.dn_w2 = dn_w2;
    g.dn_paired = w->packed == 3;
    e = launch_down(g, s);
  }
  if (e == cudaSuccess) e = rec(6);
  if (e == cudaSuccess) e = launch_finalize(acc, out, (int64_t)d.T * d.H, s);
  if (e == cudaSuccess) e = rec(7);
  return cuda_status(e);
}

fp4moe_status fp4moe_forward(const fp4moe_dims* dims, const fp4moe_weights* w, const uint16_t* x, uint16_t* out,
                             const fp4moe_debug* dbg, void* ws, size_t ws_bytes, void* stream) {
  if (!dims) return FP4MOE_ERR_INVALID_ARG;
  return forward_cols(dims, w, x, out, 0, dims->H, dbg, ws, ws_bytes, stream);
}

fp4moe_status fp4moe_forward_cols(const fp4moe_dims* dims, const fp4moe_weights* w, const uint16_t* x,
                                  uint16_t* out, int32_t h_begin, int32_t h_end, const fp4moe_debug* dbg, void* ws,
                                  size_t ws_bytes, void* stream) {
  return forward_cols(dims, w, x, out, h_begin, h_end, dbg, ws, ws_bytes, stream);
}

fp4moe_status fp4moe_forward_w8a8(const fp4moe_dims* dims, const fp4moe_fp8_weights* w, const uint16_t* x,
                                  uint16_t* out, const fp4moe_debug* dbg, void* ws, size_t ws_bytes, void* stream) {
  if (!dims || !w || !x || !out || !ws) return FP4MOE_ERR_INVALID_ARG;
  const fp4moe_dims& d = *dims;
  if (d.fmt != FP4MOE_FP8) return FP4MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(d, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < (size_t)L.ws.total_bytes) return FP4MOE_ERR_WORKSPACE;
  if (!w->w13 || !w->w13_scale || !w->w2 || !w->w2_scale || !w->w_router || !w->bias) return FP4MOE_ERR_INVALID_ARG;
  if (d.n_shared && (!w->sh13 || !w->sh13_scale || !w->sh2 || !w->sh2_scale)) return FP4MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w->w13) || !aligned16(w->w2) || !aligned16(w->w_router) || !aligned16(ws) ||
      !aligned16(out))
    return FP4MOE_ERR_INVALID_ARG;
  if (d.n_shared && (!aligned16(w->sh13) || !aligned16(w->sh2))) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return FP4MOE_ERR_DEVICE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto P = [&](int64_t off) { return base + off; };
  int32_t* status = reinterpret_cast<int32_t*>(P(L.ws.status));
  float* partial = reinterpret_cast<float*>(P(L.ws.logits));
  int32_t* idx = reinterpret_cast<int32_t*>(P(L.ws.topk_idx));
  float* tw = reinterpret_cast<float*>(P(L.ws.topk_w));
  Plan* plan = reinterpret_cast<Plan*>(P(L.plan));
  int32_t* ecount = reinterpret_cast<int32_t*>(P(L.ws.expert_count));
  int32_t* eslot = reinterpret_cast<int32_t*>(P(L.ws.expert_slot));
  int32_t* gu_start = reinterpret_cast<int32_t*>(P(L.gu_start));
  int32_t* dn_start = reinterpret_cast<int32_t*>(P(L.dn_start));
  int32_t* cc = reinterpret_cast<int32_t*>(P(L.chunk_counts));
  int32_t* route_row = reinterpret_cast<int32_t*>(P(L.ws.route_row));
  int32_t* row_tok = reinterpret_cast<int32_t*>(P(L.ws.row_tok));
  float* row_w = reinterpret_cast<float*>(P(L.ws.row_w));
  int32_t* row_e = reinterpret_cast<int32_t*>(P(L.row_e));
  uint8_t* xq = P(L.ws.xq);
  float* xsig = reinterpret_cast<float*>(P(L.ws.xsf));
  uint8_t* hq = P(L.ws.hq);
  float* hsig = reinterpret_cast<float*>(P(L.ws.hsf));
  float* h32 = reinterpret_cast<float*>(P(L.ws.h32));
  uint32_t* amax_row = reinterpret_cast<uint32_t*>(P(L.amax));
  float* acc = reinterpret_cast<float*>(P(L.ws.out_acc));
  const int n_tile = L.ws.n_tile;
  auto rec = [&](int i) -> cudaError_t {
    if (dbg && dbg->events[i]) return cudaEventRecord(static_cast<cudaEvent_t>(dbg->events[i]), s);
    return cudaSuccess;
  };

  cudaError_t e = rec(0);
  const size_t clear_bytes = (size_t)(L.chunk_counts - L.ws.status) + (size_t)L.n_chunks * L.n_exp * 4;
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, clear_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(amax_row, 0, (size_t)L.ws.rows_cap * 4, s);
  if (e == cudaSuccess) e = launch_router_logits(x, w->w_router, partial, d.T, d.H, d.E, L.ws.n_splits, status, s);
  if (e == cudaSuccess) e = rec(1);
  if (e == cudaSuccess) e = launch_topk(d, partial, L.ws.n_splits, w->bias, idx, tw, dbg ? dbg->logits : nullptr,
                                            dbg ? dbg->scores : nullptr, cc, L.n_exp, s);
  if (e == cudaSuccess) e = rec(2);
  if (e == cudaSuccess)
    e = launch_plan(d, cc, L.n_chunks, L.n_exp, n_tile, 1, d.H / 128, ecount, eslot, gu_start, dn_start, plan,
                    status + ST_TICKET_PLAN, s);
  if (e == cudaSuccess)
    e = launch_scatter(d, idx, tw, cc, L.n_chunks, L.n_exp, n_tile, eslot, route_row, row_tok, row_w, row_e, s);
  if (e == cudaSuccess) e = rec(3);
  if (e == cudaSuccess) e = launch_fp8_x_quant(d, x, route_row, xq, xsig, s);
  if (e == cudaSuccess) e = rec(4);

  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.d = &d;
  a.f8 = true;
  a.n_tile = n_tile;
  a.num_sms = num_sms;
  a.rows_cap = L.ws.rows_cap;
  a.expert_count = ecount;
  a.expert_slot = eslot;
  a.plan = plan;
  a.row_tok = row_tok;
  a.row_w = row_w;
  a.status = status;
  a.wait_ns = (dbg && dbg->wait_limit_ns > 0) ? (uint64_t)dbg->wait_limit_ns : 0;
  if (e == cudaSuccess) {
    GemmArgs g = a;
    g.w = w->w13;
    g.wrs = w->w13_scale;
    g.sh = d.n_shared ? w->sh13 : nullptr;
    g.shrs = d.n_shared ? w->sh13_scale : nullptr;
    g.b = xq;
    g.brs = xsig;
    g.unit_start = gu_start;
    g.h32 = h32;
    g.amax_h = amax_row;
    g.h_dbg = dbg ? dbg->h_pre : nullptr;
    g.out_acc = acc;
    g.zero_acc = true;
    e = launch_gateup(g, s);
  }
  if (e == cudaSuccess) e = rec(5);
  if (e == cudaSuccess) e = launch_fp8_h_quant(d, h32, route_row, amax_row, hq, hsig, s);
  if (e == cudaSuccess) {
    GemmArgs g = a;
    g.w = w->w2;
    g.wrs = w->w2_scale;
    g.sh = d.n_shared ? w->sh2 : nullptr;
    g.shrs = d.n_shared ? w->sh2_scale : nullptr;
    g.b = hq;
    g.brs = hsig;
    g.unit_start = dn_start;
    g.out_acc = acc;
    e = launch_down(g, s);
  }
  if (e == cudaSuccess) e = rec(6);
  if (e == cudaSuccess) e = launch_finalize(acc, out, (int64_t)d.T * d.H, s);
  if (e == cudaSuccess) e = rec(7);
  return cuda_status(e);
}

size_t fp4moe_emulation_workspace_size(const fp4moe_dims* dims) {
  EmuLayout M;
  if (!dims || !emulation_layout(*dims, &M)) return 0;
  return (size_t)M.total;
}

fp4moe_status fp4moe_forward_nvfp4_emulated(const fp4moe_dims* dims, const fp4moe_weights* w, const uint16_t* x,
                                            uint16_t* out, const fp4moe_debug* dbg, void* ws, size_t ws_bytes,
                                            void* stream) {
  if (!dims || !w || !x || !out || !ws) return FP4MOE_ERR_INVALID_ARG;
  const fp4moe_dims& d = *dims;
  if (d.fmt != FP4MOE_NVFP4) return FP4MOE_ERR_INVALID_ARG;
  EmuLayout M;
  if (!emulation_layout(d, &M)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  const Layout& L = M.L;
  if (ws_bytes < (size_t)M.total) return FP4MOE_ERR_WORKSPACE;
  if (!w->w13 || !w->w13_scale || !w->w2 || !w->w2_scale || !w->g13 || !w->g2 || !w->w_router || !w->bias)
    return FP4MOE_ERR_INVALID_ARG;
  if (d.n_shared && (!w->sh13 || !w->sh13_scale || !w->sh2 || !w->sh2_scale)) return FP4MOE_ERR_INVALID_ARG;
  if (w->packed < 0 || w->packed > 3) return FP4MOE_ERR_INVALID_ARG;
  if (w->packed == 3 && d.H % 256 != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w->w13) || !aligned16(w->w2) || !aligned16(w->w_router) || !aligned16(ws) ||
      !aligned16(out))
    return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return FP4MOE_ERR_DEVICE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto P = [&](int64_t off) { return base + off; };
  int32_t* status = reinterpret_cast<int32_t*>(P(L.ws.status));
  float* partial = reinterpret_cast<float*>(P(L.ws.logits));
  int32_t* idx = reinterpret_cast<int32_t*>(P(L.ws.topk_idx));
  float* tw = reinterpret_cast<float*>(P(L.ws.topk_w));
  Plan* plan = reinterpret_cast<Plan*>(P(L.plan));
  int32_t* ecount = reinterpret_cast<int32_t*>(P(L.ws.expert_count));
  int32_t* eslot = reinterpret_cast<int32_t*>(P(L.ws.expert_slot));
  int32_t* gu_start = reinterpret_cast<int32_t*>(P(L.gu_start));
  int32_t* dn_start = reinterpret_cast<int32_t*>(P(L.dn_start));
  int32_t* cc = reinterpret_cast<int32_t*>(P(L.chunk_counts));
  int32_t* route_row = reinterpret_cast<int32_t*>(P(L.ws.route_row));
  int32_t* row_tok = reinterpret_cast<int32_t*>(P(L.ws.row_tok));
  float* row_w = reinterpret_cast<float*>(P(L.ws.row_w));
  int32_t* row_e = reinterpret_cast<int32_t*>(P(L.row_e));
  float* h32 = reinterpret_cast<float*>(P(L.ws.h32));
  float* gscale = reinterpret_cast<float*>(P(L.ws.gscale));
  uint32_t* amax = reinterpret_cast<uint32_t*>(P(L.amax));
  float* acc = reinterpret_cast<float*>(P(L.ws.out_acc));
  uint16_t* xb = reinterpret_cast<uint16_t*>(P(M.xb));
  uint16_t* hb = reinterpret_cast<uint16_t*>(P(M.hb));
  uint16_t* w13b = reinterpret_cast<uint16_t*>(P(M.w13b));
  uint16_t* w2b = reinterpret_cast<uint16_t*>(P(M.w2b));
  uint16_t* sh13b = d.n_shared ? reinterpret_cast<uint16_t*>(P(M.sh13b)) : nullptr;
  uint16_t* sh2b = d.n_shared ? reinterpret_cast<uint16_t*>(P(M.sh2b)) : nullptr;
  const int n_tile = L.ws.n_tile;
  auto rec = [&](int i) -> cudaError_t {
    if (dbg && dbg->events[i]) return cudaEventRecord(static_cast<cudaEvent_t>(dbg->events[i]), s);
    return cudaSuccess;
  };

  cudaError_t e = rec(0);
  const size_t clear_bytes = (size_t)(L.chunk_counts - L.ws.status) + (size_t)L.n_chunks * L.n_exp * 4;
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, clear_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(amax, 0, (size_t)(2 + L.n_exp) * 4, s);
  if (e == cudaSuccess) e = launch_router_logits(x, w->w_router, partial, d.T, d.H, d.E, L.ws.n_splits, status, s);
  if (e == cudaSuccess) e = rec(1);
  if (e == cudaSuccess) e = launch_topk(d, partial, L.ws.n_splits, w->bias, idx, tw, dbg ? dbg->logits : nullptr,
                                            dbg ? dbg->scores : nullptr, cc, L.n_exp, s);
  if (e == cudaSuccess) e = rec(2);
  if (e == cudaSuccess)
    e = launch_plan(d, cc, L.n_chunks, L.n_exp, n_tile, 1, d.H / 128, ecount, eslot, gu_start, dn_start, plan,
                    status + ST_TICKET_PLAN, s);
  if (e == cudaSuccess)
    e = launch_scatter(d, idx, tw, cc, L.n_chunks, L.n_exp, n_tile, eslot, route_row, row_tok, row_w, row_e, s);
  if (e == cudaSuccess) e = rec(3);
  // BF16 copies of the dispatched experts' weights (at GEMM time, as the
  // emulation pipeline does) and of the QDQ'd activations
  // (paired orders: gate/up pairs of I / 128 tiles; row-tile pairs of the
  // down matrices, one tile pair per 256-row slab)
  const int gu_p = w->packed >= 2 ? d.I / 128 : 0, dn_p = w->packed == 3 ? 1 : 0;
  if (e == cudaSuccess) e = launch_nv_weight_bf16(w->w13, w->packed != 0, gu_p, w->w13_scale, w->g13, d.E, 2 * d.I, d.H, ecount, w13b, s);
  if (e == cudaSuccess) e = launch_nv_weight_bf16(w->w2, w->packed != 0, dn_p, w->w2_scale, w->g2, d.E, d.H, d.I, ecount, w2b, s);
  if (e == cudaSuccess && d.n_shared)
    e = launch_nv_weight_bf16(w->sh13, w->packed != 0, gu_p, w->sh13_scale, w->g13 + d.E, 1, 2 * d.I, d.H, nullptr, sh13b, s);
  if (e == cudaSuccess && d.n_shared)
    e = launch_nv_weight_bf16(w->sh2, w->packed != 0, dn_p, w->sh2_scale, w->g2 + d.E, 1, d.H, d.I, nullptr, sh2b, s);
  if (e == cudaSuccess) e = launch_amax(x, 0, (int64_t)d.T * d.H, amax, s);
  if (e == cudaSuccess) e = launch_nv_qdq_x_bf16(d, x, route_row, amax, gscale, xb, s);
  if (e == cudaSuccess) e = rec(4);

  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.d = &d;
  a.bf = true;
  a.n_tile = n_tile;
  a.num_sms = num_sms;
  a.rows_cap = L.ws.rows_cap;
  a.expert_count = ecount;
  a.expert_slot = eslot;
  a.plan = plan;
  a.row_tok = row_tok;
  a.row_w = row_w;
  a.status = status;
  a.wait_ns = (dbg && dbg->wait_limit_ns > 0) ? (uint64_t)dbg->wait_limit_ns : 0;
  if (e == cudaSuccess) {
    GemmArgs g = a;
    g.w = reinterpret_cast<const uint8_t*>(w13b);
    g.sh = reinterpret_cast<const uint8_t*>(sh13b);
    g.b = reinterpret_cast<const uint8_t*>(xb);
    g.unit_start = gu_start;
    g.h32 = h32;
    g.amax_h = amax + 2;
    g.h_dbg = dbg ? dbg->h_pre : nullptr;
    g.out_acc = acc;
    g.zero_acc = true;
    e = launch_gateup(g, s);
  }
  if (e == cudaSuccess) e = rec(5);
  if (e == cudaSuccess) e = launch_nv_qdq_h_bf16(d, h32, route_row, row_e, amax + 2, gscale + 2, hb, s);
  if (e == cudaSuccess) {
    GemmArgs g = a;
    g.w = reinterpret_cast<const uint8_t*>(w2b);
    g.sh = reinterpret_cast<const uint8_t*>(sh2b);
    g.b = reinterpret_cast<const uint8_t*>(hb);
    g.unit_start = dn_start;
    g.out_acc = acc;
    e = launch_down(g, s);
  }
  if (e == cudaSuccess) e = rec(6);
  if (e == cudaSuccess) e = launch_finalize(acc, out, (int64_t)d.T * d.H, s);
  if (e == cudaSuccess) e = rec(7);
  return cuda_status(e);
}

size_t fp4moe_linear_workspace_size(int32_t fmt, int32_t T, int32_t K, int32_t N) {
  Layout L;
  if (!linear_layout(fmt, T, K, N, &L)) return 0;
  return (size_t)L.ws.total_bytes;
}

fp4moe_status fp4moe_linear(int32_t fmt, int32_t T, int32_t K, int32_t N, const uint16_t* x, const uint8_t* w,
                            const uint8_t* w_scale, const float* g_w, uint16_t* out, void* ws, size_t ws_bytes,
                            void* stream) {
  if (!x || !w || !w_scale || !out || !ws) return FP4MOE_ERR_INVALID_ARG;
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return FP4MOE_ERR_INVALID_ARG;
  if (fmt == FP4MOE_NVFP4 && !g_w) return FP4MOE_ERR_INVALID_ARG;
  Layout L;
  if (!linear_layout(fmt, T, K, N, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < (size_t)L.ws.total_bytes) return FP4MOE_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(w_scale) || !aligned16(out) || !aligned16(ws))
    return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  const int num_sms = device_sm_count();
  if (num_sms <= 0) return FP4MOE_ERR_DEVICE;
  const bool nv = fmt == FP4MOE_NVFP4;
  const fp4moe_dims dg = linear_dims(fmt, T, K, N);  // GEMM view: H = N output rows, I = K
  fp4moe_dims dq = dg;                               // quantiser view: rows of K values, one route each
  dq.H = K;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto P = [&](int64_t off) { return base + off; };
  int32_t* status = reinterpret_cast<int32_t*>(P(L.ws.status));
  Plan* plan = reinterpret_cast<Plan*>(P(L.plan));
  int32_t* ecount = reinterpret_cast<int32_t*>(P(L.ws.expert_count));
  int32_t* eslot = reinterpret_cast<int32_t*>(P(L.ws.expert_slot));
  int32_t* dn_start = reinterpret_cast<int32_t*>(P(L.dn_start));
  int32_t* route_row = reinterpret_cast<int32_t*>(P(L.ws.route_row));
  int32_t* row_tok = reinterpret_cast<int32_t*>(P(L.ws.row_tok));
  float* row_w = reinterpret_cast<float*>(P(L.ws.row_w));
  uint8_t* xq = P(L.ws.hq);    // the B operand of the down GEMM: rows of K/2 bytes
  uint8_t* xsf = P(L.ws.hsf);
  float* gscale = reinterpret_cast<float*>(P(L.ws.gscale));
  uint32_t* amax = reinterpret_cast<uint32_t*>(P(L.amax));
  float* acc = reinterpret_cast<float*>(P(L.ws.out_acc));
  const int n_tile = L.ws.n_tile;
  int dn_pair = fp4_down_pair(n_tile, nv, T);
  const bool dn_w2 = fp4_down_w2(dn_pair, N, nullptr);
  if (dn_w2) dn_pair = 1;
  const bool dn_cta = fp4_down_cta_pair(dn_pair, N, nullptr);

  cudaError_t e = cudaMemsetAsync(status, 0, kStatusInts * 4, s);
  if (e == cudaSuccess && nv) e = cudaMemsetAsync(amax, 0, 8, s);
  if (e == cudaSuccess)
    e = launch_linear_plan(T, n_tile, dn_pair, N / ((dn_cta || dn_w2) ? 256 : 128), ecount, eslot, dn_start, plan, route_row,
                           row_tok, row_w, acc, (int64_t)T * N, s);
  if (e == cudaSuccess && nv) e = launch_amax(x, 0, (int64_t)T * K, amax, s);
  if (e == cudaSuccess) e = launch_gather_quant(dq, x, route_row, xq, xsf, amax, gscale, s);
  if (e == cudaSuccess) {
    GemmArgs g;
    memset(&g, 0, sizeof(g));
    g.d = &dg;
    g.nv = nv;
    g.n_tile = n_tile;
    g.num_sms = num_sms;
    g.w = w;
    g.wsf = w_scale;
    g.gw = g_w;
    g.b = xq;
    g.bsf = xsf;
    g.rows_cap = L.ws.rows_cap;
    g.expert_count = ecount;
    g.expert_slot = eslot;
    g.unit_start = dn_start;
    g.plan = plan;
    g.row_tok = row_tok;
    g.row_w = row_w;
    g.g_b = gscale;  // NVFP4: g_x
    g.out_acc = acc;
    g.status = status;
    g.dn_pair = dn_pair;
    g.dn_cta_pair = dn_cta;
    g.dn_w2 = dn_w2;
    e = launch_down(g, s);
  }
  if (e == cudaSuccess) e = launch_finalize(acc, out, (int64_t)T * N, s);
  return cuda_status(e);
}

fp4moe_status fp4moe_mxfp4_to_fp8_rowscale(const uint8_t* codes, const uint8_t* scales_e8m0, int64_t rows, int32_t K,
                                           uint8_t* fp8_out, float* row_scale, uint8_t* row_status, void* ws,
                                           size_t ws_bytes, void* stream) {
  if (!codes || !scales_e8m0 || !fp8_out || !row_scale || !ws) return FP4MOE_ERR_INVALID_ARG;
  if (rows < 0 || K <= 0 || K % 32 != 0) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < 256) return FP4MOE_ERR_WORKSPACE;
  if (!aligned16(codes) || !aligned16(fp8_out)) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  return cuda_status(launch_convert(codes, scales_e8m0, rows, K, fp8_out, row_scale, row_status,
                                    static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_check_scales(const uint8_t* scales, int64_t n, int32_t fmt, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!scales || !ws || n < 0) return FP4MOE_ERR_INVALID_ARG;
  if (fmt != FP4MOE_MXFP4 && fmt != FP4MOE_NVFP4) return FP4MOE_ERR_INVALID_ARG;
  if (ws_bytes < 256) return FP4MOE_ERR_WORKSPACE;
  if (!aligned16(scales)) return FP4MOE_ERR_INVALID_ARG;
  if (fp4moe_status st = check_device()) return st;
  return cuda_status(launch_nan_scales(scales, n, fmt == FP4MOE_NVFP4, static_cast<int32_t*>(ws),
                                       static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_clear_status(void* ws, void* stream) {
  if (!ws) return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, kStatusInts * 4, static_cast<cudaStream_t>(stream)));
}

fp4moe_status fp4moe_get_status(void* ws, void* stream, fp4moe_status* st, int64_t* count) {
  if (!ws) return FP4MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h[kStatusInts];
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP4MOE_ERR_CUDA;
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FP4MOE_ERR_CUDA;
  if (st) *st = static_cast<fp4moe_status>(h[ST_FIRST]);
  if (count) *count = h[ST_COUNT];
  return FP4MOE_OK;
}

}  // extern "C"
