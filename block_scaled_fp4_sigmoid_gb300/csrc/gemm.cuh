// Persistent grouped GEMM on block-scaled FP4 tensor cores (tcgen05) for the
// two expert projections of the MoE layer.
//
// The block-scaled product follows "Serve Kimi-K2.5-MXFP4 on MI355X with
// ATOM" (Figure 1 and section "When Is the Scale Applied?"): payloads and
// per-block scales of both operands go into the matrix instruction, which
// applies the scales inside the product.  On sm_103a that instruction is
// tcgen05.mma .kind::mxf4 (E8M0 per 32) or .kind::mxf4nvf4 (E4M3 per 16),
// with fp32 accumulators in tensor memory.
//
// Operand roles ("swap AB"): A = 128 weight rows (M = 128), B = up to N
// tokens of one expert (N = 16 / 32 / 64 / 112), both K-major.  A work unit is
// (expert, 128-row weight tile, token tile); units of one expert are laid
// out weight-tile-major so concurrent CTAs share each weight tile through L2.
//
// Warp roles (288 threads for gate/up, 256 for down; one CTA per SM,
// persistent over units):
//   warp 0     TMA producer: weight tiles (3-D tensor map over [E, rows,
//              K/2], or over the tiled payload layout), token tiles (2-D map
//              over the padded permuted rows), scale groups (bulk copies of
//              the tiled scale layout);
//   warps 1, 6 MMA issuers (warp 1 also owns tensor memory): copy each
//              stage's scale factors to tensor memory (tcgen05.cp), issue four
//              K=64 MMAs per 256-wide K tile (gate/up: one A operand each;
//              down units of two weight tiles: one tile each; other down
//              units: alternate K tiles into two accumulators, or one issuer
//              for two token slots), and commit the stage back to the
//              producer;
//   warp 7     second TMA producer: the token tile (2-D map over the padded
//              permuted rows) and its scale groups, once warp 0 has armed
//              the stage;
//   warp 8     gate/up only: zeroes the combine buffer when asked;
//   warps 2-5  epilogue, one per tensor-memory lane quadrant (down with
//              64 or more token columns: warps 8-11 as a second set):
//              gate/up: SwiGLU, then MXFP4 requantisation of h across the
//              32 lanes of a warp (= one 32-block along I), or (NVFP4) fp32
//              h plus a per-expert amax;
//              down: routing weight times y, added into the fp32 combine
//              buffer (red.global.add).
// Every wait is bounded (pipeline waits by KParams::wait_ns, and they give
// up once another role of the CTA has aborted); a timeout sets a CTA-wide
// abort flag, records FP4MOE_ERR_TIMEOUT in the status word, drains
// in-flight copies and MMAs, frees tensor memory and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

struct KParams {
  CUtensorMap tmA;     // routed weights, uint8 [E, rows_per_expert, K/2] (or the tiled layout)
  CUtensorMap tmA_sh;  // shared expert weights, uint8 [1, rows_per_expert, K/2] (or tiled)
  CUtensorMap tmB;     // activations, uint8 [rows_cap, K/2]
  const uint8_t *wsf, *shsf, *bsf;
  const float *gw, *gb;
  const int32_t *expert_count, *expert_slot, *unit_start, *total_units;
  const int32_t* row_tok;
  const float* row_w;
  // gate/up with few tokens: B is the token rows 0..T-1 for every unit (x
  // quantised once per token) and column t is kept when bit t of
  // tok_mask[expert] is set; null: B is the unit's token tile
  const uint32_t* tok_mask;
  uint8_t *hq, *hsf;
  float *h32, *h_dbg, *out_acc;
  float4* zero_buf;  // gate/up: fp32 buffer warp 7 zeroes (the down GEMM's combine buffer), nullable
  int64_t zero_n4;   // its size in float4
  uint32_t* amax_h;
  int32_t* status;
  int E, n_exp, H, I, K, rows_per_expert, m_tiles, katoms_a, katoms_b, katoms_h, has_shared, T;
  int plan_early;  // the plan was written at least two kernels back (see the kernel)
  int w_tiled;     // weights in the tiled layout (tmA / tmA_sh are views of 128-byte rows)
  int gu_pairs;    // gate/up: weights and scales in the gate/up-paired tiled order (I / 128 pairs), else 0
  int unit_mtiles;  // weight tiles per unit row (128 rows each; 256 on CTA pairs)
  int m_group;      // weight tiles per group of the unit order (divides unit_mtiles)
  uint64_t wait_ns;  // limit of the pipeline waits (drains keep kWaitLimitNs)
  int withhold;      // gate/up test knob: CTA 0 never fills its first pipeline stage
  // W8A8 (E4M3 operands): per-row fp32 scales of the weights (routed [E,
  // rows], shared [rows]) and of the B rows (per permuted row); amax_h then
  // holds the gate/up intermediate's |max| per permuted row
  const float *wrs, *shrs, *brs;
};

// Operand kinds: block-scaled FP4 (MXFP4 or NVFP4 by NV; 256-value K tiles,
// scale factors through tensor memory), E4M3 (W8A8; 128-value K tiles) and
// BF16 (the NVFP4 emulation mode; 64-value K tiles).  Every K tile is one
// 128-byte swizzle row per operand row, consumed by four MMAs of 32 bytes.
constexpr int kOpFp4 = 0, kOpE4M3 = 1, kOpBf16 = 2;

constexpr int kMaxExperts = 520;  // plan arrays cached in shared memory (E + n_shared <= 513)

template <int N, bool GATEUP, bool NV, int OP = kOpFp4, bool PAIR = false, bool W2 = false>
struct GemmCfg {
  // N = 240 (MXFP4 down only): a unit covers two slots of the padded layout
  // (two 112-token tiles of one expert), so each pipeline step carries
  // twice the MMA work of a 112-token unit.  The B tile is two 112-row
  // boxes at rows 0 and 128, so that B row r keeps the scale row r of the
  // slots' 128-row scale groups; columns 112..127 hold stale rows the
  // epilogue never reads.
  static constexpr int kPairSlots = N == 240 ? 2 : 1;
  static constexpr int kUnitRoutes = kPairSlots == 2 ? 224 : N;  // routes one unit covers
  static_assert(kPairSlots == 1 || (!GATEUP && OP == kOpFp4), "paired slots: FP4 down GEMM only");
  // PAIR: a cluster of two CTAs runs each unit as M = 256 MMAs (tcgen05
  // .cta_group::2): CTA r of the pair holds weight rows 128 r .. 128 r + 127
  // of the unit's 256 and B rows 120 r .. 120 r + 119 of the 240: CTA 0 the
  // first slot's tokens at its rows 0..111, CTA 1 the second slot's at its
  // rows 8..119 (B rows 128..239, matching the scale rows of the second
  // slot's scale group).  Both CTAs hold both slots' B scale groups, as each
  // SM's half of the MMA scales all 240 columns.
  static_assert(!PAIR || (N == 240 && !GATEUP && !NV && OP == kOpFp4), "CTA pair: MXFP4 down GEMM with paired slots");
  // W2 (MXFP4 down, 112-token tiles): a unit covers two adjacent 128-row weight
  // tiles (256 output rows) of one token tile, the gate/up GEMM's mainloop
  // shape: issuer i multiplies weight tile i (A operand i) by the shared B
  // tile into its own accumulator block, and the epilogue adds both blocks
  // into their output rows.
  static_assert(!W2 || (N == 112 && !GATEUP && !NV && !PAIR && OP == kOpFp4), "two weight tiles: MXFP4 down, 112 tokens");
  static constexpr int kBRows = PAIR ? N / 2 : N;  // B rows in this CTA's shared memory
  static constexpr int kA = (GATEUP || W2) ? 2 : 1;        // A operands per unit (gate and up, or two weight tiles)
  static constexpr int kAtoms = OP != kOpFp4 ? 0 : NV ? 4 : 2;  // scale groups per K tile
  static constexpr int kABytes = 128 * 128;          // 128 rows x 128 bytes
  static constexpr int kBBytes = kBRows * 128;
  static constexpr int kSFBytes = kAtoms * 512;      // per 128-row operand and K tile
  static constexpr int kSFBBytes = kSFBytes * kPairSlots;  // B side: one set per 128 rows of B
  static constexpr int kOffA1 = kABytes;
  static constexpr int kOffB = kA * kABytes;
  static constexpr int kOffSFA0 = kOffB + kBBytes;
  static constexpr int kOffSFA1 = kOffSFA0 + kSFBytes;
  static constexpr int kOffSFB = kOffSFA0 + kA * kSFBytes;
  static constexpr int kStage = kOffSFB + kSFBBytes;
  // bytes the copies of one stage deliver (paired slots: two 112-row boxes
  // into the 240-row B tile)
  static constexpr int kTx = kStage - kBBytes + (kPairSlots == 2 ? 2 * 112 * 128 : kBBytes);
  // Epilogue warps: one per tensor-memory lane quadrant, or (down GEMM with
  // 64 or more token columns) two per quadrant, splitting the unit's 32-column
  // chunks between them.  Gate/up transposes through shared memory (one
  // 32 x 33 fp32 tile per epilogue warp); down transposes in registers.
  static constexpr int kEpiWarps = (!GATEUP && N >= 64) ? 8 : 4;
  static constexpr int kEpiSets = kEpiWarps / 4;  // epilogue warps per lane quadrant
  static constexpr int kEpiTiles = GATEUP ? 4 : 1;
  // 227 KB per CTA = pipeline stages + 1 KB alignment slack + static shared
  // memory (epilogue transpose tiles, plan cache, barriers and flags)
  static constexpr int kStaticBytes = kEpiTiles * 32 * 33 * 4 + 4 * 4 * kMaxExperts + 512;
  static constexpr int kBudget = 232448 - 1024 - kStaticBytes;
  static constexpr int kStages = (kBudget / kStage) > 8 ? 8 : (kBudget / kStage);
  static constexpr int kSmem = kStages * kStage + 1024;
  // Two MMA-issuing threads (warps 1 and 6): a thread issues a tcgen05
  // instruction only every ~50 cycles, so one thread cannot keep the tensor
  // pipe busy with 112-token MMAs.  Gate/up: issuer i drives A operand i
  // (gate, up).  Down (one A operand): issuer i takes the K tiles kt with
  // kt % 2 == i into its own accumulator; the epilogue adds the two.  Each
  // issuer copies its own A and B scale factors.  (W2: issuer i drives
  // weight tile i, as gate/up.  N = 240: one issuer; its instructions
  // already carry twice the work.)
  static constexpr int kIssuers = kPairSlots == 2 ? 1 : 2;  // (CTA pair: in CTA 0 only)
  static constexpr bool kKSplit = !GATEUP && !W2 && kIssuers == 2;
  // warp 7: second producer; gate/up warp 8: combine-buffer zeroing; down
  // with eight epilogue warps: warps 8-11 are the second four
  static constexpr int kThreads = GATEUP ? 288 : 32 * (4 + kEpiWarps);
  static constexpr int kAccCols = kIssuers * N;  // one accumulator set: one N-column block per issuer
  // scale-factor columns of one K tile: 4 per group of 4 blocks per 128
  // rows (row r of a group at lane r % 32, column r / 32)
  static constexpr int kSfColsA = kAtoms * 4, kSfColsB = kAtoms * 4 * kPairSlots;
  static constexpr int kSfCols = kIssuers * (kSfColsA + kSfColsB);
  // two accumulator sets when they fit: the epilogue of one unit then
  // overlaps the MMAs of the next
  static constexpr int kAccStages = (2 * kAccCols + kSfCols <= 512) ? 2 : 1;
  static constexpr int kSfaCol = kAccStages * kAccCols;
  static constexpr int kSfbCol = kSfaCol + kIssuers * kSfColsA;   // issuer i's A scales at kSfaCol + i * kSfColsA, B at kSfbCol + i * kSfColsB
  static constexpr int kCols = kSfaCol + kSfCols;
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "tensor memory");
  static_assert(kStage % 1024 == 0, "stage alignment");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kStages * kStage + 1024 + kStaticBytes <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) { return smem_desc(saddr, 0, 128, 0); }

// Unit u -> (expert, weight tile, token-tile slot, tokens in the tile), from
// the plan cached in shared memory (s_start[e] = M x the token tiles of the
// experts before e, s_start[n_exp] = all units).  The M weight tiles of a
// unit row are taken in groups of G (G divides M): group g holds, expert by
// expert, tiles g G .. g G + G - 1, each with all of the expert's token
// tiles (token tile fastest).  G = M is expert-major order; a smaller G
// keeps the down GEMM's combine rows of one group (T x G x 128 fp32) in L2
// while every expert adds into them.
//
// Each role of a CTA decodes its units (u_first, u_first + u_step, ...) in
// rising order and keeps a UnitPos: the expert and group of its last unit.
// The next unit's expert is that expert again (one read of shared memory
// tells) or one after it, found by bisection of the experts that follow.
// {0, 0} is a valid position for any unit.
struct UnitPos {
  int e = 0, g = 0;
};

// The last i in [lo, n) with key(i) <= x, given key(lo) <= x and key
// nondecreasing in i.
template <class Key>
__device__ __forceinline__ int search_last_le(Key key, int lo, int n, int x) {
  if (lo + 1 >= n || key(lo + 1) > x) return lo;
  int hi = n;
  ++lo;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (key(mid) <= x) lo = mid;
    else hi = mid;
  }
  return lo;
}

template <int N, bool kGrouped>
__device__ __forceinline__ void decode_unit(const int32_t* s_start, const int32_t* s_count, const int32_t* s_slot,
                                            int n_exp, int M, int G, int u, UnitPos& pos, int& e, int& mt, int& slot,
                                            int& cnt) {
  int local;
  if (!kGrouped || G == M) {  // the expert: the last one whose first unit is <= u
    e = search_last_le([&](int i) { return s_start[i]; }, pos.e, n_exp, u);
    local = u - s_start[e];
  } else {
    const int per_group = (s_start[n_exp] / M) * G;  // units of one group
    if (u >= (pos.g + 1) * per_group) {  // a later group: search it from the first expert
      pos.g = u / per_group;
      pos.e = 0;
    }
    const int r = u - pos.g * per_group;
    // the last expert whose first unit of the group, s_start / M x G, is <= r
    // (s_start is a multiple of M)
    e = search_last_le([&](int i) { return s_start[i] * G; }, pos.e, n_exp, r * M);
    local = r - (s_start[e] / M) * G;
  }
  pos.e = e;
  const int count = s_count[e];
  constexpr int kCap = GemmCfg<N, false, false>::kUnitRoutes;
  const int nt = (count + kCap - 1) / kCap;
  const int ml = local / nt;
  const int ti = local - ml * nt;
  mt = (kGrouped ? pos.g * G : 0) + ml;
  slot = s_slot[e] + ti * GemmCfg<N, false, false>::kPairSlots;
  cnt = min(kCap, count - ti * kCap);
}

// GROUPED: the instance decodes the grouped unit order (KParams::m_group <
// unit_mtiles); the others are compiled with the expert-major order only
// (measured: the grouped decode merely present cost the decode and NVFP4
// down GEMMs 2-3%).
template <int N, bool GATEUP, bool NV, int OP = kOpFp4, bool PAIR = false, bool GROUPED = false, bool W2 = false,
          bool DPW = false>
__global__ void __launch_bounds__(GemmCfg<N, GATEUP, NV, OP, PAIR, W2>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ KParams p) {
  using C = GemmCfg<N, GATEUP, NV, OP, PAIR, W2>;
  static_assert(!DPW || (!GATEUP && OP == kOpFp4), "row-tile-paired weights: block-scaled FP4 down GEMM");
  constexpr bool F8 = OP == kOpE4M3, BF = OP == kOpBf16, SF = OP == kOpFp4;
  static_assert(SF || !NV, "one operand format");
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[C::kStages];
  __shared__ __align__(8) uint64_t bar_empty[C::kStages];
  __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_done;
  __shared__ __align__(8) uint64_t bar_pfull[PAIR ? C::kStages : 1];  // CTA pair, CTA 0: the peer's stage has landed
  __shared__ float epi_tile[C::kEpiTiles][32][33];  // gate/up, per epilogue warp: 32 lanes x 32 columns, transposed
  __shared__ int32_t s_start[kMaxExperts], s_count[kMaxExperts], s_slot[kMaxExperts];
  __shared__ uint32_t s_mask[kMaxExperts];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int armed_steps, first_done;  // split producers (down): steps the first has armed; it has finished

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pair: rank in the pair (0 issues the MMAs); both CTAs of a pair run
  // the same units
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const int u_first = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int u_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  const int KT = (p.K + (BF ? 63 : F8 ? 127 : 255)) / (BF ? 64 : F8 ? 128 : 256);  // K tiles of 128 bytes

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), C::kKSplit ? 1 : C::kIssuers);  // the issuers that read the stage
      if constexpr (PAIR) mbar_init(smem_u32(&bar_pfull[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&bar_tfull[a]), C::kIssuers);
      mbar_init(smem_u32(&bar_tempty[a]), C::kEpiWarps * (PAIR ? 2 : 1));  // (pair: both CTAs' epilogues)
    }
    mbar_init(smem_u32(&bar_done), C::kIssuers);
    abort_flag = 0;
    armed_steps = 0;
    first_done = 0;
    if constexpr (PAIR) fence_barrier_init_cluster();
    else fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // both CTAs allocate the pair's columns together
      tmem_alloc_pair(smem_u32(&tmem_slot), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tmA);
    prefetch_tmap(&p.tmB);
    if (p.has_shared) prefetch_tmap(&p.tmA_sh);
  }
  // The plan (unit table, expert counts, slots, token masks): when it was
  // written at least two kernels back (plan_early) it is complete here, as
  // the previous kernel signals its dependents only after its own dependency
  // wait; when the previous kernel wrote it, it is read after the wait.  The
  // previous kernel's activations are always read after the wait.
  if (!p.plan_early) pdl_wait();
  const int total = *p.total_units;
  for (int i = threadIdx.x; i <= p.n_exp; i += blockDim.x) {
    s_start[i] = p.unit_start[i];
    if (i < p.n_exp) {
      s_count[i] = p.expert_count[i];
      s_slot[i] = p.expert_slot[i];
      if (p.tok_mask) s_mask[i] = p.tok_mask[i];
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_arrive_wait();  // the peer's barriers are initialised before any remote arrive
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_v = &abort_flag;

  // Weight side of one pipeline step (A tiles and their scale groups): it
  // depends on nothing the previous kernel writes.
  struct Step {
    const CUtensorMap* tmA;
    int ec, row0, row1, slot;
    bool once;  // the expert has one token tile: no other unit reads these weight tiles
    bool two;   // paired slots: the unit's routes reach into its second slot
    const uint8_t *sfa0, *sfa1, *sfb;
  };
  auto unit_step = [&](int u, UnitPos& pos) {
    int e, mt, slot, cnt;
    decode_unit<N, GROUPED>(s_start, s_count, s_slot, p.n_exp, p.unit_mtiles, p.m_group, u, pos, e, mt, slot, cnt);
    const bool sh = e >= p.E;
    Step st;
    st.tmA = sh ? &p.tmA_sh : &p.tmA;
    st.ec = sh ? e - p.E : e;
    const uint8_t* sfw = sh ? p.shsf : p.wsf;
    const int rt_per_e = p.rows_per_expert >> 7;
    // (CTA pair and W2: mt counts 256-row tiles)
    st.row0 = PAIR ? mt * 256 + (int)crank * 128 : W2 ? mt * 256 : mt * 128;
    st.row1 = W2 ? mt * 256 + 128 : p.I + mt * 128;  // second A operand: up rows, or (W2) the next weight tile
    st.slot = p.tok_mask ? 0 : slot;  // slot of the B rows
    st.once = s_count[e] <= C::kUnitRoutes;
    st.two = C::kPairSlots == 2 && cnt > 112;
    st.sfa0 = sfw + ((int64_t)(st.ec * rt_per_e + (st.row0 >> 7)) * p.katoms_a) * 512;
    st.sfa1 = sfw + ((int64_t)(st.ec * rt_per_e + (st.row1 >> 7)) * p.katoms_a) * 512;
    if (GATEUP && p.gu_pairs)  // paired order: gate then up scale groups of each K tile, kSFBytes apart
      st.sfa0 = sfw + ((int64_t)(st.ec * p.gu_pairs + mt) * KT) * 2 * C::kSFBytes;
    if constexpr (DPW) {  // row-tile-paired order: row tile rt's groups of K tile kt at slot
      // ((slab * KT + kt) * 2 + rt % 2) * kSFBytes, slab = the 256-row slab (2 * kSFBytes per K tile)
      st.sfa0 = sfw + ((int64_t)(((st.ec * rt_per_e) >> 1) + (st.row0 >> 8)) * KT * 2 + ((st.row0 >> 7) & 1)) * C::kSFBytes;
      st.sfa1 = sfw + ((int64_t)(((st.ec * rt_per_e) >> 1) + (st.row1 >> 8)) * KT * 2 + ((st.row1 >> 7) & 1)) * C::kSFBytes;
    }
    st.sfb = p.bsf + ((int64_t)st.slot * p.katoms_b) * 512;
    return st;
  };
  // Weight tiles read by one unit only stream with an evict-first L2 policy
  // (measured: a 128-row-box weight stream goes from 5.0 to 5.7 TB/s); tiles
  // shared by the units of several token tiles keep the default policy so
  // that those units find them in L2.
  const uint64_t pol_once = l2_evict_first();
  // Coordinates of the (row tile, K tile) box: row-major (byte column, row)
  // or, in the tiled layout, the block's first 128-byte row of the view
  // (DPW, row-tile-paired order: block slot (slab * KT + kt) * 2 + row tile
  // % 2).  The order is a template parameter: as a run-time branch in these
  // per-K-tile computations it cost the decode-size down GEMMs 3-6%.
  auto a_x = [&](int kt) { return p.w_tiled ? 0 : kt * 128; };
  auto a_y = [&](int row, int kt) {
    if (!p.w_tiled) return row;
    if constexpr (DPW) return (((row >> 8) * KT + kt) * 2 + ((row >> 7) & 1)) * 128;
    return ((row >> 7) * KT + kt) * 128;
  };
  // scale bytes from one K tile of a row tile to the next
  constexpr int sf_kstep = DPW ? 2 * C::kSFBytes : C::kSFBytes;
  auto load_weights = [&](const Step& st, int kt, uint32_t base, uint32_t fb) {
    if constexpr ((GATEUP || W2) && SF) {
      // paired orders (gate/up pairs; W2 on row-tile pairs): one box of the
      // unit's two blocks, one copy of both scale groups
      if (GATEUP ? p.gu_pairs != 0 : DPW) {
        const int y = ((GATEUP ? st.row0 >> 7 : st.row0 >> 8) * KT + kt) * 256;
        if (st.once) {
          tma_load_3d_hint(base, st.tmA, fb, 0, y, st.ec, pol_once);
          bulk_load_hint(base + C::kOffSFA0, st.sfa0 + kt * 2 * C::kSFBytes, 2 * C::kSFBytes, fb, pol_once);
        } else {
          tma_load_3d(base, st.tmA, fb, 0, y, st.ec);
          bulk_load(base + C::kOffSFA0, st.sfa0 + kt * 2 * C::kSFBytes, 2 * C::kSFBytes, fb);
        }
        return;
      }
    }
    if (st.once) {
      tma_load_3d_hint(base, st.tmA, fb, a_x(kt), a_y(st.row0, kt), st.ec, pol_once);
      if constexpr (C::kA == 2)
        tma_load_3d_hint(base + C::kOffA1, st.tmA, fb, a_x(kt), a_y(st.row1, kt), st.ec, pol_once);
      if constexpr (SF) {
        bulk_load_hint(base + C::kOffSFA0, st.sfa0 + kt * sf_kstep, C::kSFBytes, fb, pol_once);
        if constexpr (C::kA == 2)
          bulk_load_hint(base + C::kOffSFA1, st.sfa1 + kt * sf_kstep, C::kSFBytes, fb, pol_once);
      }
    } else {
      tma_load_3d(base, st.tmA, fb, a_x(kt), a_y(st.row0, kt), st.ec);
      if constexpr (C::kA == 2) tma_load_3d(base + C::kOffA1, st.tmA, fb, a_x(kt), a_y(st.row1, kt), st.ec);
      if constexpr (SF) {
        bulk_load(base + C::kOffSFA0, st.sfa0 + kt * sf_kstep, C::kSFBytes, fb);
        if constexpr (C::kA == 2) bulk_load(base + C::kOffSFA1, st.sfa1 + kt * sf_kstep, C::kSFBytes, fb);
      }
    }
  };
  auto load_acts = [&](const Step& st, int kt, uint32_t base, uint32_t fb) {
    if constexpr (PAIR) {  // this CTA's slot box, and both slots' scale groups
      if (crank == 0) tma_load_2d(base + C::kOffB, &p.tmB, fb, kt * 128, st.slot * kSlotRows);
      else if (st.two) tma_load_2d(base + C::kOffB + 8 * 128, &p.tmB, fb, kt * 128, (st.slot + 1) * kSlotRows);
      bulk_load(base + C::kOffSFB, st.sfb + kt * C::kSFBytes, C::kSFBytes, fb);
      if (st.two)
        bulk_load(base + C::kOffSFB + C::kSFBytes, st.sfb + (int64_t)p.katoms_b * 512 + kt * C::kSFBytes, C::kSFBytes,
                  fb);
      return;
    }
    tma_load_2d(base + C::kOffB, &p.tmB, fb, kt * 128, st.slot * kSlotRows);
    if constexpr (SF) bulk_load(base + C::kOffSFB, st.sfb + kt * C::kSFBytes, C::kSFBytes, fb);
    if (st.two) {  // the unit's second slot: B rows 128..239 and their scale groups
      tma_load_2d(base + C::kOffB + 128 * 128, &p.tmB, fb, kt * 128, (st.slot + 1) * kSlotRows);
      bulk_load(base + C::kOffSFB + C::kSFBytes, st.sfb + (int64_t)p.katoms_b * 512 + kt * C::kSFBytes, C::kSFBytes,
                fb);
    }
  };

  // bytes one stage of the unit receives (paired slots: the second slot's
  // box and scale groups only when the unit reaches into it)
  auto stage_tx = [&](const Step& st) -> uint32_t {
    if constexpr (PAIR)
      return C::kABytes + C::kSFBytes + ((crank == 0 || st.two) ? 112 * 128 : 0) + (st.two ? 2 : 1) * C::kSFBytes;
    return (C::kPairSlots == 2 && !st.two) ? C::kTx - 112 * 128 - C::kSFBytes : C::kTx;
  };
  // Test knob (gate/up): CTA 0 never fills pipeline step 0, so its MMA
  // issuer's wait for it runs out (KParams::withhold).
  const int withheld = (GATEUP && p.withhold && blockIdx.x == 0) ? 0 : -1;
  // The first pipeline stages start streaming weights before the wait, so
  // they overlap the tail of the previous kernel.
  int pre = 0;
  if (warp == 0 && lane == 0) {
    UnitPos pos;
    for (int u = u_first; u < total && pre < C::kStages; u += u_step) {
      const Step st = unit_step(u, pos);
      for (int kt = 0; kt < KT && pre < C::kStages; ++kt, ++pre) {
        if (pre == withheld) continue;
        const uint32_t fb = smem_u32(&bar_full[pre]);
        mbar_arrive_expect_tx(fb, stage_tx(st));  // stage is empty: first use
        load_weights(st, kt, sbase + pre * C::kStage, fb);
      }
    }
  }
  if (p.plan_early) pdl_wait();
  pdl_trigger();  // the plan is complete, so the next kernel may launch now
  volatile int* armed_v = &armed_steps;
  volatile int* first_done_v = &first_done;

  // A second thread (warp 7) issues the activation copies of every stage:
  // a thread is held ~90-140 cycles by each copy it issues, so one thread's
  // issue time paced the stages (measured: DeepSeek NVFP4 down 268 -> 240
  // us; gate/up, prefill 0.604 -> 0.590 ms and skewed 1.955 -> 1.846 ms).
  constexpr bool kSplitProducer = true;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      if constexpr (kSplitProducer) *armed_v = pre;
      int stage = 0, step = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      UnitPos pos;
      for (int u = u_first; u < total && !*abort_v; u += u_step) {
        const Step st = unit_step(u, pos);
        bool ok = true;
        for (int kt = 0; kt < KT; ++kt, ++step) {
          const uint32_t fb = smem_u32(&bar_full[stage]);
          const uint32_t base = sbase + stage * C::kStage;
          if (step == withheld) {  // never armed, never filled
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            continue;
          }
          if (step >= pre) {
            if (!mbar_wait_abortable<PAIR>(smem_u32(&bar_empty[stage]), phase ^ 1u, p.wait_ns, abort_v)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(fb, stage_tx(st));
            if constexpr (kSplitProducer) {  // the stage is free and armed (release to the second producer)
              __threadfence_block();
              *armed_v = step + 1;
            }
            load_weights(st, kt, base, fb);
          }
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if constexpr (!kSplitProducer) load_acts(st, kt, base, fb);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) {
          if (!*abort_v) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
          *abort_v = 1;
          break;
        }
      }
      if constexpr (kSplitProducer) {
        // prologue stages this loop did not reach (abort): the second
        // producer completes them, and they are waited on below
        for (int s2 = step; s2 < pre; ++s2) {
          if (s2 == withheld) continue;
          armed |= 1u << s2;
          armed_par &= ~(1u << s2);  // first use: phase 0
        }
        __threadfence_block();
        *first_done_v = 1;
      }
      // stages whose weights were requested before the wait but whose unit
      // was not reached (abort) get their activation copies too, so that
      // their barriers complete (split: the second producer does it)
      if (!kSplitProducer && step < pre) {
        int s2 = 0;
        UnitPos pos2;
        for (int u = u_first; u < total && s2 < pre; u += u_step) {
          const Step st = unit_step(u, pos2);
          for (int kt = 0; kt < KT && s2 < pre; ++kt, ++s2)
            if (s2 >= step && s2 != withheld) {
              load_acts(st, kt, sbase + s2 * C::kStage, smem_u32(&bar_full[s2]));
              armed |= 1u << s2;
              armed_par &= ~(1u << s2);  // first use: phase 0
            }
        }
      }
      // every armed stage must have landed before the CTA exits
      for (int s = 0; s < C::kStages; ++s)
        if ((armed >> s) & 1u) (void)mbar_wait<PAIR>(smem_u32(&bar_full[s]), (armed_par >> s) & 1u);
    }
  } else if (warp == 7) {
    if constexpr (kSplitProducer) {
      // -------------------------------------------------------- second producer
      // The activation side of every stage, in the first producer's order,
      // once the first producer has armed the stage (it waited for the
      // stage's release; its arrive.expect_tx counts these bytes too).  So
      // every copy issued here belongs to a stage the first producer waits on
      // before the CTA exits.
      if (lane == 0) {
        // bounded wait until the first producer has armed more than j steps
        auto wait_armed = [&](int j) {
          const uint64_t t0 = globaltimer();
          while (*armed_v <= j) {
            if (*abort_v || globaltimer() - t0 > p.wait_ns) return false;
            __nanosleep(32);
          }
          return true;
        };
        int step = 0;
        bool ok = true;
        UnitPos pos;
        for (int u = u_first; u < total && ok && !*abort_v; u += u_step) {
          const Step st = unit_step(u, pos);
          for (int kt = 0; kt < KT; ++kt, ++step) {
            if (step == withheld) continue;  // never armed
            if (!wait_armed(step)) { ok = false; break; }
            __threadfence_block();  // acquire: the stage's release precedes these copies
            const int stage = step % C::kStages;
            load_acts(st, kt, sbase + stage * C::kStage, smem_u32(&bar_full[stage]));
          }
        }
        if (!ok && !*abort_v) {
          *abort_v = 1;
          record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
        }
        if (!ok || *abort_v) {
          // abort: once the first producer has stopped, the armed stages not
          // reached here get their activation copies, so that its final
          // waits on them complete
          const uint64_t t0 = globaltimer();
          while (!*first_done_v && globaltimer() - t0 < kWaitLimitNs) __nanosleep(64);
          __threadfence_block();
          const int armed = *armed_v;
          int s2 = 0;
          UnitPos pos2;
          for (int u = u_first; u < total && s2 < armed; u += u_step) {
            const Step st = unit_step(u, pos2);
            for (int kt = 0; kt < KT && s2 < armed; ++kt, ++s2)
              if (s2 >= step && s2 != withheld)
                load_acts(st, kt, sbase + (s2 % C::kStages) * C::kStage, smem_u32(&bar_full[s2 % C::kStages]));
          }
        }
      }
    }
  } else if (GATEUP && warp == 8) {
    // ------------------------------------------------------------ zeroing
    // The combine buffer is read by the down GEMM, which starts after this
    // grid has completed; the writes overlap this kernel's MMAs.
    if (p.zero_buf) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int64_t i = (int64_t)blockIdx.x * 32 + lane; i < p.zero_n4; i += (int64_t)gridDim.x * 32) p.zero_buf[i] = z;
    }
  } else if (warp == 1 || warp == 6) {
   if (PAIR && crank == 1) {
    if (warp == 1) {
      // ---------------------------------------------------------- pair relay
      // CTA 1 of a pair: once a stage of this CTA has landed, tell CTA 0's
      // issuer (its MMAs read this CTA's half of the operands).
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = u_first; ok && u < total && !__any_sync(0xffffffffu, *abort_v); u += u_step) {
        for (int kt = 0; kt < KT; ++kt) {
          if (!__all_sync(0xffffffffu, mbar_wait_abortable<PAIR>(smem_u32(&bar_full[stage]), phase, p.wait_ns, abort_v))) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_remote(smem_u32(&bar_pfull[stage]), 0u);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        if (lane == 0 && !*abort_v) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
        __syncwarp();
        *abort_v = 1;
      }
    }
   } else if (warp == 1 || C::kIssuers == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer mi (warp 1 or 6) drives its MMAs into accumulator block mi.  The
    // whole warp runs the loop, so every operand (descriptors, tensor-memory
    // addresses) is warp-uniform; each tcgen05 instruction is issued by one
    // lane picked with elect.sync.
    const int mi = warp == 1 ? 0 : 1;
    const uint32_t t_sfa = tmem + C::kSfaCol + mi * C::kSfColsA;
    const uint32_t t_sfb = tmem + C::kSfbCol + mi * C::kSfColsB;
    const uint32_t off_a = (!C::kKSplit && mi) ? C::kOffA1 : 0u;
    const uint32_t off_sfa = (!C::kKSplit && mi) ? C::kOffSFA1 : C::kOffSFA0;
    // descriptors of stage 0; a stage s adds s * kStage / 16 to the start
    // address field (every address stays below 2^18, so the 14-bit field
    // does not carry)
    const uint64_t a_desc0 = desc_sw128(sbase + off_a), b_desc0 = desc_sw128(sbase + C::kOffB);
    const uint64_t sfa_desc0 = desc_sf(sbase + off_sfa), sfb_desc0 = desc_sf(sbase + C::kOffSFB);
    // bounded wait with a warp-uniform outcome
    auto wait_w = [&](uint32_t bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait_abortable<PAIR>(bar, par, p.wait_ns, abort_v));
    };
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    int as = 0;  // accumulator set of this unit
    UnitPos pos;
    for (int u = u_first; u < total && !__any_sync(0xffffffffu, *abort_v); u += u_step) {
      // paired slots: a unit within its first slot multiplies 112 columns
      // (decoded before the accumulator wait, off the MMAs' path)
      bool two = true;
      if constexpr (C::kPairSlots == 2) {
        int e_, mt_, slot_, cnt_;
        decode_unit<N, GROUPED>(s_start, s_count, s_slot, p.n_exp, p.unit_mtiles, p.m_group, u, pos, e_, mt_, slot_,
                                cnt_);
        two = cnt_ > 112;
      }
      bool ok = wait_w(smem_u32(&bar_tempty[as]), acc_phase ^ 1u);
      tc_fence_after();
      const uint32_t t_acc = tmem + as * C::kAccCols + mi * N;
      const uint32_t n_mma = two ? N : 112;
      for (int kt = 0; ok && kt < KT; ++kt) {
        if (C::kKSplit && (kt & 1) != mi) {  // the other issuer's K tile
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
          continue;
        }
        if (!wait_w(smem_u32(&bar_full[stage]), phase)) { ok = false; break; }
        if constexpr (PAIR)  // and the peer's half of the stage
          if (!wait_w(smem_u32(&bar_pfull[stage]), phase)) { ok = false; break; }
        tc_fence_after();
        const uint64_t so = (uint64_t)((stage * C::kStage) >> 4);
        const bool first = C::kKSplit ? kt == mi : kt == 0;  // first K tile of this accumulator
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) {
          // 512 bytes per scale group (pair: into both CTAs, each from its own
          // shared memory)
          if constexpr (PAIR) tc_cp_sf_pair_elect(t_sfa + 4 * a, sfa_desc0 + so + 32 * a);
          else tc_cp_sf_elect(t_sfa + 4 * a, sfa_desc0 + so + 32 * a);
#pragma unroll
          for (int h = 0; h < C::kPairSlots; ++h)  // B rows 128 h .. 128 h + 127: columns 4 h .. 4 h + 3 of the group
            if (h == 0 || two) {
              const uint32_t tb = t_sfb + 4 * C::kPairSlots * a + 4 * h;
              const uint64_t sb = sfb_desc0 + so + 32 * a + h * (C::kSFBytes >> 4);
              if constexpr (PAIR) tc_cp_sf_pair_elect(tb, sb);
              else tc_cp_sf_elect(tb, sb);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // 32 bytes of the 128-byte swizzle row per MMA
          const uint32_t accum = (!first || j) ? 1u : 0u;
          if constexpr (F8) {
            tc_mma_f8_elect(t_acc, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc_f8(N), accum);  // K = 32
          } else if constexpr (BF) {
            tc_mma_bf16_elect(t_acc, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc_bf16(N), accum);  // K = 16
          } else {
            const int atom = NV ? j : (j >> 1);
            const uint32_t sfid = NV ? 0u : (uint32_t)(j & 1) * 2u;
            if constexpr (PAIR) {  // M = 256 over the pair, all 240 columns
              tc_mma_mx_pair_elect(t_acc, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc_fp4(N, false, sfid, sfid, 256),
                                   t_sfa + 4 * atom, t_sfb + 4 * C::kPairSlots * atom, accum);
            } else {
              const uint32_t idesc = idesc_fp4(n_mma, NV, sfid, sfid);
              tc_mma_fp4_elect<NV>(t_acc, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, idesc, t_sfa + 4 * atom,
                                   t_sfb + 4 * C::kPairSlots * atom, accum);  // K = 64
            }
          }
        }
        if constexpr (PAIR) tc_commit_pair_elect(smem_u32(&bar_empty[stage]), 0x3);  // both CTAs' stage
        else tc_commit_elect(smem_u32(&bar_empty[stage]));
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) {
        if (lane == 0 && !*abort_v) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
        __syncwarp();
        *abort_v = 1;
        break;
      }
      if constexpr (PAIR) tc_commit_pair_elect(smem_u32(&bar_tfull[as]), 0x3);  // both CTAs' epilogues
      else tc_commit_elect(smem_u32(&bar_tfull[as]));
      if (++as == C::kAccStages) { as = 0; acc_phase ^= 1u; }
    }
    // all issued MMAs must finish before tensor memory is released
    if constexpr (PAIR) tc_commit_pair_elect(smem_u32(&bar_done), 0x1);
    else tc_commit_elect(smem_u32(&bar_done));
    (void)mbar_wait<PAIR>(smem_u32(&bar_done), 0);
   }
  } else if (warp < 6 || C::kEpiWarps > 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quadrant of this warp
    // set of this warp (warps 2-5: set 0, then four warps per set from warp
    // 8): which part of the unit it takes
    const int eset = warp < 8 ? 0 : (warp - 4) >> 2;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    float(*tile)[33] = epi_tile[GATEUP ? warp - 2 : 0];
    uint32_t acc_phase = 0;
    int as = 0;
    UnitPos pos;
    for (int u = u_first; u < total; u += u_step) {
      if (__any_sync(0xffffffffu, *abort_v)) break;  // warp-uniform: the loop body holds .sync.aligned loads
      int e, mt, slot, cnt;
      decode_unit<N, GROUPED>(s_start, s_count, s_slot, p.n_exp, p.unit_mtiles, p.m_group, u, pos, e, mt, slot, cnt);
      // the unit's accumulator set is complete (bounded; warp-uniform outcome)
      auto wait_acc = [&]() {
        if (!__all_sync(0xffffffffu, mbar_wait_abortable<PAIR>(smem_u32(&bar_tfull[as]), acc_phase, p.wait_ns, abort_v))) {
          if (lane == 0 && !*abort_v) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
          __syncwarp();
          *abort_v = 1;
          return false;
        }
        tc_fence_after();
        return true;
      };
      const int64_t row0 = (int64_t)slot * kSlotRows;
      if constexpr (GATEUP) {
        if (!wait_acc()) break;
        const uint32_t ta = tq + as * C::kAccCols;
        const int i0 = mt * 128 + 32 * q;  // first intermediate index of this warp's lanes
        float sc = 1.f;
        if constexpr (NV) sc = __fmul_rn(__ldg(p.gb), __ldg(p.gw + e));
        float amax = 0.f;
        const uint32_t mask = p.tok_mask ? s_mask[e] : 0u;
        const int ncol = p.tok_mask ? p.T : cnt;  // accumulator columns holding tokens
        // W8A8: this lane's gate and up row scales (channel scales of the
        // converted weights)
        float rg = 1.f, ru = 1.f;
        if constexpr (F8) {
          const float* rs = e >= p.E ? p.shrs : p.wrs + (int64_t)e * p.rows_per_expert;
          rg = __ldg(rs + i0 + lane);
          ru = __ldg(rs + p.I + i0 + lane);
        }
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          float g[32], uu[32];
          tc_ld32(ta + c0, g);
          tc_ld32(ta + N + c0, uu);
          float sx = 0.f;  // W8A8: scale of the activation row of column c0 + lane
          if constexpr (F8) sx = c0 + lane < ncol ? __ldg(p.brs + row0 + c0 + lane) : 0.f;
          tc_wait_ld();
          // lane l holds h(i0 + l, token c0 + j); transpose through shared memory
          // so that lane j then holds the 32 values of token c0 + j, one block
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float gv = g[j], uv = uu[j];
            if constexpr (NV) {
              gv = gv * sc;
              uv = uv * sc;
            }
            if constexpr (F8) {
              const float sxj = __shfl_sync(0xffffffffu, sx, j);
              gv = gv * rg * sxj;
              uv = uv * ru * sxj;
            }
            // silu(g) u with the hardware exponential and reciprocal (each
            // within a few units in the last place; e^-g = inf for g < -88
            // gives -0, the limit).  With the IEEE-rounded reciprocal this
            // loop took 4,300 cycles per 32-column chunk, 657 with this one.
            tile[j][lane] = gv * rcp_approx(1.0f + __expf(-gv)) * uv;
          }
          __syncwarp();
          const int n = c0 + lane;
          // column n -> row of the unit's tile: n itself, or (token columns)
          // the token's rank among the expert's tokens
          const bool keep = p.tok_mask ? (n < ncol && ((mask >> n) & 1u)) : n < cnt;
          if (keep) {
            const int64_t row = row0 + (p.tok_mask ? __popc(mask & ((1u << n) - 1u)) : n);
            float v[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) v[r] = tile[lane][r];
            if (p.h_dbg) {
              float4* dst = reinterpret_cast<float4*>(p.h_dbg + row * p.I + i0);
#pragma unroll
              for (int r = 0; r < 8; ++r) dst[r] = make_float4(v[4 * r], v[4 * r + 1], v[4 * r + 2], v[4 * r + 3]);
            }
            if constexpr (NV || F8 || BF) {
              float4* dst = reinterpret_cast<float4*>(p.h32 + row * p.I + i0);
#pragma unroll
              for (int r = 0; r < 8; ++r) dst[r] = make_float4(v[4 * r], v[4 * r + 1], v[4 * r + 2], v[4 * r + 3]);
              float m = 0.f;
#pragma unroll
              for (int r = 0; r < 32; ++r) m = fmaxf(m, fabsf(v[r]));
              if constexpr (F8) atomicMax(p.amax_h + row, __float_as_uint(m));  // per permuted row
              else amax = fmaxf(amax, m);                                      // per expert
            } else {
              uint32_t pk[4], sb;
              mx_quant32(v, pk, &sb);
              *reinterpret_cast<uint4*>(p.hq + row * (p.I >> 1) + (i0 >> 1)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              p.hsf[sf_tiled_offset(row, i0 >> 5, p.katoms_h)] = (uint8_t)sb;
              if (mt == p.m_tiles - 1 && p.katoms_h > p.m_tiles)  // pad group up to the K tile: scale 1.0
                p.hsf[sf_tiled_offset(row, 4 * p.m_tiles + q, p.katoms_h)] = 127;
            }
          }
          __syncwarp();
        }
        if constexpr (NV || BF) {  // the intermediate's NVFP4 tensor scale is per expert
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          if (lane == 0) atomicMax(p.amax_h + e, __float_as_uint(amax));
        }
      } else {
        // routing weight times y added into the fp32 combine buffer.  Lane l
        // holds output row 32 q + l of the unit's 128 for the 32 token
        // columns of a chunk; a 4 x 4 transpose within each group of four
        // lanes (two shuffle rounds) leaves lane 4 m + r with rows 4 m ..
        // 4 m + 3 of column 4 g + r, which one 16-byte reduction adds.
        // (W2: the warps of an even set take accumulator block 0, the unit's
        // first weight tile, those of an odd set block 1.)
        const int m4 = lane >> 2, r4 = lane & 3;
        const int blk = W2 ? (eset & 1) : 0;
        const int h0 = (PAIR ? mt * 256 + (int)crank * 128 : mt * (128 * C::kA) + 128 * blk) + 32 * q + 4 * m4;
        float sc = 1.f;
        if constexpr (NV) sc = __fmul_rn(__ldg(p.gb + e), __ldg(p.gw + e));
        float rho = 1.f;  // W8A8: channel scale of this lane's output row
        if constexpr (F8)
          rho = __ldg((e >= p.E ? p.shrs : p.wrs + (int64_t)e * p.rows_per_expert) + mt * 128 + 32 * q + lane);
        // the unit's routes: columns 0 .. cnt0 - 1 and (paired slots) 128 ..
        // 128 + cnt1 - 1, column n holding row row0 + n
        const int cnt0 = C::kPairSlots == 2 ? min(cnt, 112) : cnt;
        const int cnt1 = cnt - cnt0;
        const int ncol = cnt1 > 0 ? 128 + cnt1 : cnt0;
        auto col_ok = [&](int n) { return n < cnt0 || (n >= 128 && n < ncol); };
        // this warp's chunks: 32-column chunk ci with ci % kHalves == part
        // (the sets sharing its accumulator block), skipping chunks of stale
        // columns only
        constexpr int kHalves = W2 ? C::kEpiSets / 2 : C::kEpiSets;
        const int part = W2 ? (eset >> 1) : eset;
        auto chunk_ok = [&](int ci) { return !(C::kPairSlots == 2 && 32 * ci >= cnt0 && 32 * ci < 128); };
        auto next_chunk = [&](int ci) {
          while (32 * ci < ncol && !chunk_ok(ci)) ci += kHalves;
          return ci;
        };
        // token and weight of column 32 ci + lane, fetched one chunk ahead
        // (the first before the accumulator is ready)
        int tk_n = 0;
        float wk_n = 0.f;
        auto fetch = [&](int ci) {
          tk_n = 0;
          wk_n = 0.f;
          const int n = 32 * ci + lane;
          if (32 * ci < ncol && col_ok(n)) {
            const int64_t rr = row0 + n;
            tk_n = __ldg(p.row_tok + rr);
            wk_n = __ldg(p.row_w + rr) * sc;
            if constexpr (F8) wk_n = __ldg(p.row_w + rr) * __ldg(p.brs + rr);
          }
        };
        int ci = next_chunk(part);
        fetch(ci);
        if (!wait_acc()) break;
        const uint32_t ta = tq + as * C::kAccCols + blk * N;
        while (32 * ci < ncol) {
          const int c0 = 32 * ci;
          const int tk = tk_n;
          const float wk = wk_n;
          const int cn = next_chunk(ci + kHalves);
          fetch(cn);
          float y[32];
          tc_ld32(ta + c0, y);  // even K tiles (all of them with one issuer)
          if (C::kKSplit && KT > 1) {  // odd K tiles (the second issuer's accumulator)
            float y1[32];
            tc_ld32(ta + N + c0, y1);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) y[j] += y1[j];
          }
          tc_wait_ld();
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = F8 ? y[4 * g + i] * rho : y[4 * g + i];
            // lane r of the group: v[i] = (row r, column 4 g + i) -> (row i, column 4 g + r)
#pragma unroll
            for (int m = 1; m <= 2; m <<= 1) {
              const bool up = (r4 & m) != 0;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (i & m) continue;
                const float got = __shfl_xor_sync(0xffffffffu, up ? v[i] : v[i | m], m);
                if (up) v[i] = got;
                else v[i | m] = got;
              }
            }
            const int src = 4 * g + r4;  // column of this lane's four rows
            const int t = __shfl_sync(0xffffffffu, tk, src);
            const float w = __shfl_sync(0xffffffffu, wk, src);
            if (col_ok(c0 + src)) red_add_v4(p.out_acc + (int64_t)t * p.H + h0, v[0] * w, v[1] * w, v[2] * w, v[3] * w);
          }
          ci = cn;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // (pair: the issuer's barrier is in CTA 0)
        if (PAIR && crank != 0) mbar_arrive_remote(smem_u32(&bar_tempty[as]), 0u);
        else mbar_arrive(smem_u32(&bar_tempty[as]));
      }
      if (++as == C::kAccStages) { as = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  // (pair: CTA 0's MMAs, which read this CTA's shared memory and write its
  // tensor memory, have completed once CTA 0 passes its bar_done wait)
  if constexpr (PAIR) cluster_arrive_wait();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, C::kTmemCols);
    else tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int N, bool GATEUP, bool NV, int OP = kOpFp4, bool PAIR = false, bool GROUPED = false, bool W2 = false,
          bool DPW = false>
cudaError_t launch_gemm_t(const KParams& p, int grid, cudaStream_t s) {
  using C = GemmCfg<N, GATEUP, NV, OP, PAIR, W2>;
  auto k = moe_gemm_kernel<N, GATEUP, NV, OP, PAIR, GROUPED, W2, DPW>;
  static bool attr_set[64] = {};  // once per device and template instance
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  if constexpr (PAIR) {
    // CTA pairs: as many as can be resident at once (a pair needs two SMs
    // of one cluster-capable group), at most grid / 2
    static int max_pairs[64] = {};
    if (dev >= 0 && dev < 64 && max_pairs[dev] == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(C::kThreads);
      cfg.dynamicSmemBytes = C::kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
      if (e != cudaSuccess) return e;
      max_pairs[dev] = n > 0 ? n : 1;
    }
    int pairs = grid / 2;
    if (dev >= 0 && dev < 64 && pairs > max_pairs[dev]) pairs = max_pairs[dev];
    if (pairs < 1) pairs = 1;
    return launch_pdl_cluster(k, dim3(2 * pairs), dim3(C::kThreads), C::kSmem, s, 2u, p);
  }
  return launch_pdl(k, dim3(grid), dim3(C::kThreads), C::kSmem, s, p);
}

}  // namespace fp4moe
