// Router (logits, sigmoid + bias grouped top-k) and the token permutation
// (expert histogram, prefix sum over experts, stable scatter into the padded
// slot layout).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

namespace {

// ---------------------------------------------------------------- router logits, few tokens
// One warp per (expert, K split): streams the expert's router row once and
// forms the dot products with all T <= 16 token rows.
template <int TMAX>
__device__ __forceinline__ void gemv_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                                          float* __restrict__ partial, int T, int H, int E, int n_splits, int warp,
                                          int lane) {
  const int e = warp % E, sp = warp / E;
  const int kc = H / n_splits;  // multiple of 256
  const int k0 = sp * kc;
  float acc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
  const uint16_t* wrow = wr + (int64_t)e * H;
#pragma unroll 4
  for (int k = k0 + lane * 8; k < k0 + kc; k += 256) {
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wrow + k));
    const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
    float wf[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wf[2 * j] = __uint_as_float(wu[j] << 16);
      wf[2 * j + 1] = __uint_as_float(wu[j] & 0xFFFF0000u);
    }
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)t * H + k));
        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[t] = fmaf(__uint_as_float(xu[j] << 16), wf[2 * j], acc[t]);
          acc[t] = fmaf(__uint_as_float(xu[j] & 0xFFFF0000u), wf[2 * j + 1], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && t < T) partial[((int64_t)sp * T + t) * E + e] = v;
  }
}

template <int TMAX>
__global__ void router_gemv_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                                   float* __restrict__ partial, int T, int H, int E, int n_splits) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (warp >= E * n_splits) return;
  gemv_warp<TMAX>(x, wr, partial, T, H, E, n_splits, warp, threadIdx.x & 31);
}

// ---------------------------------------------------------------- sigmoid + bias grouped top-k
// One warp per token.  Scores live in shared memory (E <= 512).
// Selection for one token from its scores in shared memory: sv = sigmoid
// scores, cv = scores + bias (overwritten: unselected groups become -inf).
// Group selection, then top-k over the corrected scores.  Lane j < k returns
// the j-th chosen expert in *idx and its routing weight in *w (ties to the
// lower group and expert index).
__device__ __forceinline__ void topk_select(const float* sv, float* cv, int E, int k, int n_group, int topk_group,
                                            float scaling, int renorm, int lane, int* idx, float* w);

// Routes token t with one warp: sums the split-K partial logits, sigmoid,
// bias, then topk_select.  sv / cv: E floats of shared memory for this warp.
__device__ __forceinline__ void topk_token(const float* __restrict__ partial, int n_splits,
                                           const float* __restrict__ bias, int T, int t, int E, int k,
                                           int n_group, int topk_group, float scaling, int renorm,
                                           float* __restrict__ logits_out, float* __restrict__ scores_out,
                                           float* sv, float* cv, int lane, int* idx, float* w) {
  // E <= 512: at most 16 logits per lane; issue each split's loads together
  float lv[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) lv[q] = 0.f;
#pragma unroll 4
  for (int sp = 0; sp < n_splits; ++sp) {  // unrolled: several splits' loads in flight
    const float* src = partial + ((int64_t)sp * T + t) * E;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (lane + 32 * q < E) lv[q] += src[lane + 32 * q];
  }
  float bv16[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) bv16[q] = lane + 32 * q < E ? bias[lane + 32 * q] : 0.f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = lane + 32 * q;
    if (e < E) {
      if (logits_out) logits_out[(int64_t)t * E + e] = lv[q];
      const float s = 1.0f / (1.0f + expf(-lv[q]));
      if (scores_out) scores_out[(int64_t)t * E + e] = s;
      sv[e] = s;
      cv[e] = s + bv16[q];
    }
  }
  __syncwarp();
  topk_select(sv, cv, E, k, n_group, topk_group, scaling, renorm, lane, idx, w);
}

__device__ __forceinline__ void topk_select(const float* sv, float* cv, int E, int k, int n_group, int topk_group,
                                            float scaling, int renorm, int lane, int* idx, float* w) {
  // group selection: group score = sum of the two largest corrected scores
  uint32_t group_ok = 0xffffffffu;
  if (n_group > 1) {
    const int gsz = E / n_group;
    float gs = -INFINITY;
    if (lane < n_group) {
      float a = -INFINITY, b = -INFINITY;
      for (int i = 0; i < gsz; ++i) {
        const float v = cv[lane * gsz + i];
        if (v > a) { b = a; a = v; } else if (v > b) { b = v; }
      }
      gs = a + b;
    }
    group_ok = 0;
    for (int r = 0; r < topk_group; ++r) {
      float bv = (lane < n_group && !((group_ok >> lane) & 1u)) ? gs : -INFINITY;
      int bi = lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      group_ok |= 1u << bi;
    }
    for (int e = lane; e < E; e += 32)
      if (!((group_ok >> (e / gsz)) & 1u)) cv[e] = -INFINITY;
    __syncwarp();
  }
  // top-k over corrected scores, ties to the lower expert index; each lane
  // keeps its (at most 16) candidates in registers (absent or NaN: -inf,
  // never chosen).  Per round: the lane's best by a pairwise tournament (ties
  // keep the lower index), then the warp's largest score (order-preserving
  // integer key, one warp reduction) and the lowest index holding it (a
  // second reduction).
  float cr[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float v = lane + 32 * q < E ? cv[lane + 32 * q] : -INFINITY;
    cr[q] = v > -INFINITY ? v : -INFINITY;
  }
  int my_idx = -1;
  float my_s = 0.f;
  for (int j = 0; j < k; ++j) {
    float v8[8], v4[4], v2[2];
    int q8[8], q4[4], q2[2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool r = cr[2 * i + 1] > cr[2 * i];
      v8[i] = r ? cr[2 * i + 1] : cr[2 * i];
      q8[i] = r ? 2 * i + 1 : 2 * i;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool r = v8[2 * i + 1] > v8[2 * i];
      v4[i] = r ? v8[2 * i + 1] : v8[2 * i];
      q4[i] = r ? q8[2 * i + 1] : q8[2 * i];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const bool r = v4[2 * i + 1] > v4[2 * i];
      v2[i] = r ? v4[2 * i + 1] : v4[2 * i];
      q2[i] = r ? q4[2 * i + 1] : q4[2 * i];
    }
    const bool r = v2[1] > v2[0];
    const float bv = r ? v2[1] : v2[0];
    const int li = bv > -INFINITY ? lane + 32 * (r ? q2[1] : q2[0]) : 0x7fffffff;
    const uint32_t bits = __float_as_uint(bv);
    const uint32_t key = li != 0x7fffffff ? ((bits & 0x80000000u) ? ~bits : (bits | 0x80000000u)) : 0u;
    const uint32_t m = __reduce_max_sync(0xffffffffu, key);
    int bi = __reduce_min_sync(0xffffffffu, key == m ? li : 0x7fffffff);
    if (bi >= E) bi = 0;  // only reachable without k valid candidates (out of contract): keep the index in range
    if (lane == j) my_idx = bi;
    if ((bi & 31) == lane) {  // the owner drops the winner from its candidates
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (lane + 32 * q == bi) cr[q] = -INFINITY;
    }
  }
  if (lane < k) my_s = sv[my_idx];
  float tot = 0.f;
  for (int j = 0; j < k; ++j) tot += __shfl_sync(0xffffffffu, my_s, j);
  *idx = my_idx;
  *w = renorm ? my_s / tot * scaling : my_s * scaling;
}

constexpr int kTopkWarps = 4;

__global__ void topk_kernel(const float* __restrict__ partial, int n_splits, const float* __restrict__ bias,
                            int T, int E, int k, int n_group, int topk_group, float scaling, int renorm,
                            int32_t* __restrict__ idx_out, float* __restrict__ w_out, float* __restrict__ logits_out,
                            float* __restrict__ scores_out, int32_t* __restrict__ chunk_counts, int n_exp) {
  __shared__ float s_s[kTopkWarps][512];
  __shared__ float s_c[kTopkWarps][512];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + wib;
  if (t >= T) return;
  int my_idx;
  float my_w;
  topk_token(partial, n_splits, bias, T, t, E, k, n_group, topk_group, scaling, renorm, logits_out, scores_out,
             s_s[wib], s_c[wib], lane, &my_idx, &my_w);
  if (lane < k) {
    idx_out[(int64_t)t * k + lane] = my_idx;
    w_out[(int64_t)t * k + lane] = my_w;
    atomicAdd(&chunk_counts[(t / kChunkTokens) * n_exp + my_idx], 1);
  }
}

// ---------------------------------------------------------------- plan
// One warp per expert: exclusive prefix of the expert's per-chunk counts (in
// place: they become the chunk bases of the stable scatter), the expert's
// total.  Lane l takes a contiguous run of chunks, so one warp scan orders
// them.  The CTA that finishes last (a ticket; no CTA waits for another)
// turns the totals into tiles, 128-row slots and the unit prefixes of both
// GEMMs by a block scan.
constexpr int kPlanWarps = 8;

__global__ void __launch_bounds__(32 * kPlanWarps) plan_kernel(int32_t* chunk_counts, int n_chunks, int n_exp, int E,
                                                                int T, int n_tile, int dn_pair, int gu_mtiles,
                                                                int dn_mtiles,
                                                                int32_t* expert_count, int32_t* expert_slot,
                                                                int32_t* gu_start, int32_t* dn_start, Plan* plan,
                                                                int32_t* ticket) {
  __shared__ int s_last;
  __shared__ long long s_wsum[kPlanWarps];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int e = blockIdx.x * kPlanWarps + wib;
  if (e < n_exp) {
    const int per = (n_chunks + 31) / 32;
    const int c0 = lane * per, c1 = min(n_chunks, c0 + per);
    auto count = [&](int c) {  // the shared expert takes every token of the chunk
      return e >= E ? min(kChunkTokens, T - c * kChunkTokens) : chunk_counts[(int64_t)c * n_exp + e];
    };
    int sum = 0;
#pragma unroll 8
    for (int c = c0; c < c1; ++c) sum += count(c);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int c = c0; c < c1; ++c) {
      const int v = count(c);
      chunk_counts[(int64_t)c * n_exp + e] = run;
      run += v;
    }
    if (lane == 31) expert_count[e] = incl;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA: exclusive scans over the experts of their tiles (slots) and
  // of their down tiles (dn_pair slots each), both in one 64-bit scan (tiles
  // low, down tiles high); thread j owns experts 3j .. 3j + 2 (n_exp <= 520
  // < 3 * 256)
  constexpr int kT = 32 * kPlanWarps;
  int tl[3], td[3];
  long long my = 0;
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int ee = threadIdx.x * 3 + q;
    const int c = ee < n_exp ? __ldcg(expert_count + ee) : 0;
    tl[q] = (c + n_tile - 1) / n_tile;
    td[q] = (c + n_tile * dn_pair - 1) / (n_tile * dn_pair);
    my += (long long)tl[q] + ((long long)td[q] << 32);
  }
  long long incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[wib] = incl;
  __syncthreads();
  long long b = incl - my;
  for (int w2 = 0; w2 < wib; ++w2) b += s_wsum[w2];
  int base = (int)(b & 0xffffffffll), base_d = (int)(b >> 32);
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int ee = threadIdx.x * 3 + q;
    if (ee < n_exp) {
      expert_slot[ee] = base;
      gu_start[ee] = base * gu_mtiles;
      dn_start[ee] = base_d * dn_mtiles;
    }
    base += tl[q];
    base_d += td[q];
  }
  if (threadIdx.x == kT - 1) {
    const int total = base, total_d = base_d;  // the last thread's running sums cover every expert
    gu_start[n_exp] = total * gu_mtiles;
    dn_start[n_exp] = total_d * dn_mtiles;
    plan->n_exp = n_exp;
    plan->gu_units = total * gu_mtiles;
    plan->dn_units = total_d * dn_mtiles;
    plan->slots = total;
  }
}

// ---------------------------------------------------------------- stable scatter
// One warp per chunk of 256 tokens.  Routes are visited in (token, slot)
// order; __match_any_sync groups the routes of one expert inside each 32-route
// step, so the position of a route is the chunk base + earlier routes of the
// same expert in this chunk.
constexpr int kScatterWarps = 2;

__global__ void scatter_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w,
                               const int32_t* __restrict__ chunk_base, int T, int k, int E, int n_exp, int n_chunks,
                               int n_tile, const int32_t* __restrict__ expert_slot, int32_t* __restrict__ route_row,
                               int32_t* __restrict__ row_tok, float* __restrict__ row_w, int32_t* __restrict__ row_e) {
  __shared__ int32_t s_cnt[kScatterWarps][520];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * kScatterWarps + wib;
  if (c >= n_chunks) return;
  int32_t* cnt = s_cnt[wib];
  for (int e = lane; e < n_exp; e += 32) cnt[e] = 0;
  __syncwarp();
  const int rpt = k + (n_exp - E);
  const int t0 = c * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  const int64_t r0 = (int64_t)t0 * k, r1 = (int64_t)t1 * k;
  for (int64_t base = r0; base < r1; base += 32) {
    const int64_t r = base + lane;
    const bool valid = r < r1;
    const int e = valid ? idx[r] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int prior = valid ? cnt[e] : 0;
    __syncwarp();
    if (valid && rank == 0) cnt[e] = prior + __popc(peers);
    __syncwarp();
    if (valid) {
      const int pos = chunk_base[(int64_t)c * n_exp + e] + prior + rank;
      const int64_t row = (int64_t)(expert_slot[e] + pos / n_tile) * kSlotRows + pos % n_tile;
      const int64_t t = r / k;
      const int j = (int)(r - t * k);
      route_row[t * rpt + j] = (int32_t)row;
      row_tok[row] = (int32_t)t;
      row_w[row] = w[r];
      row_e[row] = e;
    }
  }
  for (int s = E; s < n_exp; ++s) {  // shared experts: every token, in order
    for (int t = t0 + lane; t < t1; t += 32) {
      const int pos = t;
      const int64_t row = (int64_t)(expert_slot[s] + pos / n_tile) * kSlotRows + pos % n_tile;
      route_row[(int64_t)t * rpt + k + (s - E)] = (int32_t)row;
      row_tok[row] = t;
      row_w[row] = 1.0f;
      row_e[row] = s;
    }
  }
}

// ---------------------------------------------------------------- fused front end for few tokens
// Phase A: CTA (group of 16 experts, K split sp) stages the tokens' x
// columns of its split in shared memory, and each warp forms the split's
// partial logits of two experts (every lane issues all its router-weight
// loads in one batch).  The n_splits CTAs of a group form one thread-block
// cluster; after a cluster barrier the rank-0 CTA reads the others' partials
// from their shared memory, sums them in split order, and stores the sigmoid
// scores.  All CTAs zero the combine buffer and quantise x to MXFP4 once per
// token (token t is row t of the layout; the gate/up GEMM reads every token
// and keeps the routed ones).  The rank-0 CTA that finishes last (a ticket
// counter; no CTA ever waits for another outside its cluster) runs phase B:
// top-k per token, expert counts, token masks and stable positions (each
// token routes to an expert at most once, so a route's position is the
// number of earlier tokens routed to the same expert), the plan, and the
// route -> row map.
constexpr int kFrontThreads = 256;
constexpr int kFrontWarps = kFrontThreads / 32;
constexpr int kFrontExperts = 2 * kFrontWarps;  // experts per CTA: two per warp
static_assert(kFrontExperts * kFrontMaxT == kFrontThreads, "one rank-0 thread per (expert, token)");

// fp32 at a shared-memory address of CTA `rank` of this cluster
__device__ __forceinline__ float ld_dsmem(const float* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Partial logits of experts e0 and e0 + 1 over this CTA's K split (nk <= NK
// pieces of 256 columns, x staged in xs).  Lane t returns token t's sums.
template <int TMAX, int NK>
__device__ __forceinline__ float2 front_gemv(const FrontArgs& a, uint16_t* xs, int sp, int e0, int lane) {
  const int T = a.d.T, H = a.d.H, E = a.d.E;
  const int kc = H / a.n_splits, k0 = sp * kc, nk = kc / 256;
  float acc0[TMAX], acc1[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) acc0[t] = acc1[t] = 0.f;
  // rows past E load a valid row and are never stored
  const uint16_t* w0 = a.wr + (int64_t)min(e0, E - 1) * H + k0 + 8 * lane;
  const uint16_t* w1 = a.wr + (int64_t)min(e0 + 1, E - 1) * H + k0 + 8 * lane;
  uint4 wv0[NK], wv1[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i)
    if (i < nk) {
      wv0[i] = __ldg(reinterpret_cast<const uint4*>(w0 + 256 * i));
      wv1[i] = __ldg(reinterpret_cast<const uint4*>(w1 + 256 * i));
    }
  const int per_row = kc / 8;  // 16-byte pieces of one token's columns
  for (int v = threadIdx.x; v < T * per_row; v += kFrontThreads) {
    const int t = v / per_row, c = v - t * per_row;
    reinterpret_cast<uint4*>(xs + (int64_t)t * kc)[c] = __ldg(reinterpret_cast<const uint4*>(a.x + (int64_t)t * H + k0) + c);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    if (i >= nk) break;
    const uint32_t u0[4] = {wv0[i].x, wv0[i].y, wv0[i].z, wv0[i].w};
    const uint32_t u1[4] = {wv1[i].x, wv1[i].y, wv1[i].z, wv1[i].w};
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
      if (t < T) {
        const uint4 xv = reinterpret_cast<const uint4*>(xs + (int64_t)t * kc + 256 * i)[lane];
        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float xa = __uint_as_float(xu[j] << 16), xb = __uint_as_float(xu[j] & 0xFFFF0000u);
          acc0[t] = fmaf(xa, __uint_as_float(u0[j] << 16), acc0[t]);
          acc0[t] = fmaf(xb, __uint_as_float(u0[j] & 0xFFFF0000u), acc0[t]);
          acc1[t] = fmaf(xa, __uint_as_float(u1[j] << 16), acc1[t]);
          acc1[t] = fmaf(xb, __uint_as_float(u1[j] & 0xFFFF0000u), acc1[t]);
        }
      }
    }
  }
  float2 mine = make_float2(0.f, 0.f);
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    float v0 = acc0[t], v1 = acc1[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v0 += __shfl_xor_sync(0xffffffffu, v0, o);
      v1 += __shfl_xor_sync(0xffffffffu, v1, o);
    }
    if (lane == t) mine = make_float2(v0, v1);
  }
  return mine;
}

template <int TMAX>
__device__ __forceinline__ float2 front_gemv_any(const FrontArgs& a, uint16_t* xs, int sp, int e0, int lane) {
  const int nk = a.d.H / a.n_splits / 256;
  if (nk <= 2) return front_gemv<TMAX, 2>(a, xs, sp, e0, lane) ;
  if (nk <= 4) return front_gemv<TMAX, 4>(a, xs, sp, e0, lane);
  return front_gemv<TMAX, kFrontMaxKc / 256>(a, xs, sp, e0, lane);
}

__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Prefetch of a 16-byte aligned global range into L2 with a cache policy (a
// hint: nothing waits for it); size a multiple of 16.
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(policy)
               : "memory");
}

__global__ void __launch_bounds__(kFrontThreads, 2) decode_front_kernel(FrontArgs a) {
  extern __shared__ __align__(16) uint16_t front_xs[];  // [T][kc] bf16 of this CTA's split
  __shared__ __align__(16) float s_sc[kFrontWarps][2][512];  // scores of the token a warp routes
  __shared__ float s_part[kFrontExperts][kFrontMaxT];        // this split's partial logits
  __shared__ int s_last;
  __shared__ int32_t s_idx[kFrontMaxT][16];
  __shared__ float s_w[kFrontMaxT][16];
  __shared__ int32_t s_count[520];
  __shared__ int32_t s_slot[520];
  __shared__ uint32_t s_mask[520];
  __shared__ int32_t s_wsum[kFrontWarps];
  const fp4moe_dims& d = a.d;
  const int T = d.T, H = d.H, E = d.E, k = d.top_k;
  const int tid = threadIdx.x, lane = tid & 31, wib = tid >> 5;

  pdl_trigger();  // the next kernel may launch and wait for this one
  // ---- phase A
  const int sp = (int)cluster_ctarank();  // the cluster is one expert group, rank = K split
  const int e0 = (blockIdx.x / a.n_splits) * kFrontExperts + 2 * wib;  // this warp: experts e0, e0 + 1
  const float2 part = T <= 8 ? front_gemv_any<8>(a, front_xs, sp, e0, lane)
                             : front_gemv_any<kFrontMaxT>(a, front_xs, sp, e0, lane);
  if (lane < T) {
    s_part[2 * wib][lane] = part.x;
    s_part[2 * wib + 1][lane] = part.y;
  }
  cluster_arrive_wait();  // every split's partials are in its CTA's shared memory
  if (sp == 0) {  // thread (expert slot, token)
    const int j = tid / kFrontMaxT, t = tid % kFrontMaxT, e = (blockIdx.x / a.n_splits) * kFrontExperts + j;
    if (e < E && t < T) {
      // every split's partial in flight at once, then summed in split order
      float v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) v[r] = r < a.n_splits ? ld_dsmem(&s_part[j][t], (uint32_t)r) : 0.f;
      float l = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < a.n_splits) l += v[r];
      const float sc = 1.0f / (1.0f + expf(-l));
      a.partial[(int64_t)t * E + e] = sc;  // sigmoid scores [T, E]
      if (a.logits_dbg) a.logits_dbg[(int64_t)t * E + e] = l;
      if (a.scores_dbg) a.scores_dbg[(int64_t)t * E + e] = sc;
    }
  }
  cluster_arrive_wait();  // the other CTAs' shared memory stays valid until rank 0 has read it
  // Off the critical path (the ranks other than 0 are done; with one split
  // the rank-0 CTAs do it): zero the combine buffer and quantise x to MXFP4
  // once per token, token t in row t of the layout.  The next kernel reads
  // both only after this grid has completed.
  if (sp != 0 || a.n_splits == 1) {
    const int64_t helpers = a.n_splits == 1 ? gridDim.x : gridDim.x - gridDim.x / a.n_splits;
    const int64_t hid = a.n_splits == 1 ? blockIdx.x : blockIdx.x - blockIdx.x / a.n_splits - 1;
    const int64_t hthr = hid * kFrontThreads + tid, hn = helpers * kFrontThreads;
    // DRAM is idle until routing ends: pull this CTA's slice of the shared
    // expert's weights into L2 (evict-last, so that they outlast the routed
    // weight stream that follows) for the two expert GEMMs.
    if (tid == 0) {
      const uint64_t pol = l2_evict_last();
      for (int r = 0; r < 4; ++r) {
        const int64_t n = a.l2_pf_bytes[r];
        if (!a.l2_pf[r] || n <= 0) continue;
        const int64_t slice = ((n + helpers - 1) / helpers + 255) / 256 * 256;
        const int64_t lo = hid * slice, hi = lo + slice < n ? lo + slice : n;
        for (int64_t o = lo; o < hi; o += 32768)
          l2_prefetch(a.l2_pf[r] + o, (uint32_t)(hi - o < 32768 ? hi - o : 32768), pol);
      }
    }
    for (int64_t i = hthr; i < (int64_t)T * H / 4; i += hn)
      reinterpret_cast<float4*>(a.out_acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int per_row = H >> 5;
    const int64_t katoms = katoms_padded(H, false);
    for (int64_t i = hthr; i < (int64_t)T * per_row; i += hn) {
      const int t = (int)(i / per_row), b = (int)(i - (int64_t)t * per_row);
      const uint4* src = reinterpret_cast<const uint4*>(a.x + (int64_t)t * H + 32 * b);
      float v[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = __ldg(src + q);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          v[8 * q + 2 * r] = __uint_as_float(ws[r] << 16);
          v[8 * q + 2 * r + 1] = __uint_as_float(ws[r] & 0xFFFF0000u);
        }
      }
      uint32_t pk[4], sb;
      mx_quant32(v, pk, &sb);
      *reinterpret_cast<uint4*>(a.xq + (int64_t)t * (H >> 1) + 16 * b) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      a.xsf[sf_tiled_offset(t, b, katoms)] = (uint8_t)sb;
    }
    if (sp != 0) return;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.ticket, 1) == (int)(gridDim.x / a.n_splits) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- phase B (one CTA)
  const int n_exp = a.n_exp, rpt = k + d.n_shared;
  for (int t = wib; t < T; t += kFrontWarps) {
    float* sv = s_sc[wib][0];
    float* cv = s_sc[wib][1];
    float sg[16], bv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int ee = lane + 32 * q;
      sg[q] = ee < E ? __ldcg(a.partial + (int64_t)t * E + ee) : 0.f;
      bv[q] = ee < E ? __ldg(a.bias + ee) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int ee = lane + 32 * q;
      if (ee < E) {
        sv[ee] = sg[q];
        cv[ee] = sg[q] + bv[q];
      }
    }
    __syncwarp();
    int id;
    float wt;
    topk_select(sv, cv, E, k, d.n_group, d.topk_group, d.routed_scaling, d.renormalize, lane, &id, &wt);
    if (lane < k) {
      s_idx[t][lane] = id;
      s_w[t][lane] = wt;
      a.idx[t * k + lane] = id;
      a.w[t * k + lane] = wt;
    }
    __syncwarp();
  }
  for (int e = tid; e < n_exp; e += blockDim.x) {
    s_count[e] = e >= E ? T : 0;
    s_mask[e] = e >= E ? (1u << T) - 1u : 0u;  // T <= 16
  }
  __syncthreads();
  for (int r = tid; r < T * k; r += blockDim.x) {
    const int e = s_idx[r / k][r % k];
    atomicAdd(&s_count[e], 1);
    atomicOr(&s_mask[e], 1u << (r / k));  // token mask of the expert
  }
  __syncthreads();
  for (int e = tid; e < n_exp; e += blockDim.x) a.tok_mask[e] = s_mask[e];
  // plan: exclusive scan of tiles over experts; thread j owns experts 3j..3j+2
  const int gm = d.I / 128, dm = a.dn_mtiles;
  int tl[3], my = 0;
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int e = 3 * tid + q;
    tl[q] = e < n_exp ? (s_count[e] + a.n_tile - 1) / a.n_tile : 0;
    my += tl[q];
  }
  int incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[wib] = incl;
  __syncthreads();
  int base = incl - my;
  for (int w2 = 0; w2 < wib; ++w2) base += s_wsum[w2];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int e = 3 * tid + q;
    if (e < n_exp) {
      s_slot[e] = base;
      a.expert_count[e] = s_count[e];
      a.expert_slot[e] = base;
      a.gu_start[e] = base * gm;
      a.dn_start[e] = base * dm;
    }
    base += tl[q];
  }
  if (tid == 0) {
    int total = 0;
    for (int w2 = 0; w2 < kFrontWarps; ++w2) total += s_wsum[w2];
    a.gu_start[n_exp] = total * gm;
    a.dn_start[n_exp] = total * dm;
    a.plan->n_exp = n_exp;
    a.plan->gu_units = total * gm;
    a.plan->dn_units = total * dm;
    a.plan->slots = total;
  }
  __syncthreads();
  for (int r = tid; r < T * rpt; r += blockDim.x) {
    const int t = r / rpt, j = r - t * rpt;
    int e, pos;
    float wt;
    if (j < k) {
      e = s_idx[t][j];
      wt = s_w[t][j];
      pos = __popc(s_mask[e] & ((1u << t) - 1u));  // earlier tokens routed to e
    } else {
      e = E + (j - k);
      wt = 1.0f;
      pos = t;
    }
    const int row = (s_slot[e] + pos / a.n_tile) * kSlotRows + pos % a.n_tile;
    a.route_row[r] = row;
    a.row_tok[row] = t;
    a.row_w[row] = wt;
    a.row_e[row] = e;
  }
}

// ---------------------------------------------------------------- dense linear plan
// The dense linear runs the down GEMM's mainloop with one "expert" that every
// token routes to once with weight 1: token t sits at row (t / n_tile) * 128 +
// t % n_tile of the padded layout.  Also zeroes the fp32 output accumulator.
__global__ void linear_plan_kernel(int T, int n_tile, int dn_pair, int m_tiles, int32_t* __restrict__ count,
                                   int32_t* __restrict__ slot, int32_t* __restrict__ dn_start, Plan* __restrict__ plan,
                                   int32_t* __restrict__ route_row, int32_t* __restrict__ row_tok,
                                   float* __restrict__ row_w, float4* __restrict__ acc, int64_t acc_n4) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, nthr = (int64_t)gridDim.x * blockDim.x;
  const int tiles = (T + n_tile - 1) / n_tile;
  const int tiles_d = (T + n_tile * dn_pair - 1) / (n_tile * dn_pair);
  if (tid == 0) {
    count[0] = T;
    slot[0] = 0;
    dn_start[0] = 0;
    dn_start[1] = tiles_d * m_tiles;
    plan->n_exp = 1;
    plan->gu_units = 0;
    plan->dn_units = tiles_d * m_tiles;
    plan->slots = tiles;
  }
  for (int64_t t = tid; t < T; t += nthr) {
    const int row = (int)(t / n_tile) * kSlotRows + (int)(t % n_tile);
    route_row[t] = row;
    row_tok[row] = (int32_t)t;
    row_w[row] = 1.0f;
  }
  for (int64_t i = tid; i < acc_n4; i += nthr) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* wr, float* partial, int T, int H, int E,
                                 int n_splits, int32_t* status, cudaStream_t s) {
  if (T <= 16) {
    const int warps = E * n_splits;
    const int threads = 256;
    const unsigned blocks = (unsigned)((warps * 32 + threads - 1) / threads);
    if (T <= 8) router_gemv_kernel<8><<<blocks, threads, 0, s>>>(x, wr, partial, T, H, E, n_splits);
    else router_gemv_kernel<16><<<blocks, threads, 0, s>>>(x, wr, partial, T, H, E, n_splits);
    return cudaGetLastError();
  }
  return launch_router_tc(x, wr, partial, T, H, E, n_splits, status, s);
}

cudaError_t launch_topk(const fp4moe_dims& d, const float* partial, int n_splits, const float* bias, int32_t* idx,
                        float* w, float* logits_out, float* scores_out, int32_t* chunk_counts, int n_exp,
                        cudaStream_t s) {
  const unsigned blocks = (unsigned)((d.T + kTopkWarps - 1) / kTopkWarps);
  topk_kernel<<<blocks, 32 * kTopkWarps, 0, s>>>(partial, n_splits, bias, d.T, d.E, d.top_k, d.n_group,
                                                 d.topk_group, d.routed_scaling, d.renormalize, idx, w, logits_out,
                                                 scores_out, chunk_counts, n_exp);
  return cudaGetLastError();
}

cudaError_t launch_plan(const fp4moe_dims& d, int32_t* chunk_counts, int n_chunks, int n_exp, int n_tile, int dn_pair,
                        int dn_mtiles, int32_t* expert_count, int32_t* expert_slot, int32_t* gu_start,
                        int32_t* dn_start, Plan* plan, int32_t* ticket, cudaStream_t s) {
  const unsigned blocks = (unsigned)((n_exp + kPlanWarps - 1) / kPlanWarps);
  plan_kernel<<<blocks, 32 * kPlanWarps, 0, s>>>(chunk_counts, n_chunks, n_exp, d.E, d.T, n_tile, dn_pair, d.I / 128,
                                                 dn_mtiles, expert_count, expert_slot, gu_start, dn_start, plan,
                                                 ticket);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const fp4moe_dims& d, const int32_t* idx, const float* w, const int32_t* chunk_counts,
                           int n_chunks, int n_exp, int n_tile, const int32_t* expert_slot, int32_t* route_row,
                           int32_t* row_tok, float* row_w, int32_t* row_e, cudaStream_t s) {
  const unsigned blocks = (unsigned)((n_chunks + kScatterWarps - 1) / kScatterWarps);
  scatter_kernel<<<blocks, 32 * kScatterWarps, 0, s>>>(idx, w, chunk_counts, d.T, d.top_k, d.E, n_exp, n_chunks,
                                                        n_tile, expert_slot, route_row, row_tok, row_w, row_e);
  return cudaGetLastError();
}

cudaError_t launch_decode_front(const FrontArgs& a, cudaStream_t s) {
  const int kc = a.d.H / a.n_splits;
  if (a.d.T > kFrontMaxT || kc > kFrontMaxKc || kc % 256 != 0 || a.n_splits > 8) return cudaErrorInvalidValue;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_front_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFrontMaxT * kFrontMaxKc * 2);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((a.d.E + kFrontExperts - 1) / kFrontExperts) * a.n_splits));
  cfg.blockDim = dim3(kFrontThreads);
  cfg.dynamicSmemBytes = (size_t)a.d.T * kc * 2;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // one cluster per expert group: its K splits
  attr[0].val.clusterDim.x = (unsigned)a.n_splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_front_kernel, a);
}

cudaError_t launch_linear_plan(int T, int n_tile, int dn_pair, int m_tiles, int32_t* count, int32_t* slot, int32_t* dn_start,
                               Plan* plan, int32_t* route_row, int32_t* row_tok, float* row_w, float* acc,
                               int64_t acc_n, cudaStream_t s) {
  linear_plan_kernel<<<4 * 152, 256, 0, s>>>(T, n_tile, dn_pair, m_tiles, count, slot, dn_start, plan, route_row, row_tok,
                                            row_w, reinterpret_cast<float4*>(acc), acc_n / 4);
  return cudaGetLastError();
}

}  // namespace fp4moe
