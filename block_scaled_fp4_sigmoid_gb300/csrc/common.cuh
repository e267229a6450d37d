// Shared device helpers of the fp4moe library: status word, bounded waits,
// PTX wrappers for mbarrier / TMA / tcgen05, and the FP4 / FP8 encoders.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fp4moe.h"

namespace fp4moe {

// ---------------------------------------------------------------- status word
// int32[16] at the start of every workspace: [0] first status code recorded,
// [1] number of records, [2] NaN-scale rows, [3] below-floor rows,
// [4] timeouts, [5] where the last timeout happened, [8..9] tickets of the
// kernels whose last CTA finishes a step.
enum { ST_FIRST = 0, ST_COUNT = 1, ST_NAN = 2, ST_INEXACT = 3, ST_TIMEOUT = 4, ST_WHERE = 5,
       ST_TICKET_FRONT = 8, ST_TICKET_DOWN = 9, ST_TICKET_PLAN = 10 };  // [8]-[10]: last-CTA tickets, cleared per call
constexpr int kStatusInts = 16;

__device__ __forceinline__ void record_status(int32_t* st, int code, int which, int n = 1) {
  if (st == nullptr) return;
  atomicCAS(st + ST_FIRST, 0, code);
  atomicAdd(st + ST_COUNT, n);
  atomicAdd(st + which, n);
}

// Wall-clock limit of every device-side wait, in nanoseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start before
// its predecessor finishes; it must call pdl_wait() before touching anything
// the predecessor writes.  pdl_trigger() lets the successor launch early.
// Adds four floats to four consecutive fp32 words (16-byte aligned) as one
// reduction.
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- shared memory / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// kCluster: acquire at cluster scope (arrivals released by the other CTA of
// a pair).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Gives up after
// kWaitLimitNs and returns false; the caller records the timeout and unwinds.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// As mbar_wait with a limit of its own (limit_ns), and giving up as soon as
// *abort is set (another role of the CTA has stopped, so the phase may
// never complete).  Returns false on either; only waits whose arrivals
// depend on other roles use it.  Drains of copies already issued keep
// mbar_wait: those copies always land.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_abortable(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                    const volatile int* abort) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if ((i & 255u) == 0 && (*abort || globaltimer() - t0 > limit_ns)) return false;
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// As tma_load_3d, with an L2 cache policy (from l2_evict_first()).
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                                 int32_t c1, int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// L2 policy for data read once: its lines are the first to be replaced, so
// a stream does not push reused data (activations, other CTAs' tiles) out.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// As bulk_load, with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Scale factors: 32 lanes x 128 bits from shared memory, replicated into the
// four lane quadrants.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <bool kNV>
__device__ __forceinline__ void tc_mma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                           uint32_t sfb, uint32_t accumulate) {
  if constexpr (kNV) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  }
}

// Warp-issued forms: the whole (converged) warp executes the call and
// elect.sync picks the one lane that issues the instruction, so the operands
// are computed warp-uniformly instead of in one divergent lane.
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_cp_sf_elect(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
      : "memory");
}

template <bool kNV>
__device__ __forceinline__ void tc_mma_fp4_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                                 uint32_t sfb, uint32_t accumulate) {
  if constexpr (kNV) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %6, 0;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], q;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %6, 0;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], q;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  }
}

// ---------------------------------------------------------------- CTA pairs
// A cluster of two CTAs on two SMs shares one M = 256 block-scaled MMA
// (tcgen05 .cta_group::2): rank 0 issues it, each CTA supplies half of A
// (its 128 rows) and half of B (N / 2 rows) from the same shared-memory
// offsets, and each CTA's tensor memory holds its own 128 accumulator lanes
// and scale factors at the same addresses.  Every tcgen05 allocation, copy,
// MMA and commit of such a kernel uses .cta_group::2.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_wait() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_barrier_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive (release, cluster scope) on the barrier at the same shared-memory
// offset in CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\tmapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(bar), "r"(rank)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
// Arrives on the barrier at this offset in every CTA of cta_mask once the
// pair MMAs and copies issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair_elect(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
// Scale factors into both CTAs' tensor memory, each from its own shared memory.
__device__ __forceinline__ void tc_cp_sf_pair_elect(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
      : "memory");
}
// MXFP4 (E8M0 per 32) MMA with M = 256 over the CTA pair.
__device__ __forceinline__ void tc_mma_mx_pair_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                                     uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %6, 0;\n\t"
      "@p tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], q;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// E4M3 x E4M3 MMA (kind::f8f6f4, K = 32 per instruction), fp32 accumulate,
// issued by one elected lane of the calling warp.
__device__ __forceinline__ void tc_mma_f8_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, q;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// BF16 x BF16 MMA (kind::f16, K = 16 per instruction), fp32 accumulate,
// issued by one elected lane of the calling warp.
__device__ __forceinline__ void tc_mma_bf16_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (sm_100 family): start address, leading and
// stride byte offsets (in 16-byte units), fixed version bits 46..47 = 1,
// layout type in bits 61..63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// Instruction descriptor of a block-scaled FP4 MMA: E2M1 x E2M1, K-major A and
// B, M = m, N = n, scale type E8M0 (MXFP4) or E4M3 (NVFP4), scale-factor
// byte ids for A and B.
__host__ __device__ constexpr uint32_t idesc_fp4(uint32_t n, bool nv, uint32_t sfa_id, uint32_t sfb_id,
                                                 uint32_t m = 128) {
  return (sfb_id & 3u) << 4        // B scale-factor id
         | 1u << 7                 // A format: E2M1
         | 1u << 10                // B format: E2M1
         | (n >> 3) << 17          // N / 8
         | (nv ? 0u : 1u) << 23    // scale format: 0 = UE4M3, 1 = UE8M0
         | (m >> 4) << 24          // M / 16 (256: a CTA pair)
         | (sfa_id & 3u) << 29;    // A scale-factor id
}

// Instruction descriptor of kind::f16 with fp32 D and bf16 A and B, both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
  return 1u << 4 | 1u << 7 | 1u << 10 | (n >> 3) << 17 | (128u >> 4) << 24;
}

// Instruction descriptor of a dense E4M3 MMA: fp32 D, E4M3 A and B (format
// code 0), both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f8(uint32_t n) {
  return 1u << 4              // D format: fp32
         | 0u << 7            // A format: E4M3
         | 0u << 10           // B format: E4M3
         | (n >> 3) << 17     // N / 8
         | (128u >> 4) << 24; // M / 16
}

// ---------------------------------------------------------------- FP4 / FP8 encoders
// E2M1 codes of eight fp32 values packed into one word, value j in bits
// 4j..4j+3.  The hardware conversion rounds to nearest even on the grid
// 0, .5, 1, 1.5, 2, 3, 4, 6, saturates at +-6 and keeps the sign bit (zero
// included); cvt.rn.satfinite.e2m1x2.f32 puts its first source in the high
// nibble of the byte.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Round-to-nearest-even E4M3 (OCP FN) byte of a non-negative finite value,
// saturating at 448.
__device__ __forceinline__ uint32_t e4m3_pos(float x) {
  if (!(x > 0.f)) return 0u;
  if (x >= 448.f) return 0x7Eu;
  if (x < 0.015625f) {  // below 2^-6: subnormal step 2^-9
    return (uint32_t)__float2int_rn(x * 512.f);  // 8 means 2^-6, i.e. code 0x08
  }
  const uint32_t b = __float_as_uint(x);
  const int e = (int)((b >> 23) & 0xFF) - 127 + 7;  // 1..15
  const uint32_t mant = b & 0x7FFFFFu;
  uint32_t r = (mant + 0x7FFFFu + ((mant >> 20) & 1u)) >> 20;
  uint32_t code = ((uint32_t)e << 3) + r;  // a carry out of r bumps the exponent
  return code > 0x7Eu ? 0x7Eu : code;
}

// Signed E4M3 byte of v / sigma (W8A8 activations): round-to-nearest-even,
// saturating at 448; sigma = 0 gives the signed zero of v.
__device__ __forceinline__ uint32_t fp8_code(float v, float sigma) {
  const uint32_t sign = (__float_as_uint(v) >> 24) & 0x80u;
  return (sigma > 0.f ? e4m3_pos(fabsf(__fdiv_rn(v, sigma))) : 0u) | sign;
}

__device__ __forceinline__ float e4m3_value(uint32_t s) {
  const uint32_t e = (s >> 3) & 15u, m = s & 7u;
  if (e == 0) return (float)m * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((e - 7u + 127u) << 23) | (m << 20));
}

__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  const float v = mag[c & 7u];
  return (c & 8u) ? -v : v;
}

// 2^n as a float for n in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2i(int n) {
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23) : __uint_as_float(0x00400000u);
}

// MXFP4 block exponent e = floor(log2 amax) - 2, clamped to [-127, 127];
// amax = 0 gives -127.
__device__ __forceinline__ int floor_log2_pos(float x) {  // x finite, > 0
  const uint32_t b = __float_as_uint(x);
  const int ef = (int)((b >> 23) & 0xFF);
  return ef ? ef - 127 : -118 - __clz(b & 0x7FFFFFu);  // subnormal: mant * 2^-149
}

__device__ __forceinline__ int mx_block_exp(float amax) {
  if (!(amax > 0.f)) return -127;
  int e = floor_log2_pos(amax) - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Quantises 32 values of one MXFP4 block: 16 packed code bytes and the scale byte.
__device__ __forceinline__ void mx_quant32(const float* v, uint32_t* packed4, uint32_t* scale_byte) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mx_block_exp(amax);
  const float inv = exp2i(-e);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float q[8];  // |v| * inv < 8; inv = 2^-e, so the product is exact above the subnormal range
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = v[8 * w + j] * inv;
    packed4[w] = e2m1x8(q);
  }
  *scale_byte = (uint32_t)(e + 127);
}

// Hardware reciprocal (rcp.approx.ftz: relative error within about one unit
// in the last place; subnormal results flush to zero).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// NVFP4: tensor scale g = amax / 2688 (correctly rounded fp32 division).
__device__ __forceinline__ float nv_global(float amax) { return __fdiv_rn(amax, 2688.0f); }

// Quantises 16 values of one NVFP4 block with tensor scale g: 8 packed code
// bytes (two words) and the E4M3 scale byte.  Every step is one correctly
// rounded fp32 operation: s = E4M3(amax / (6 g)), d = s * g, code = E2M1(v / d).
__device__ __forceinline__ void nv_quant16(const float* v, float g, uint32_t* packed2, uint32_t* scale_byte) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float six_g = __fmul_rn(6.0f, g);
  const uint32_t s = six_g > 0.f ? e4m3_pos(__fdiv_rn(amax, six_g)) : 0u;
  const float d = __fmul_rn(e4m3_value(s), g);
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = v[8 * w + j];
      q[j] = d > 0.f ? __fdiv_rn(x, d) : x * 0.f;
    }
    packed2[w] = e2m1x8(q);
  }
  *scale_byte = s;
}

// ---------------------------------------------------------------- tiled weight layout
// Byte offset of (row r, byte cb) of an FP4 payload in the layout of
// fp4moe_pack_weights: blocks of 128 rows x 128 bytes (one K tile of 256
// values), K tiles innermost, rows counted over all matrices (rows per
// matrix a multiple of 128); ktb = K tiles per row.
// Block (row tile rt, K tile kt) of the tiled layouts sits at slot
// rt * KT + kt.  Gate/up-paired (P = I / 128 > 0, matrices of 2P row tiles:
// gate tiles 0..P-1, up tiles P..2P-1): the gate and up blocks of pair p and
// K tile kt are adjacent, slot ((m * P + p) * KT + kt) * 2 + h (h: 0 gate,
// 1 up), so that one copy fetches both.
__host__ __device__ __forceinline__ int64_t tile_slot(int64_t rt, int64_t kt, int64_t ktiles, int64_t pairs) {
  if (pairs == 0) return rt * ktiles + kt;
  const int64_t m = rt / (2 * pairs), lr = rt - m * 2 * pairs, h = lr / pairs, pp = lr - h * pairs;
  return ((m * pairs + pp) * ktiles + kt) * 2 + h;
}

__host__ __device__ __forceinline__ int64_t w_tiled_offset(int64_t r, int64_t cb, int64_t ktb, int64_t pairs = 0) {
  return (tile_slot(r >> 7, cb >> 7, ktb, pairs) << 14) + ((r & 127) << 7) + (cb & 127);
}

// ---------------------------------------------------------------- tiled scale layout
// For a matrix of `rows` rows and `katoms` groups of four scale blocks
// (padded to whole K tiles), the byte of (row r, block kb) sits at
//   ((r / 128) * katoms + kb / 4) * 512 + 16 * (r % 32) + 4 * ((r / 32) % 4) + kb % 4.
__host__ __device__ __forceinline__ int64_t sf_tiled_offset(int64_t r, int64_t kb, int64_t katoms) {
  return ((r >> 7) * katoms + (kb >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (kb & 3);
}
// The same in the gate/up-paired order (tile_slot): `apk` groups per K tile.
__host__ __device__ __forceinline__ int64_t sf_tiled_offset_gu(int64_t r, int64_t kb, int64_t katoms, int64_t apk,
                                                               int64_t pairs) {
  const int64_t atom = kb >> 2, kt = atom / apk;
  return (tile_slot(r >> 7, kt, katoms / apk, pairs) * apk + (atom - kt * apk)) * 512 + 16 * (r & 31) +
         4 * ((r >> 5) & 3) + (kb & 3);
}

// Scale-block groups per 256-value K tile: MXFP4 8 blocks = 2 groups,
// NVFP4 16 blocks = 4 groups.
__host__ __device__ constexpr int atoms_per_ktile(bool nv) { return nv ? 4 : 2; }

__host__ __device__ inline int64_t katoms_padded(int64_t K, bool nv) {
  const int64_t ktiles = (K + 255) / 256;
  return ktiles * atoms_per_ktile(nv);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;  // NaN
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

}  // namespace fp4moe
