// Router logits for many tokens on the tensor cores (tcgen05, bf16 inputs,
// fp32 accumulation in tensor memory).
//
// The router stays in high precision ("Serving NVFP4 models on AMD Instinct
// MI355 accelerators", Layer Selection): l[t, e] = sum_h x[t, h] * Wr[e, h]
// with bf16 x and Wr.  One CTA computes a tile of 128 tokens x N experts
// (N <= 256) over one K split, written as fp32 to partial[split][t][e]; the
// top-k kernel sums the splits in split order.
//
// Warp roles (192 threads): warp 0 TMA producer (x tile 128 rows x 64
// columns, Wr tile N rows x 64 columns, both K-major with the 128-byte
// swizzle), warp 1 tensor-memory owner and single-thread issuer of
// tcgen05.mma.kind::f16 (four K = 16 steps per 64-column stage), warps 2-5
// epilogue (one tensor-memory lane quadrant each).  Every wait is bounded; a
// timeout records FP4MOE_ERR_TIMEOUT in the status word, drains in-flight
// copies and MMAs, frees tensor memory and returns.
#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {

namespace {

constexpr int kRtStages = 4;
constexpr int kRtMaxN = 256;
constexpr int kRtABytes = 128 * 128;        // 128 tokens x 64 bf16
constexpr int kRtBBytes = kRtMaxN * 128;    // up to 256 experts x 64 bf16
constexpr int kRtStage = kRtABytes + kRtBBytes;
constexpr int kRtSmem = kRtStages * kRtStage + 1024;  // + 17 KB static: within 227 KB

struct RtParams {
  CUtensorMap tmx, tmw;
  float* partial;
  int32_t* status;  // nullable: a timeout is then only an early exit
  int T, E, N, kc, mtiles, ntiles;
};

__device__ __forceinline__ void tc_mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint64_t desc_sw128_rt(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }

__global__ void __launch_bounds__(192, 1) router_tc_kernel(const __grid_constant__ RtParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_full[kRtStages], bar_empty[kRtStages];
  __shared__ __align__(8) uint64_t bar_tfull, bar_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float epi[4][32][33];  // per epilogue warp: 32 tokens x 32 experts

  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the expert tiles of one token tile are adjacent CTAs, so they run at
  // the same time and x is read from DRAM once, not once per expert tile
  // (measured: the 16k-token router 0.122 -> 0.111 ms)
  const int nt = blockIdx.x % p.ntiles, mt = blockIdx.x / p.ntiles;
  const int k0 = blockIdx.y * p.kc, ksteps = p.kc / 64;
  const uint32_t bbytes = (uint32_t)p.N * 128u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_tfull), 1);
    mbar_init(smem_u32(&bar_done), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), kRtMaxN);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tmx);
    prefetch_tmap(&p.tmw);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_v = &abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      for (int ks = 0; ks < ksteps && !*abort_v; ++ks) {
        if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1u)) {
          *abort_v = 1;
          if (p.status) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
          break;
        }
        const uint32_t fb = smem_u32(&bar_full[stage]);
        const uint32_t base = sbase + stage * kRtStage;
        mbar_arrive_expect_tx(fb, kRtABytes + bbytes);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        const int kb = (k0 + 64 * ks) * 2;  // byte column of the stage
        tma_load_2d(base, &p.tmx, fb, kb, mt * 128);
        tma_load_2d(base + kRtABytes, &p.tmw, fb, kb, nt * p.N);
        if (++stage == kRtStages) { stage = 0; phase ^= 1u; }
      }
      for (int s = 0; s < kRtStages; ++s)  // every armed stage lands before the CTA exits
        if ((armed >> s) & 1u) (void)mbar_wait(smem_u32(&bar_full[s]), (armed_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16((uint32_t)p.N);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int ks = 0; ks < ksteps && ok && !*abort_v; ++ks) {
        if (!mbar_wait(smem_u32(&bar_full[stage]), phase)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = sbase + stage * kRtStage;
#pragma unroll
        for (int j = 0; j < 4; ++j)  // K = 16 bf16 = 32 bytes of the swizzled row per step
          tc_mma_bf16(tmem, desc_sw128_rt(base + 32 * j), desc_sw128_rt(base + kRtABytes + 32 * j), idesc,
                      (ks | j) ? 1u : 0u);
        tc_commit(smem_u32(&bar_empty[stage]));
        if (++stage == kRtStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) {
        *abort_v = 1;
        if (p.status) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
      }
      tc_commit(smem_u32(&bar_tfull));  // the accumulator is final (or abandoned)
      tc_commit(smem_u32(&bar_done));
      (void)mbar_wait(smem_u32(&bar_done), 0);  // every issued MMA has finished
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const bool ok = mbar_wait(smem_u32(&bar_tfull), 0);
    tc_fence_after();
    if (!ok) {
      *abort_v = 1;
      if (lane == 0 && p.status) record_status(p.status, FP4MOE_ERR_TIMEOUT, ST_TIMEOUT);
    } else if (!*abort_v) {
      // lane l holds token t0 + l (its tensor-memory lane); each 32 x 32 block
      // goes through shared memory so that a store writes 32 consecutive
      // experts of one token
      const int t0 = mt * 128 + 32 * q;
      const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
      float(*tile)[33] = epi[warp - 2];
      const int ncol = min(p.N, p.E - nt * p.N);
      float* dst0 = p.partial + ((int64_t)blockIdx.y * p.T + t0) * p.E + (int64_t)nt * p.N;
      for (int c0 = 0; c0 < p.N; c0 += 32) {
        float v[32];
        tc_ld32(tq + c0, v);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) tile[lane][j] = v[j];
        __syncwarp();
        if (c0 + lane < ncol)
          for (int r = 0; r < 32 && t0 + r < p.T; ++r) dst0[(int64_t)r * p.E + c0 + lane] = tile[r][lane];
        __syncwarp();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kRtMaxN);
  }
}

}  // namespace

// Tile width over the experts: the fewest tiles of at most 256, split evenly,
// rounded up to a multiple of 16 (the MMA's N step).
int router_tc_n(int E) {
  const int ntiles = (E + kRtMaxN - 1) / kRtMaxN;
  const int per = (E + ntiles - 1) / ntiles;
  return (per + 15) / 16 * 16;
}

cudaError_t launch_router_tc(const uint16_t* x, const uint16_t* wr, float* partial, int T, int H, int E, int n_splits,
                             int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  RtParams p;
  memset(&p, 0, sizeof(p));
  const int N = router_tc_n(E);
  {
    const uint64_t dims[2] = {(uint64_t)H * 2, (uint64_t)T};  // bytes of a row, rows
    const uint64_t strides[1] = {(uint64_t)H * 2};
    const uint32_t box[2] = {128, 128};
    if (!encode_tmap_u8(&p.tmx, x, 2, dims, strides, box, true)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)H * 2, (uint64_t)E};
    const uint64_t strides[1] = {(uint64_t)H * 2};
    const uint32_t box[2] = {128, (uint32_t)N};
    if (!encode_tmap_u8(&p.tmw, wr, 2, dims, strides, box, true)) return cudaErrorInvalidValue;
  }
  p.partial = partial;
  p.status = status;
  p.T = T;
  p.E = E;
  p.N = N;
  p.kc = H / n_splits;  // a multiple of 256
  p.mtiles = (T + 127) / 128;
  p.ntiles = (E + N - 1) / N;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const dim3 grid((unsigned)(p.mtiles * p.ntiles), (unsigned)n_splits);
  router_tc_kernel<<<grid, 192, kRtSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace fp4moe
