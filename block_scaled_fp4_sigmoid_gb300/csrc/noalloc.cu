// Router entry point for callers that cannot allocate device memory.
//
// fp4moe_route needs scratch (the split-K partial logits and the per-chunk
// expert counts) in a caller-provided workspace.  Some callers cannot provide
// one: engines that plan every byte of device memory up front and forbid
// allocations afterwards, or code that must not call cudaMalloc because it can
// synchronise the device and stall other streams.  fp4moe_route_noalloc keeps
// that scratch in a file-scope device array instead, so the caller passes only
// inputs and outputs.
//
// The array is fixed in size (FP4MOE_NOALLOC_SCRATCH_BYTES) and every GPU that
// loads this library holds it until the process exits.  All calls share it, so
// calls that overlap on the GPU (different streams, or different host threads
// on one device) race; serialise them.  The array keeps the last call's
// contents; the part that must start at zero (status word, counts) is cleared
// by every call.
//
// Layout of the array: status word int32[16] (padded to 256 bytes), per-chunk
// expert counts int32[ceil(T / 32), E + n_shared] (padded to 256 bytes), then
// the partial logits fp32[n_splits, T, E].  n_splits is fp4moe_route's split
// count when that fits, else the largest smaller split count that does (the
// sum order of the logits then differs from fp4moe_route's).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr size_t kScratchBytes = FP4MOE_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;

static __device__ __align__(256) uint8_t g_route_scratch[kScratchBytes];

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Scratch bytes of one call with n_splits splits.
size_t scratch_bytes(const fp4moe_dims& d, const Layout& L, int n_splits) {
  return kStatusBytes + align256((size_t)L.n_chunks * L.n_exp * 4) + (size_t)n_splits * d.T * d.E * 4;
}

// The split count: fp4moe_route's when it fits, else the largest divisor of
// H / 256 below it that fits; 0 when not even one split fits.
int noalloc_splits(const fp4moe_dims& d, const Layout& L) {
  for (int s = L.ws.n_splits; s >= 1; --s)
    if ((d.H / 256) % s == 0 && scratch_bytes(d, L, s) <= kScratchBytes) return s;
  return 0;
}

// Device address of g_route_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress with the device current, looked up on every call (no
// cached pointer can outlive a context).
fp4moe_status scratch_for_current_device(uint8_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return FP4MOE_ERR_CUDA;
  *out = static_cast<uint8_t*>(p);
  return FP4MOE_OK;
}

}  // namespace
}  // namespace fp4moe

using namespace fp4moe;

extern "C" size_t fp4moe_route_noalloc_scratch_bytes(const fp4moe_dims* dims) {
  if (!dims) return 0;
  Layout L;
  if (!make_layout(*dims, &L)) return 0;
  const int s = noalloc_splits(*dims, L);
  return s ? scratch_bytes(*dims, L, s) : 0;
}

extern "C" fp4moe_status fp4moe_route_noalloc(const fp4moe_dims* dims, const uint16_t* x, const uint16_t* w_router,
                                              const float* bias, int32_t* topk_idx, float* topk_w,
                                              float* logits_out, void* stream) {
  if (!dims || !x || !w_router || !bias || !topk_idx || !topk_w) return FP4MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(*dims, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_router) & 15u))
    return FP4MOE_ERR_INVALID_ARG;
  const fp4moe_dims& d = *dims;
  const int n_splits = noalloc_splits(d, L);
  if (n_splits == 0) return FP4MOE_ERR_WORKSPACE;  // beyond the fixed maximum
  if (fp4moe_status st = check_device()) return st;
  uint8_t* base = nullptr;
  if (fp4moe_status st = scratch_for_current_device(&base)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = reinterpret_cast<int32_t*>(base);
  const size_t counts_bytes = (size_t)L.n_chunks * L.n_exp * 4;
  int32_t* cc = reinterpret_cast<int32_t*>(base + kStatusBytes);
  float* partial = reinterpret_cast<float*>(base + kStatusBytes + align256(counts_bytes));
  // status word and counts (which accumulate atomically) start at zero
  cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes + counts_bytes, s);
  if (e == cudaSuccess) e = launch_router_logits(x, w_router, partial, d.T, d.H, d.E, n_splits, status, s);
  if (e == cudaSuccess)
    e = launch_topk(d, partial, n_splits, bias, topk_idx, topk_w, logits_out, nullptr, cc, L.n_exp, s);
  return cuda_status(e);
}

extern "C" fp4moe_status fp4moe_route_noalloc_status(void* stream, fp4moe_status* st, int64_t* count) {
  if (fp4moe_status c = check_device()) return c;
  uint8_t* base = nullptr;
  if (fp4moe_status c = scratch_for_current_device(&base)) return c;
  int32_t h[kStatusInts];
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP4MOE_ERR_CUDA;
  if (cudaMemcpy(h, base, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FP4MOE_ERR_CUDA;
  if (st) *st = static_cast<fp4moe_status>(h[ST_FIRST]);
  if (count) *count = h[ST_COUNT];
  return FP4MOE_OK;
}
