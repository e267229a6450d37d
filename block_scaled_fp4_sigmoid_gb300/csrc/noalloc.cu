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
// contents; the part that must start at zero is cleared by every call.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr size_t kScratchBytes = FP4MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_route_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
fp4moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return FP4MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FP4MOE_OK;
}

}  // namespace
}  // namespace fp4moe

using namespace fp4moe;

extern "C" fp4moe_status fp4moe_route_noalloc(const fp4moe_dims* dims, const uint16_t* x, const uint16_t* w_router,
                                              const float* bias, int32_t* topk_idx, float* topk_w,
                                              float* logits_out, void* stream) {
  if (!dims || !x || !w_router || !bias || !topk_idx || !topk_w) return FP4MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(*dims, &L)) return FP4MOE_ERR_UNSUPPORTED_SHAPE;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_router) & 15u))
    return FP4MOE_ERR_INVALID_ARG;
  const fp4moe_dims& d = *dims;
  // scratch: partial logits [n_splits, T, E] fp32, then chunk counts [n_chunks, n_exp] int32
  const size_t partial_bytes = (size_t)L.ws.n_splits * d.T * d.E * 4;
  const size_t counts_off = (partial_bytes + 255) / 256 * 256;
  const size_t counts_bytes = (size_t)L.n_chunks * L.n_exp * 4;
  if (counts_off + counts_bytes > kScratchBytes) return FP4MOE_ERR_WORKSPACE;  // beyond the fixed maximum
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4MOE_ERR_DEVICE;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FP4MOE_ERR_DEVICE;
  void* base = nullptr;
  if (fp4moe_status st = scratch_for_current_device(&base)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* partial = static_cast<float*>(base);
  int32_t* cc = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(base) + counts_off);
  cudaError_t e = cudaMemsetAsync(cc, 0, counts_bytes, s);  // counts accumulate atomically
  if (e == cudaSuccess) e = launch_router_logits(x, w_router, partial, d.T, d.H, d.E, L.ws.n_splits, nullptr, s);
  if (e == cudaSuccess)
    e = launch_topk(d, partial, L.ws.n_splits, bias, topk_idx, topk_w, logits_out, cc, L.n_exp, s);
  return e == cudaSuccess ? FP4MOE_OK : FP4MOE_ERR_CUDA;
}
