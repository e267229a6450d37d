// Device-side draws of the seeded synthetic inputs; the same definitions as
// synth/__init__.py (SplitMix64 finaliser over key + index * golden ratio).
// The host passes the stream key; these kernels hold no arithmetic of the
// MoE layer.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint64_t key, uint64_t i) { return mix(key + i * kGolden); }

__global__ void bytes_kernel(uint64_t key, uint64_t start_word, uint64_t n_words, uint64_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n_words; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = word(key, start_word + i);
}

__global__ void e8m0_kernel(uint64_t key_blk, uint64_t key_row, uint64_t row0, uint64_t rows, int nblk, int lo,
                            int span, uint8_t* out) {
  const uint64_t n = rows * (uint64_t)nblk;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t r = i / nblk;
    const int base = lo + (int)((word(key_row, row0 + r) >> 32) % (uint64_t)span);
    const uint64_t top = word(key_blk, row0 * nblk + i) >> 32;
    const int off = top < 3006477107ull ? 0 : (top < 4080218931ull ? -1 : -2);
    out[i] = (uint8_t)(127 + base + off);
  }
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t start, uint64_t n, double c, uint16_t* out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t w = word(key, start + i);
    const int64_t s = (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) + (int64_t)((w >> 32) & 0xFFFF) +
                      (int64_t)(w >> 48) - 131070;
    const float f = __double2float_rn(__dmul_rn((double)s, c));
    uint32_t u = __float_as_uint(f);
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    out[i] = (uint16_t)u;
  }
}

unsigned grid_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  return (unsigned)(b > 65535 * 8 ? 65535 * 8 : (b == 0 ? 1 : b));
}

}  // namespace

extern "C" {

// Words start_word .. start_word + n_words - 1 of a stream, as raw uint64
// (viewed as bytes: the uniform byte stream).
int synth_words(uint64_t key, uint64_t start_word, uint64_t n_words, void* out, void* stream) {
  if (n_words == 0) return 0;
  bytes_kernel<<<grid_for(n_words), 256, 0, (cudaStream_t)stream>>>(key, start_word, n_words, (uint64_t*)out);
  return (int)cudaGetLastError();
}

int synth_e8m0(uint64_t key_blk, uint64_t key_row, uint64_t row0, uint64_t rows, int nblk, int lo, int hi, void* out,
               void* stream) {
  if (rows == 0) return 0;
  e8m0_kernel<<<grid_for(rows * nblk), 256, 0, (cudaStream_t)stream>>>(key_blk, key_row, row0, rows, nblk, lo,
                                                                       hi - lo + 1, (uint8_t*)out);
  return (int)cudaGetLastError();
}

int synth_normal_bf16(uint64_t key, uint64_t start, uint64_t n, double c, void* out, void* stream) {
  if (n == 0) return 0;
  normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(key, start, n, c, (uint16_t*)out);
  return (int)cudaGetLastError();
}

}  // extern "C"
