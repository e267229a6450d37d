// Gate/up grouped GEMM instances: SwiGLU epilogue with MXFP4 requantisation
// (or fp32 h for NVFP4).
#include <cstring>

#include "gemm_launch.cuh"

namespace fp4moe {
cudaError_t launch_gateup(const GemmArgs& a, cudaStream_t s) { return launch_grouped<true>(a, s); }
}  // namespace fp4moe
