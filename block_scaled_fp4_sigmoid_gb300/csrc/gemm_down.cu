// Down grouped GEMM instances: routing-weighted combine in the epilogue.
#include <cstring>

#include "gemm_launch.cuh"

namespace fp4moe {
cudaError_t launch_down(const GemmArgs& a, cudaStream_t s) { return launch_grouped<false>(a, s); }
}  // namespace fp4moe
