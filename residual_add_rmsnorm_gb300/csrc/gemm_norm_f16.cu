// gemm_norm_f16.cu -- GEMM + fused residual-add RMSNorm instantiated for __half.
#include "gemm_norm_launch.cuh"

namespace rarn {
template cudaError_t launch_gemm_norm<__half>(const GemmCall &, cudaStream_t);
}  // namespace rarn
