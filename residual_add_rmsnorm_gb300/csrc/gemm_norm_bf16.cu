// gemm_norm_bf16.cu -- GEMM + fused residual-add RMSNorm instantiated for __nv_bfloat16.
#include "gemm_norm_launch.cuh"

namespace rarn {
template cudaError_t launch_gemm_norm<__nv_bfloat16>(const GemmCall &, cudaStream_t);
}  // namespace rarn
