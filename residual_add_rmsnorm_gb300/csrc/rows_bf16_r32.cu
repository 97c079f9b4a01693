// rows_bf16_r32.cu -- register-staged row kernels for __nv_bfloat16 inputs with a binary32 residual.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows<__nv_bfloat16, float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
