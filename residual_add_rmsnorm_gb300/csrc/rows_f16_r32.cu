// rows_f16_r32.cu -- register-staged row kernels for __half inputs with a binary32 residual.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows<__half, float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
