// rows_bf16_q8.cu -- register-staged row kernels with an 8-bit output, instantiated
// for __nv_bfloat16 inputs.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows_q8<__nv_bfloat16>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
