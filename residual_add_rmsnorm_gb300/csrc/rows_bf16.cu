// rows_bf16.cu -- register-staged row kernels instantiated for __nv_bfloat16 storage.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows<__nv_bfloat16, __nv_bfloat16>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
