// rows_f32_q8.cu -- register-staged row kernels with an 8-bit output, instantiated
// for float inputs.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows_q8<float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
