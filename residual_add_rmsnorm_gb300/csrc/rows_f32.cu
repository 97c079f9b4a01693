// rows_f32.cu -- register-staged row kernels instantiated for float storage.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows<float, float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
