// rows_f16.cu -- register-staged row kernels instantiated for __half storage.
#include "rows.cuh"

namespace rarn {
template cudaError_t launch_rows<__half, __half>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
