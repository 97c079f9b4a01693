// stream_bf16.cu -- TMA-fed persistent kernel instantiated for __nv_bfloat16 storage.
#include "stream.cuh"

namespace rarn {
template cudaError_t launch_stream<__nv_bfloat16>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
