// stream_f16.cu -- TMA-fed persistent kernel instantiated for __half storage.
#include "stream.cuh"

namespace rarn {
template cudaError_t launch_stream<__half>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
