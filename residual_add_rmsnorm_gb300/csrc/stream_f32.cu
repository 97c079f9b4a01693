// stream_f32.cu -- TMA-fed persistent kernel instantiated for float storage.
#include "stream.cuh"

namespace rarn {
template cudaError_t launch_stream<float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
