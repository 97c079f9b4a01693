// q8in_f16.cu -- reduce over 8-bit partials instantiated for __half.
#include "q8in.cuh"

namespace rarn {
template cudaError_t launch_q8in<__half>(const q8in::Params &,
                                                const q8in::KernelChoice &, int, bool,
                                                cudaStream_t);
}  // namespace rarn
