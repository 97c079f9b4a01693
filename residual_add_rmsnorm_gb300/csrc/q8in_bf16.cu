// q8in_bf16.cu -- reduce over 8-bit partials instantiated for __nv_bfloat16.
#include "q8in.cuh"

namespace rarn {
template cudaError_t launch_q8in<__nv_bfloat16>(const q8in::Params &,
                                                const q8in::KernelChoice &, int, bool,
                                                cudaStream_t);
}  // namespace rarn
