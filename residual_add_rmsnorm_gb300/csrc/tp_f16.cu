// tp_f16.cu -- tensor-parallel form instantiated for __half.
#include "tp_launch.cuh"

namespace rarn {
template cudaError_t tp_blocks_per_sm<__half>(int64_t, int *);
template cudaError_t launch_tp<__half>(const tp::Params &, int, bool, bool, cudaStream_t);
}  // namespace rarn
