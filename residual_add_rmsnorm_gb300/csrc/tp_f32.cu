// tp_f32.cu -- tensor-parallel form instantiated for float.
#include "tp_launch.cuh"

namespace rarn {
template cudaError_t tp_blocks_per_sm<float>(int64_t, int *);
template cudaError_t launch_tp<float>(const tp::Params &, int, bool, bool, cudaStream_t);
}  // namespace rarn
