// tp_bf16.cu -- tensor-parallel form instantiated for __nv_bfloat16.
#include "tp_launch.cuh"

namespace rarn {
template cudaError_t tp_blocks_per_sm<__nv_bfloat16>(int64_t, int *);
template cudaError_t launch_tp<__nv_bfloat16>(const tp::Params &, int, bool, bool, cudaStream_t);
}  // namespace rarn
