// cluster_bf16_r32.cu -- cluster-per-row kernel for __nv_bfloat16 inputs with a binary32 residual.
#include "cluster.cuh"

namespace rarn {
template cudaError_t launch_cluster<__nv_bfloat16, float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
