// cluster_f16_r32.cu -- cluster-per-row kernel for __half inputs with a binary32 residual.
#include "cluster.cuh"

namespace rarn {
template cudaError_t launch_cluster<__half, float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
