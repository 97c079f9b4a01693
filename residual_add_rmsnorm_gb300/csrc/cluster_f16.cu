// cluster_f16.cu -- cluster-per-row kernel instantiated for __half storage.
#include "cluster.cuh"

namespace rarn {
template cudaError_t launch_cluster<__half, __half>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
