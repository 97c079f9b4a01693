// cluster_f32.cu -- cluster-per-row kernel instantiated for float storage.
#include "cluster.cuh"

namespace rarn {
template cudaError_t launch_cluster<float, float>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
