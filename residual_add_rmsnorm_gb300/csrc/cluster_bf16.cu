// cluster_bf16.cu -- cluster-per-row kernel instantiated for __nv_bfloat16 storage.
#include "cluster.cuh"

namespace rarn {
template cudaError_t launch_cluster<__nv_bfloat16, __nv_bfloat16>(const Problem &, const Plan &, cudaStream_t);
}  // namespace rarn
