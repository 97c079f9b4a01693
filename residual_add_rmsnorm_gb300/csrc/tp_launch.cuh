// tp_launch.cuh -- host launcher of the tensor-parallel kernel, included once
// per storage type by tp_{bf16,f16,f32}.cu.
#pragma once

#include "tp.cuh"

namespace rarn {

namespace tp {
template <typename T>
using TpKernel = void (*)(Params);

template <typename T>
TpKernel<T> tp_kernel(int64_t H, int &block) {
    int vpt = 0;
    tp_shape(H / DT<T>::EPV, vpt, block);
    return vpt == 1 ? k_tp_rows<T, 1> : vpt == 2 ? k_tp_rows<T, 2> : k_tp_rows<T, 4>;
}
}  // namespace tp

template <typename T>
cudaError_t tp_blocks_per_sm(int64_t H, int *blocks) {
    int block = 0;
    const tp::TpKernel<T> k = tp::tp_kernel<T>(H, block);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k, block, 0);
}

template <typename T>
cudaError_t launch_tp(const tp::Params &p, int grid, bool cooperative, bool pdl,
                      cudaStream_t st) {
    int block = 0;
    const tp::TpKernel<T> k = tp::tp_kernel<T>(p.H, block);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    int n = 0;
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    } else if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rarn
