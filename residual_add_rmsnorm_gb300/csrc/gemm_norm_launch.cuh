// gemm_norm_launch.cuh -- host side of the GEMM + fused RMSNorm kernel:
// tensor-map encoding (through the driver entry point, so the library needs
// no link-time dependency on the driver library) and the cluster launch.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_norm.cuh"

namespace rarn {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Row-major [rows, cols] 16-bit matrix with row stride ld (elements); box of
// box_rows x bk elements, bk * 2-byte swizzle, out-of-bounds elements read
// as zero.
inline bool encode_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld,
                       int box_rows, int bk, bool bf16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           2, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename T, int BK>
static cudaError_t launch_gemm_bk(const GemmCall &c, cudaStream_t st) {
    using namespace gemm;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap ma, mw, mr, my;
    if (!encode_map(&ma, c.a, c.T, c.K, c.lda, kBM, BK, bf16) ||
        !encode_map(&mw, c.w, c.H, c.K, c.ldw, kMmaN, BK, bf16) ||
        !encode_map(&mr, c.residual, c.T, c.H, c.ldr, kBM, kChunkCols, bf16) ||
        !encode_map(&my, c.y, c.T, c.H, c.ldy, kBM, kChunkCols, bf16))
        return cudaErrorInvalidValue;
    // the epilogue stages the residual / y tile in the operand ring
    if (c.stages * layout(c.stages, c.ns, BK).stage_bytes < (c.ns / kChunkCols) * kChunkBytes)
        return cudaErrorInvalidValue;
    Params p{};
    p.y = c.y;
    p.residual = c.residual;
    p.gamma = c.gamma;
    p.T = c.T;
    p.H = c.H;
    p.K = c.K;
    p.ldr = c.ldr;
    p.ldy = c.ldy;
    p.eps = c.eps;
    p.ns = c.ns;
    p.stages = c.stages;
    p.kblocks = static_cast<int>((c.K + BK - 1) / BK);
    p.watchdog = c.watchdog;
    p.wait_limit_ns = kWaitLimitNs;
    const int C = static_cast<int>(c.H / c.ns);
    const int smem = layout(c.stages, c.ns, BK).total;
    auto kernel = k_gemm_norm<T, BK>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (C > 8 &&
        (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
            cudaSuccess)
        return e;
    const int64_t mblocks = (c.T + kBM - 1) / kBM;
    return launch_kernel(kernel, dim3(static_cast<unsigned>(mblocks * C)), dim3(kThreads),
                         static_cast<size_t>(smem), st, c.pdl, C, ma, mw, mr, my, p);
}

template <typename T>
cudaError_t launch_gemm_norm(const GemmCall &c, cudaStream_t st) {
    if (c.T == 0) return cudaSuccess;
    const cudaError_t e = c.bk == 64 ? launch_gemm_bk<T, 64>(c, st) : launch_gemm_bk<T, 32>(c, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int BK>
static int max_clusters_bk(int cluster, int ns, int stages) {
    using namespace gemm;
    auto kernel = k_gemm_norm<T, BK>;
    const int smem = layout(stages, ns, BK).total;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return 0;
    if (cluster > 8 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <typename T>
int gemm_norm_max_clusters(int cluster, int ns, int stages, int bk) {
    return bk == 64 ? max_clusters_bk<T, 64>(cluster, ns, stages)
                    : max_clusters_bk<T, 32>(cluster, ns, stages);
}

}  // namespace rarn
