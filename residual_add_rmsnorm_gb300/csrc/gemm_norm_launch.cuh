// gemm_norm_launch.cuh -- host side of the GEMM + fused RMSNorm kernels:
// tensor-map encoding (through the driver entry point, so the library needs
// no link-time dependency on the driver library) and the two launches.
#pragma once

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gemm_norm.cuh"

namespace rarn {

// K slabs (of 64 elements) per ring stage of the pair kernel: two (three
// 64 KB stages, eight MMAs per stage and per handshake) measured faster than
// one (six 32 KB stages): T = K = H = 4096 98.4 -> 96.6 us, [8192, 4096,
// 4096] 171.6 -> 168.4, [16384, 5120, 5120] 502.9 -> 496.5.
constexpr int kPairSlabsPerStage = 2;

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

// Clusters of two CTAs of the pair kernel that can be resident at once on the
// current device (SM pairs that share a cluster domain), once per device.
template <typename T>
static int pair_clusters(int num_sms) {
    constexpr int kDevs = 64;
    static std::atomic<int> cache[kDevs];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return num_sms / 2;
    int n = cache[dev].load();
    if (n > 0) return n;
    auto kernel = gemm::k_gemm_res_pair<T, 64, false, kPairSlabsPerStage>;
    constexpr int smem = gemm::PairLayout<64, kPairSlabsPerStage>::total;
    n = num_sms / 2;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
        cfg.blockDim = dim3(gemm::kWsThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int q = 0;
        if (cudaOccupancyMaxActiveClusters(&q, kernel, &cfg) == cudaSuccess && q > 0) n = q;
    }
    (void)cudaGetLastError();
    cache[dev].store(n);
    return n;
}

template <typename T, int BK>
static cudaError_t launch_gemm_bk(const GemmCall &c, cudaStream_t st) {
    using namespace gemm;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap ma, mw, mr;
    if (!encode_map(&ma, c.a, c.T, c.K, c.lda, kBM, BK, bf16) ||
        !encode_map(&mw, c.w, c.H, c.K, c.ldw, kMmaN, BK, bf16) ||
        !encode_map(&mr, c.residual, c.T, c.H, c.ldr, kBM, kChunkCols, bf16))
        return cudaErrorInvalidValue;
    // the non-persistent kernel's epilogue stages the residual tile in the ring
    if (!c.persistent &&
        c.stages * layout(c.stages, c.ns, BK).stage_bytes < (c.ns / kChunkCols) * kChunkBytes)
        return cudaErrorInvalidValue;
    Params p{};
    p.ss = c.workspace;
    p.T = c.T;
    p.H = c.H;
    p.K = c.K;
    p.ns = c.ns;
    p.C = static_cast<int>(c.H / c.ns);
    p.stages = c.stages;
    p.kblocks = static_cast<int>((c.K + BK - 1) / BK);
    p.watchdog = c.watchdog;
    p.wait_limit_ns = c.wait_limit_ns;
    p.stall_fill = c.stall_fill;
    const int64_t mblocks = (c.T + kBM - 1) / kBM;
    const bool pair_path = BK == 64 && c.persistent && c.ns == 256 && c.pair;
    const bool single_path = BK == 64 && c.persistent && c.ns == 256 && !c.pair;
    PairSchedule ps;
    if (pair_path) {
        ps = pair_schedule(c.T, p.C, pair_clusters<T>(c.num_sms), c.tail_split);
        p.full_items = ps.full_items;
        p.items = ps.items;
    }
    // y in the persistent kernels' epilogue: the row-block counters follow the
    // partial sums in the workspace and start each call at zero
    const bool fused = c.fuse_norm && ((pair_path && ps.fuse_ok) ||
                                       (single_path && single_fuse_ok(c.T, p.C, c.num_sms)));
    p.counters = nullptr;
    if (fused) {
        p.counters = reinterpret_cast<unsigned int *>(c.workspace + gemm_counters_offset(c.T, c.H));
        p.y = c.y;
        p.ldy = c.ldy;
        p.gamma = c.gamma;
        p.eps = c.eps;
        const cudaError_t ez = launch_kernel(k_zero_counters, dim3(1), dim3(256), 0, st, c.pdl, 1,
                                             p.counters, mblocks);
        if (ez != cudaSuccess) return ez;
    }
    cudaError_t e = cudaErrorInvalidValue;
    bool launched = false;
    // the persistent kernels' epilogue moves whole 32-byte sectors when every
    // residual row starts on one
    const bool wide = (reinterpret_cast<uintptr_t>(c.residual) & 31u) == 0 && c.ldr % 16 == 0 &&
                      (reinterpret_cast<uintptr_t>(c.y) & 31u) == 0 && c.ldy % 16 == 0;
    if constexpr (BK == 64) {  // the persistent kernels take 128-byte K slabs only
        if (pair_path) {
            // each CTA of a pair stages half of an item's W rows: 128 of a
            // whole tile's 256, 64 of a half tile's 128
            CUtensorMap mw2, mw4;
            if (!encode_map(&mw2, c.w, c.H, c.K, c.ldw, kMmaN / 2, BK, bf16) ||
                !encode_map(&mw4, c.w, c.H, c.K, c.ldw, kMmaN / 4, BK, bf16))
                return cudaErrorInvalidValue;
            const int64_t grid = 2 * ps.walkers;
            auto kernel = wide ? k_gemm_res_pair<T, BK, true, kPairSlabsPerStage>
                               : k_gemm_res_pair<T, BK, false, kPairSlabsPerStage>;
            constexpr int smem = PairLayout<BK, kPairSlabsPerStage>::total;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e == cudaSuccess)
                e = launch_kernel(kernel, dim3(static_cast<unsigned>(grid)), dim3(kWsThreads),
                                  static_cast<size_t>(smem), st, c.pdl, 2, ma, mw2, mw4,
                                  c.residual, c.ldr, p);
            launched = true;
        } else if (single_path) {
            const int64_t grid = std::min<int64_t>(mblocks * p.C, c.num_sms);
            auto kernel = wide ? k_gemm_res_ws<T, 256, BK, true> : k_gemm_res_ws<T, 256, BK, false>;
            constexpr int smem = WsLayout<256, BK>::total;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e == cudaSuccess)
                e = launch_kernel(kernel, dim3(static_cast<unsigned>(grid)), dim3(kWsThreads),
                                  static_cast<size_t>(smem), st, c.pdl, 1, ma, mw, c.residual,
                                  c.ldr, p);
            launched = true;
        }
    }
    if (!launched) {
        const int smem = layout(c.stages, c.ns, BK).total;
        auto kernel = k_gemm_res<T, BK>;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = launch_kernel(kernel, dim3(static_cast<unsigned>(mblocks * p.C)), dim3(kThreads),
                              static_cast<size_t>(smem), st, c.pdl, 1, ma, mw, mr, p);
    }
    if (e != cudaSuccess) return e;
    if (fused) return cudaSuccess;

    NormParams q{};
    q.y = c.y;
    q.h = c.residual;
    q.gamma = c.gamma;
    q.ss = c.workspace;
    q.T = c.T;
    q.H = c.H;
    q.ldh = c.ldr;
    q.ldy = c.ldy;
    q.C = (pair_path || single_path) ? 2 * p.C : p.C;  // 128-column slots, or tiles
    q.eps = c.eps;
    const int64_t slices = (c.H / DT<T>::EPV + 32 * kNormVPT - 1) / (32 * kNormVPT);
    const int64_t warps = c.T * slices;
    const int64_t ctas = std::min<int64_t>((warps + kNormThreads / 32 - 1) / (kNormThreads / 32),
                                           (int64_t)c.num_sms * 8);
    return launch_kernel(k_norm_ss<T>, dim3(static_cast<unsigned>(ctas)), dim3(kNormThreads), 0, st,
                         c.pdl, 1, q);
}

// The split-K sum and norm with registers for at most SMAX splits' partials:
// k_splitk_norm_cluster (a cluster of CTAs per row) for few wide rows, else
// k_splitk_norm (a CTA per row).
template <typename T, int SMAX>
static cudaError_t launch_splitk_norm(const gemm::NormParams &q, const GemmCall &c, int nv,
                                      int used, cudaStream_t st) {
    using namespace gemm;
    const dim3 g2(static_cast<unsigned>(c.T));
    const float *part = static_cast<const float *>(c.part);
    // a cluster of CTAs per row for up to 8 rows of at least 4096 columns,
    // or 128 of at least 8192 (measured, µs, split K + norm against a CTA per
    // row: K = H = 4096 T = 1 8.1 -> 7.3, T = 8 8.2 -> 7.8, T = 16 8.2 ->
    // 8.2-8.5, T = 64 11.2 -> 11.1, T = 256 15.5 -> 17.9; K = H = 8192 T = 1
    // 30.1 -> 27.0, T = 16 30.7 -> 27.7, T = 64 33.3 -> 32.1, T = 128 37.5
    // -> 36.1; T = 1, H = 2048, K = 8192 8.7 -> 9.1)
    if ((c.T <= 8 && c.H >= 4096) || (c.T <= 128 && c.H >= 8192)) {
        const int per = nv / kSplitNormCS;
        return launch_kernel(k_splitk_norm_cluster<T, SMAX>,
                             dim3(static_cast<unsigned>(c.T * kSplitNormCS)),
                             dim3(static_cast<unsigned>((per + 31) / 32 * 32)), 0, st, c.pdl,
                             kSplitNormCS, q, part, used, c.residual);
    }
    if (nv <= 256)
        return launch_kernel(k_splitk_norm<T, 1, SMAX>, g2, dim3((nv + 31) / 32 * 32), 0, st,
                             c.pdl, 1, q, part, used, c.residual);
    if (nv <= 512)
        return launch_kernel(k_splitk_norm<T, 2, SMAX>, g2, dim3(256), 0, st, c.pdl, 1, q, part,
                             used, c.residual);
    return launch_kernel(k_splitk_norm<T, 4, SMAX>, g2, dim3(256), 0, st, c.pdl, 1, q, part,
                         used, c.residual);
}

// Split K (few row blocks): M x C x splits CTAs write binary32 partial products, then a
// CTA (or a cluster of CTAs) per row sums them in split order, adds the residual and
// normalises.
template <typename T>
static cudaError_t launch_gemm_splitk(const GemmCall &c, cudaStream_t st) {
    using namespace gemm;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap ma, mw;
    if (!encode_map(&ma, c.a, c.T, c.K, c.lda, c.T < kBM ? (int)((c.T + 7) / 8 * 8) : kBM, 64, bf16) ||
        !encode_map(&mw, c.w, c.H, c.K, c.ldw, kMmaN, 64, bf16))
        return cudaErrorInvalidValue;
    Params p{};
    p.T = c.T;
    p.H = c.H;
    p.K = c.K;
    p.ns = kMmaN;
    p.C = static_cast<int>(c.H / kMmaN);
    p.stages = 4;
    // with one row block, each fill brings only the rows up to T (in 8-row
    // units of the 128-byte swizzle; the MMA rows past them are never
    // written out): T = 1 moves 1 KB of A per fill instead of 16
    p.a_rows = c.T < kBM ? (int)((c.T + 7) / 8 * 8) : kBM;
    p.kblocks = static_cast<int>((c.K + 63) / 64);
    p.watchdog = c.watchdog;
    p.wait_limit_ns = c.wait_limit_ns;
    p.stall_fill = c.stall_fill;
    p.part = c.part;
    p.kb_per_split = (p.kblocks + c.splitk - 1) / c.splitk;
    // splits that hold K slabs (ceil(kblocks / per split) <= splitk)
    const int used = (p.kblocks + p.kb_per_split - 1) / p.kb_per_split;
    p.splits = used;
    auto kernel = k_gemm_splitk<T>;
    constexpr int smem = layout(4, kMmaN, 64).total;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = launch_kernel(kernel,
                          dim3(static_cast<unsigned>(p.C * ((c.T + kBM - 1) / kBM) * used)),
                          dim3(kThreads),
                          static_cast<size_t>(smem), st, c.pdl, 1, ma, mw, p);
    if (e != cudaSuccess) return e;
    NormParams q{};
    q.y = c.y;
    q.h = c.residual;
    q.gamma = c.gamma;
    q.T = c.T;
    q.H = c.H;
    q.ldh = c.ldr;
    q.ldy = c.ldy;
    q.eps = c.eps;
    const int nv = static_cast<int>(c.H / 8);
    if (used <= 2) return launch_splitk_norm<T, 2>(q, c, nv, used, st);
    if (used <= 4) return launch_splitk_norm<T, 4>(q, c, nv, used, st);
    return launch_splitk_norm<T, kGemmMaxSplitK>(q, c, nv, used, st);
}

template <typename T>
cudaError_t launch_gemm_norm(const GemmCall &c, cudaStream_t st) {
    if (c.T == 0) return cudaSuccess;
    if (c.splitk >= 2) {
        const cudaError_t e = launch_gemm_splitk<T>(c, st);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const cudaError_t e = c.bk == 64 ? launch_gemm_bk<T, 64>(c, st) : launch_gemm_bk<T, 32>(c, st);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rarn
