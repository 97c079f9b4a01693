// plan.h -- kernel plan (which kernel, launch shape) and the per-dtype
// launchers the C ABI dispatches to.  Host-side declarations only.
#pragma once

#include <algorithm>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace rarn {

enum Kind : int {
    KIND_NONE = 0,
    KIND_WARP = 1,      // one warp per row, several rows per CTA, row in registers
    KIND_CTA = 2,       // one CTA per row, row in registers
    KIND_TWO_PASS = 3,  // one CTA per row; the normalise pass re-reads the row
    KIND_STREAM = 4,    // persistent CTAs fed by TMA bulk copies (shared-memory row)
    KIND_CLUSTER = 5,   // a cluster of CTAs per row, DSMEM sum of squares
};

struct Plan {
    int kind = KIND_NONE;
    bool vec = false;    // 16-byte packs (true) or single elements (false)
    int per_thread = 0;  // packs (vec) or elements (scalar) each thread holds
    int block = 0;       // threads per CTA
    int grid = 0;        // CTAs
    int smem = 0;        // dynamic shared memory per CTA, bytes
    int cluster = 1;     // CTAs per cluster
    int stages = 0;      // pipeline depth (stream kernel)
    int chunk = 0;       // bytes per stream per pipeline stage (stream kernel)
    int groups = 1;      // consumer groups (stream kernel)
    bool prefetch_gamma = false;  // CTA register kernel keeps gamma in registers
    bool pdl = false;    // programmatic dependent launch
    bool pipe = false;   // CTA register kernel loads the next row before finishing this one
};

// Register budget of the register-staged row kernels.  A thread holding P
// 16-byte packs of the row keeps, per pack: the load buffers of the streams
// loaded together (4 registers each; a binary32 residual with 16-bit inputs
// takes rn = 2 words per pack), the binary32 accumulators (EPV), the staged
// row (4 * rn) and, if gamma is held in registers, gamma (4); about 32 more
// for addresses and loop state.  Single-element kernels hold per element one
// value per stream buffer, the residual, the accumulator and the row copy,
// plus its address arithmetic (6 registers measured).  The CTA size a kernel is compiled
// for follows from 64 K registers per SM (and at most 255 per thread); 0 means
// the combination is not built.
__host__ __device__ constexpr int rows_loads_together(int op, int rn) {
    return op == 2 ? (rn == 1 ? 4 : 4 + rn) : op == 1 ? 1 + rn : 1;
}

__host__ __device__ constexpr int rows_regs_vec(int P, int epv, int op, bool gamma_regs,
                                                int rn = 1) {
    return P * (4 * rows_loads_together(op, rn) + epv + 4 * rn + (gamma_regs ? 4 : 0)) + 32;
}

__host__ __device__ constexpr int rows_regs_scalar(int NE, int op) {
    return NE * (rows_loads_together(op, 1) + 6) + 32;
}

__host__ __device__ constexpr int rows_max_block(int regs) {
    return regs <= 64 ? 1024 : regs <= 128 ? 512 : regs <= 256 ? 256 : 0;
}

// Shape of the TMA-fed persistent kernel (stream.cuh), shared with the planner.
namespace stream {
constexpr int kConsumerWarps = 8;                // per consumer group
constexpr int kConsumers = kConsumerWarps * 32;  // threads per group
constexpr int kPackBytes = 16;
constexpr int kMaxStages = 32;
constexpr int kMaxGroups = 2;
constexpr int kMaxPacksPerThread = 4;            // per chunk
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned int kWatchConsumer = 1u, kWatchProducer = 2u;

__host__ __device__ constexpr int threads(int groups) { return 32 + groups * kConsumers; }
// Bytes of one stream's chunk when each consumer thread takes `ppt` packs.
__host__ __device__ constexpr int chunk_bytes(int ppt) { return kConsumers * ppt * kPackBytes; }

// Dynamic shared memory layout (all offsets 128-byte aligned), per consumer
// group g < G its own ring of `stages` stages of NS chunks:
//   [g * stages * NS * chunk, ...)   group g's stage ring
//   G x row copy (H * sizeof(T) bytes each)
//   control: full[G * stages], empty[G * stages] mbarriers (G * stages <=
//            kMaxStages), red[G][2][kConsumerWarps] floats, abort word
struct Layout {
    int stages, ns, row_bytes, groups, chunk;
    int ring_stride, row_off, row_stride, ctl_off, total;
};

__host__ __device__ inline int align128(int v) { return (v + 127) & ~127; }

__host__ __device__ inline Layout layout(int stages, int ns, int row_bytes, int groups,
                                         int chunk) {
    Layout L;
    L.stages = stages;
    L.ns = ns;
    L.row_bytes = row_bytes;
    L.groups = groups;
    L.chunk = chunk;
    L.ring_stride = stages * ns * chunk;
    L.row_off = align128(groups * L.ring_stride);
    L.row_stride = align128(row_bytes);
    L.ctl_off = L.row_off + groups * L.row_stride;
    L.total = L.ctl_off + 2 * kMaxStages * 8 + groups * 2 * kConsumerWarps * 4 + 16;
    return L;
}

}  // namespace stream

// Per-storage-type launchers.  TR is the residual's type: T, or binary32 with
// a 16-bit T (register and cluster kernels only).
template <typename T, typename TR>
cudaError_t launch_rows(const Problem &p, const Plan &plan, cudaStream_t stream);
// Register row kernels with an 8-bit output (residual of type T).
template <typename T>
cudaError_t launch_rows_q8(const Problem &p, const Plan &plan, cudaStream_t stream);
template <typename T>
cudaError_t launch_stream(const Problem &p, const Plan &plan, cudaStream_t stream);
template <typename T, typename TR>
cudaError_t launch_cluster(const Problem &p, const Plan &plan, cudaStream_t stream);

// GEMM producer with the fused residual-add RMSNorm epilogue (gemm_norm.cuh).
struct GemmCall {
    const void *a;
    int64_t lda;
    const void *w;
    int64_t ldw;
    void *residual;
    int64_t ldr;
    void *y;
    int64_t ldy;
    const void *gamma;
    int64_t T, H, K;
    float eps;
    int ns, stages, bk;  // columns per CTA, ring stages, K slab (elements)
    float *workspace;    // [T][H / ns] partial sums of squares
    int num_sms;
    bool persistent;     // the warp-specialised persistent kernel (256-column tiles)
    bool pdl;
    unsigned int *watchdog;
    unsigned long long wait_limit_ns;  // bound on every shared-memory barrier wait
    long long stall_fill;              // test hook (-1: off)
};

template <typename T>
cudaError_t launch_gemm_norm(const GemmCall &c, cudaStream_t stream);

// Tile plan of the GEMM kernel: columns per CTA, K slab and ring depth within
// the shared memory given to one CTA (one or two CTAs per SM).  ns = 0:
// unsupported H.
struct GemmPlan {
    int ns = 0, tiles_n = 0, bk = 0, stages = 0, smem = 0;
    int64_t grid = 0;
    bool persistent = false;
};

constexpr int kGemmMaxTilesN = 32;

// Measured on GB300 (T = K = H = 4096, bf16): 256 columns per CTA with
// 128-byte K slabs and two CTAs per SM (one CTA's epilogue overlaps the
// other's main loop) 124.5 us; 512 columns, one CTA per SM, 147 us.  Rows
// wider than 32 tiles of 256 use 512-column tiles.
inline GemmPlan plan_gemm(int64_t T, int64_t H, int64_t K, int bk_override = 0,
                          int ns_override = 0, int ctas_override = 0, int persist_override = -1,
                          int num_sms = 152) {
    GemmPlan g;
    const bool fit256 = H % 256 == 0 && H / 256 <= kGemmMaxTilesN;
    const bool fit512 = H % 512 == 0 && H / 512 <= kGemmMaxTilesN;
    int ctas;
    if (fit256 && ns_override != 512) {
        g.ns = 256;
        g.bk = 64;
        ctas = 2;
    } else if (fit512) {
        g.ns = 512;
        g.bk = 32;
        ctas = 1;
    } else {
        return g;
    }
    if (bk_override == 32 || bk_override == 64) g.bk = bk_override;
    if (ctas_override == 1 || ctas_override == 2) ctas = ctas_override;
    const int smem_budget = ctas == 2 ? 113 * 1024 : 227 * 1024;
    g.tiles_n = (int)(H / g.ns);
    const int stage = (128 + g.ns) * g.bk * 2;
    const int fixed = 1024 + 1024;  // barriers, alignment slack
    g.stages = (smem_budget - fixed) / stage;
    if (g.stages > 8) g.stages = 8;
    // the epilogue stages the residual tile ([128 x ns] 16-bit) in the ring
    if (g.stages < 2 || g.stages * stage < 128 * g.ns * 2) return GemmPlan{};
    g.smem = g.stages * stage + fixed;
    g.grid = ((T + 127) / 128) * g.tiles_n;
    // 256-column tiles with 128-byte K slabs run persistent and
    // warp-specialised by default (one CTA per SM, 4 stages, two
    // accumulators: the main loop hides the epilogue), except for short K,
    // where there is little main loop to hide it behind and the two-CTA
    // kernel's TMA-staged epilogue is faster (K = 64: 26 vs 39 us at T = H =
    // 4096)
    g.persistent = g.ns == 256 && g.bk == 64 && ctas_override == 0 &&
                   (persist_override == 1 || (persist_override != 0 && K >= 512));
    if (g.persistent) {
        g.stages = 4;
        g.smem = 4 * stage + 1024 + 1024;
        g.grid = std::min<int64_t>(g.grid, num_sms);
    }
    return g;
}

// Workspace of the GEMM form: one binary32 per row and column tile (the
// column tiling depends on H only; -1: H not supported).
inline int64_t gemm_workspace_bytes(int64_t T, int64_t H) {
    const GemmPlan g = plan_gemm(T, H, 0);
    return g.ns == 0 ? -1 : T * g.tiles_n * 4;
}

}  // namespace rarn
