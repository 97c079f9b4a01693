// plan.h -- kernel plan (which kernel, launch shape) and the per-dtype
// launchers the C ABI dispatches to.  Host-side declarations only.
#pragma once

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

}  // namespace rarn
