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
};

// Largest CTA the register row kernels are compiled for, by the number of row
// values F each thread holds (16-byte packs x elements per pack, or single
// elements).  Keeps the pass-1 accumulators, load buffers and the staged row
// in registers without spilling.
__host__ __device__ constexpr int rows_max_block(int F) {
    return F <= 8 ? 1024 : F <= 16 ? 512 : F <= 32 ? 256 : 128;
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

template <typename T>
cudaError_t launch_rows(const Problem &p, const Plan &plan, cudaStream_t stream);
template <typename T>
cudaError_t launch_stream(const Problem &p, const Plan &plan, cudaStream_t stream);
template <typename T>
cudaError_t launch_cluster(const Problem &p, const Plan &plan, cudaStream_t stream);

}  // namespace rarn
