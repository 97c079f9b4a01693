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
};

// Largest CTA the register row kernels are compiled for, by the number of row
// values F each thread holds (16-byte packs x elements per pack, or single
// elements).  Keeps the pass-1 accumulators, load buffers and the staged row
// in registers without spilling.
__host__ __device__ constexpr int rows_max_block(int F) {
    return F <= 8 ? 1024 : F <= 16 ? 512 : F <= 32 ? 256 : 128;
}

template <typename T>
cudaError_t launch_rows(const Problem &p, const Plan &plan, cudaStream_t stream);

}  // namespace rarn
