// gemm_plan.h -- the GEMM form's call description, tile planner and the
// launcher the C ABI dispatches to.  Host-side declarations only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

namespace rarn {

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
    float *workspace;    // [T][H / ns] partial sums of squares, then the row-block counters
    int num_sms;
    bool persistent;     // the warp-specialised persistent kernel (256-column tiles)
    bool pair;           // ... on SM pairs: 256 x 256 tiles, cta_group::2 MMAs
    bool fuse_norm;      // the persistent kernels may write y (no norm kernel)
    bool tail_split;     // the pair kernel may split the last round's tiles
    int splitk;          // K split over this many CTAs per column tile (0: none)
    float *part;         // split-K partial products [splitk][T][H] in the workspace
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
    bool pair = false;
    bool fuse_norm = false;
    bool tail_split = false;
    int splitk = 0;  // K split over this many CTAs per column tile (0: none)
};

// Split K applies while the 128 x 256 tiles of the ceil(T / 128) row blocks
// leave at least half of the SMs idle, using up to the SMs they leave idle
// (counted as at most 152, the count the workspace is sized for), each split
// at least 8 K slabs of 64 and at most 9 splits (the parity bound allows 8
// extra binary32 roundings per element).  Measured (bf16, K = H = 4096,
// against the one-SM persistent kernel, us): T = 192 28.8 -> 15.2, T = 256
// 29.2 -> 15.6, T = 384 29.4 -> 18.8, T = 512 29.6 -> 21.6; T = 256,
// K = H = 8192 60.6 -> 44.1; T = 640 (no split) 30.3.
constexpr int kGemmMaxSplitK = 9;
constexpr int kGemmSplitKSMs = 152;

// Splits the workspace of T x H has room for (K unknown): 0 where split K
// cannot apply.
inline int splitk_room(int64_t T, int tiles_n) {
    if (tiles_n <= 0) return 0;
    const int64_t tiles = ((T + 127) / 128) * tiles_n;
    const int64_t s = std::min<int64_t>(kGemmMaxSplitK, kGemmSplitKSMs / tiles);
    return s >= 2 ? (int)s : 0;
}

inline int plan_splitk(int64_t T, int tiles_n, int64_t K, int num_sms) {
    if (tiles_n <= 0) return 0;
    const int64_t tiles = ((T + 127) / 128) * tiles_n;
    const int64_t kb = (K + 63) / 64;
    const int64_t sms = std::min<int64_t>(num_sms, kGemmSplitKSMs);
    int64_t s = std::min<int64_t>(kGemmMaxSplitK, std::min<int64_t>(sms / tiles, kb / 8));
    return s >= 2 ? (int)s : 0;
}

// The pair kernel's schedule: `walkers` two-CTA clusters walk items in
// row-major order (item i, i + walkers, ...).  When the last partial round
// holds at most half as many tiles as there are walkers, those tiles are
// split into two 128-column halves each.  y in the epilogue (a tile waits for
// the rest of its row block) needs at least as many walkers as a row block
// has items: then a wait only ever depends on items that no walker reaches
// through a wait on it.
struct PairSchedule {
    int64_t walkers = 0, full_items = 0, items = 0;
    bool fuse_ok = false;
};

inline PairSchedule pair_schedule(int64_t T, int tiles_n, int64_t clusters, bool allow_split) {
    PairSchedule s;
    const int64_t ptiles = ((T + 255) / 256) * tiles_n;
    s.walkers = std::min<int64_t>(ptiles, clusters);
    const int64_t tail = ptiles % s.walkers;
    const bool split = allow_split && tail > 0 && 2 * tail <= s.walkers;
    s.full_items = split ? ptiles - tail : ptiles;
    s.items = split ? ptiles + tail : ptiles;
    s.fuse_ok = s.walkers >= (split ? 2 : 1) * (int64_t)tiles_n;
    return s;
}

// The one-SM persistent kernel: CTAs walk 128 x 256 tiles in row-major order.
inline bool single_fuse_ok(int64_t T, int tiles_n, int num_sms) {
    return std::min<int64_t>(((T + 127) / 128) * tiles_n, num_sms) >= tiles_n;
}

constexpr int kGemmMaxTilesN = 32;

// Measured on GB300 (T = K = H = 4096, bf16): 256 columns per CTA with
// 128-byte K slabs and two CTAs per SM (one CTA's epilogue overlaps the
// other's main loop) 124.5 us; 512 columns, one CTA per SM, 147 us.  Rows
// wider than 32 tiles of 256 use 512-column tiles.
inline GemmPlan plan_gemm(int64_t T, int64_t H, int64_t K, int bk_override = 0,
                          int ns_override = 0, int ctas_override = 0, int persist_override = -1,
                          int num_sms = 152, int pair_override = -1, int fuse_override = -1,
                          int split_override = -1, int splitk_override = -1) {
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
    // a single row block with long K splits K over the SMs the column tiles
    // leave idle (measured, bf16, T x H x K: 1 x 4096 x 4096 11.8 us against
    // 25.5 on the persistent kernel, 16 x 4096 x 4096 9.6 against 25.7,
    // 32 x 2048 x 8192 11.0 against 43.1)
    if (g.ns == 256 && ctas_override == 0 && bk_override == 0 && persist_override == -1 &&
        splitk_override != 0) {
        g.splitk = plan_splitk(T, g.tiles_n, K, num_sms);
        if (g.splitk) {
            g.bk = 64;
            g.stages = 4;
            g.smem = 4 * (128 + 256) * 64 * 2 + 2048;
            g.grid = ((T + 127) / 128) * g.tiles_n * g.splitk;
            return g;
        }
    }
    // 256-column tiles with 128-byte K slabs run persistent and
    // warp-specialised by default (one CTA per SM, 4 stages, two
    // accumulators: the main loop hides the epilogue), except for short K,
    // where there is little main loop to hide it behind and the two-CTA
    // kernel's TMA-staged epilogue is faster (K = 64: 26 vs 39 us at T = H =
    // 4096)
    g.persistent = g.ns == 256 && g.bk == 64 && ctas_override == 0 &&
                   (persist_override == 1 || (persist_override != 0 && K >= 512));
    if (g.persistent) {
        g.stages = std::min(9, (227 * 1024 - 3 * 1024) / stage);
        g.smem = g.stages * stage + 3 * 1024;
        g.grid = std::min<int64_t>(g.grid, num_sms);
        // SM pairs (256-row tiles, each CTA staging half of the W slab) from
        // 2048 rows, or, for K >= 2048, wherever one SM per 128-row tile
        // would take more than one round of the SMs; measured (one SM per
        // tile / pairs, us): K = H = 4096 T = 768 31.0 / 31.3, T = 1024
        // 31.6 / 32.2, T = 1280 52.1 / 45.6, T = 1536 52.7 / 45.8, T = 1792
        // 53.4 / 50.1, T = 2048 56.4 / 53.1; T = 1024, K = H = 8192
        // 112.4 / 100.9; T = 1536, K = H = 5120 69.8 / 64.2; but T = 1200,
        // H = 4096, K = 1024 23.9 / 27.1
        g.pair = pair_override == 1 ||
                 (pair_override != 0 &&
                  (T >= 2048 || (K >= 2048 && ((T + 127) / 128) * g.tiles_n > num_sms)));
        if (g.pair) {
            // the pair kernel's ring: 3 stages of two K slabs, 64 KB each
            // (gemm_norm.cuh PairLayout, gemm_norm_launch.cuh)
            const int half = (128 + g.ns / 2) * g.bk * 2;
            g.stages = 3;
            g.smem = g.stages * 2 * half + 4 * 1024;
            g.grid = 2 * std::min<int64_t>(((T + 255) / 256) * g.tiles_n, num_sms / 2);
        }
        // y in the epilogue only where the main loop is long enough to hide
        // it; with short K a separate norm kernel costs less (y separate /
        // in the epilogue, us): K = H = 4096 T = 4096 K = 4096 94.0 / 88.6,
        // K = 3072 75.3 / 71.6, K = 1024 43.5 / 49.8, K = 512 39.0 / 45.8;
        // T = 2048, K = 3072 43.2 / 41.7, K = 2048 34.1 / 35.0; T = 8192,
        // K = 2048 108.2 / 104.2; T = 1536, K = 1024 23.0 / 27.4
        const bool fuse_wanted =
            fuse_override == 1 || (fuse_override == -1 && (K >= 3072 || (K >= 2048 && T >= 4096)));
        if (g.pair) {
            const PairSchedule ps = pair_schedule(T, g.tiles_n, num_sms / 2, split_override != 0);
            g.tail_split = ps.items != ps.full_items;
            g.fuse_norm = fuse_wanted && ps.fuse_ok;
        } else {
            g.fuse_norm = fuse_wanted && single_fuse_ok(T, g.tiles_n, num_sms);
        }
    }
    return g;
}

// Workspace of the GEMM form: partial sums of squares (one binary32 per row
// and 128 columns: the persistent kernels' slots; the other kernel's 256- or
// 512-column tiles use fewer), then, 16-byte aligned, one 32-bit counter per
// 128-row block.
inline int64_t gemm_counters_offset(int64_t T, int64_t H) {  // in floats
    return (T * (H / 128) + 3) / 4 * 4;
}

inline int64_t gemm_workspace_bytes_for(int64_t T, int64_t H) {
    return (gemm_counters_offset(T, H) + (T + 127) / 128) * 4;
}

// Split K (few row blocks): the partial products follow, 256-byte aligned, as
// splits x T x H binary32 values.
inline int64_t gemm_splitk_offset(int64_t T, int64_t H) {  // in floats
    return (gemm_workspace_bytes_for(T, H) / 4 + 63) / 64 * 64;
}

inline int64_t gemm_splitk_bytes(int64_t T, int64_t H, int splits) {
    return (gemm_splitk_offset(T, H) + (int64_t)splits * T * H) * 4;
}

// -1: H not supported.
inline int64_t gemm_workspace_bytes(int64_t T, int64_t H) {
    const GemmPlan g = plan_gemm(T, H, 0);
    if (g.ns == 0) return -1;
    // room for split K at its largest whenever it can apply
    const int room = g.ns == 256 ? splitk_room(T, (int)(H / 256)) : 0;
    return room ? gemm_splitk_bytes(T, H, room) : gemm_workspace_bytes_for(T, H);
}

}  // namespace rarn
