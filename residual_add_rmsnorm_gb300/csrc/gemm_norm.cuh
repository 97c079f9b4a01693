// gemm_norm.cuh -- a GEMM whose epilogue is the fused residual-add RMSNorm.
//
//   P = A W^T          A [T, K] activations, W [H, K] a linear layer's weight
//   h = RN(P + r)      residual <- h   (the accumulator plus the residual, one rounding)
//   y = RN((h * inv) * gamma),  inv = rsqrt(mean(h^2) + eps)
//
// The partial P is never written: the epilogue consumes the accumulator tile
// where the matrix unit left it ("sm80 GEMM + ReduceScatter", the flux
// epilogue, consumes the accumulator tile before anything is written;
// "Tokenweave fused-RMSNorm-AR kernel", Code walkthrough, for the norm steps).
//
// Blackwell mapping (sm_103a); the kernels of this file, by problem shape:
//   * K >= 512, T >= 2048 (H <= 8192; also fewer rows with K >= 2048 when
//     one SM per 128 x 256 tile would need more than a round of the SMs):
//     k_gemm_res_pair, persistent on SM
//     pairs (two-CTA clusters, tcgen05.mma.cta_group::2 on 256 x 256 tiles;
//     the last partial round as 128-column halves), warp-specialised: a TMA
//     producer, one MMA-issuing thread, 8 epilogue warps per CTA draining one
//     of two TMEM accumulators while the next tile's MMAs run.  The epilogue
//     adds the residual (one rounding), publishes per-128-column partial
//     sums of squares (adding to its 128-row block's counter, which
//     k_zero_counters zeroes first), writes h, and once the counter shows
//     every column writes y -- for a tile whose row block ends in the next
//     round of tiles, during the pair's next tile.  (Where K is short,
//     k_norm_ss writes y after the kernel instead.)  The epilogue's streams
//     (residual in, h and y out) carry an L2 evict-first policy.
//   * K >= 512, 128 < T < 2048 (or T <= 128 with short K): k_gemm_res_ws,
//     the same on one SM per 128 x 256 tile (M = 128 MMAs).
//   * K >= 1024 and so few 128 x 256 tiles that they leave half of the SMs
//     idle (up to 512 rows at H = 4096, 1152 at H = 2048): k_gemm_splitk,
//     M x C x S CTAs each multiplying a K range of one tile and writing
//     binary32 partial products; k_splitk_norm (a CTA per row, or
//     k_splitk_norm_cluster, 8 per row, for few wide rows) sums them in
//     split order, adds the residual and normalises.
//   * K < 512: k_gemm_res, one CTA per [128 x NS] tile (NS = 256 or 512), the
//     operand ring staging the epilogue: the residual tile arrives by TMA in
//     [128 x 32] chunks (64-byte swizzle), each thread adds its accumulator
//     row (tcgen05.ld), rounds once and writes h back for a TMA store; the
//     tile's partial sums of squares go to the workspace; k_norm_ss (a warp
//     per row slice, PDL-chained) then sums them in order and writes y.
// In every form the accumulator is binary32 in TMEM, operands arrive by TMA
// (cp.async.bulk.tensor, 2-D tiles in the 128- or 64-byte swizzle) and one
// thread issues tcgen05.mma (kind::f16) and commits each ring stage back.
//
// Every mbarrier wait is bounded (global timer); a wait that runs out sets the
// watchdog word and the CTA's abort flag, the CTA drains what it issued (also
// bounded), frees its tensor memory and returns with its outputs invalid.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the map is encoded on the host)

#include <type_traits>

#include "common.cuh"
#include "gemm_plan.h"

namespace rarn {
namespace gemm {

constexpr int kBM = 128;       // tile rows = TMEM lanes
constexpr int kMmaN = 256;     // N of one tcgen05.mma
constexpr int kMmaK = 16;      // K of one tcgen05.mma (16-bit inputs)
constexpr int kThreads = 128;  // 4 warps
constexpr unsigned int kWatchGemm = 4u;  // watchdog bit
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int kChunkCols = 32;                      // epilogue chunk: 128 rows x 32 columns
constexpr int kChunkBytes = kBM * kChunkCols * 2;   // 8 KB
constexpr int kMaxChunks = 16;                      // 512 columns per CTA

// Shared-memory layout of one CTA (dynamic, 1024-byte aligned base).
struct Layout {
    int a_bytes, b_bytes, stage_bytes, ctl_off, total;
};

__host__ __device__ constexpr Layout layout(int stages, int ns, int bk) {
    Layout L{};
    L.a_bytes = kBM * bk * 2;
    L.b_bytes = ns * bk * 2;
    L.stage_bytes = L.a_bytes + L.b_bytes;
    L.ctl_off = stages * L.stage_bytes;
    // full[S], empty[S], accum, chunk[16] (8 B each), tmem slot, abort word
    L.total = L.ctl_off + (2 * stages + 1 + kMaxChunks) * 8 + 8 + 1024;  // + alignment slack
    return L;
}

struct Params {
    float *ss;         // workspace [T][C]: per row, each column tile's sum of squares of h
    int64_t T, H, K;
    int ns;            // columns per CTA
    int C;             // column tiles (H / ns); the persistent kernels' partial sums
                       // come in 2 C slots of 128 columns per row
    int stages;
    int kblocks;       // ceil(K / BK)
    unsigned int *watchdog;
    unsigned long long wait_limit_ns;
    long long stall_fill;  // test hook: in CTA 0 this ring fill (0-based, in issue order)
                           // expects 16 bytes more than it brings, so it never completes
    // The norm in the persistent kernels' epilogue: a tile publishes its rows'
    // partial sums by adding 1 to its 128-row block's counter; once the
    // counter reaches C every tile of the block scales the h it still holds
    // by inv and gamma and writes y.  counters == nullptr: the norm kernel
    // writes y instead.
    unsigned int *counters;  // [ceil(T / 128)], zero when the kernel starts
    // the pair kernel's items: tiles [0, full_items) whole, then the
    // remaining tiles as two 128-column halves each (items in all)
    int64_t full_items, items;
    // split K (few row blocks): CTA (row block m, tile n, split s) multiplies K slabs
    // [s * kb_per_split, ...) and writes its binary32 partial products to
    // part[s][row][column]
    float *part;
    int splits, kb_per_split;
    int a_rows;  // rows of A each fill brings (a multiple of 8 up to 128; the
                 // MMA's other rows of the tile are not written out)
    void *y;
    int64_t ldy;
    const void *gamma;
    float eps;
};

// Kernel 2 arguments.
struct NormParams {
    void *y;
    const void *h;     // the updated residual
    const void *gamma;
    const float *ss;   // [T][C] partial sums of squares, added in order
    int64_t T, H, ldh, ldy;
    int C;             // partial sums per row (at most 64)
    float eps;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same with acquire semantics at cluster scope: for a barrier that
// threads of the peer CTA arrive on (release at cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on a phase of `bar`.  Gives up when the CTA's abort word is
// set (unless `ignore_abort`) or after `limit_ns`: then sets the abort word
// and the watchdog bit and returns false.
// kCluster: acquire at cluster scope (arrivals from the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned int *watchdog, unsigned long long limit_ns,
                                           bool ignore_abort = false) {
    auto try_wait = [&] {
        return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (try_wait()) return true;
    unsigned long long t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (try_wait()) return true;
        if ((i & 127u) == 0) {
            if (!ignore_abort && *abort_flag) return false;
            const unsigned long long t = now_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(watchdog, kWatchGemm);
                return false;
            }
        }
    }
}

// Sum of a row's n partial sums (n even, the row 8-byte aligned), added in
// order; loaded past L1 (other SMs wrote them) 32 at a time, so a row costs
// n / 32 round trips to L2.  Rows of a multiple of 8 sums that start on a
// 32-byte boundary are read a whole sector per load (8-byte loads would
// touch each sector four times).
__device__ __forceinline__ float row_sum(const float *sr, int n) {
    float tot = 0.f;
    if (n % 8 == 0 && (reinterpret_cast<uintptr_t>(sr) & 31u) == 0) {
        for (int q0 = 0; q0 < n; q0 += 32) {
            uint32_t x[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (q0 + 8 * j < n) {
                    asm volatile("ld.global.cg.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                                 : "=r"(x[j][0]), "=r"(x[j][1]), "=r"(x[j][2]), "=r"(x[j][3]),
                                   "=r"(x[j][4]), "=r"(x[j][5]), "=r"(x[j][6]), "=r"(x[j][7])
                                 : "l"(sr + q0 + 8 * j));
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[j][e] = 0u;
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (q0 + 8 * j < n) {
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        tot = (tot + __uint_as_float(x[j][e])) + __uint_as_float(x[j][e + 1]);
                }
        }
        return tot;
    }
    for (int q0 = 0; q0 < n; q0 += 32) {
        float2 x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            x[j] = q0 + 2 * j < n ? __ldcg(reinterpret_cast<const float2 *>(sr + q0) + j)
                                  : make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (q0 + 2 * j < n) tot = (tot + x[j].x) + x[j].y;
    }
    return tot;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *cnt >= target (other CTAs' tiles published); gives up
// like wait_phase.
__device__ __forceinline__ bool wait_count(const unsigned int *cnt, unsigned int target,
                                           volatile int *abort_flag, unsigned int *watchdog,
                                           unsigned long long limit_ns) {
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire_u32(cnt) >= target) return true;
        if ((i & 15u) == 15u) {
            if (*abort_flag) return false;
            const unsigned long long t = now_ns();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(watchdog, kWatchGemm);
                return false;
            }
        }
        __nanosleep(64);
    }
}

// 2-D TMA tile load into shared memory, completion on `bar` (byte count).
// c0 is the innermost (K) coordinate: a multiple of BK, so c0 * 2 bytes is a
// multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 32-byte global accesses (one full sector per thread): a thread of the
// persistent kernels' epilogue owns one row, so its accesses are the only
// ones to that row's sectors in a warp-wide instruction.
struct Pack32 {
    uint4 a, b;
};

__device__ __forceinline__ Pack32 ld_stream32(const void *p) {
    Pack32 v;
    asm volatile("ld.global.cs.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.a.x), "=r"(v.a.y), "=r"(v.a.z), "=r"(v.a.w), "=r"(v.b.x), "=r"(v.b.y),
                   "=r"(v.b.z), "=r"(v.b.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_global32(void *p, const uint4 &a, const uint4 &b) {
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y),
                 "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// The persistent kernels' epilogue streams (the residual in, h and y out)
// with an L2 policy that lets those lines go first when L2 needs room: the
// operands, re-read by every tile, stay (T = K = H = 4096: 94.3 -> 92.0 us;
// [8192, 4096, 4096] 168.5 -> 165.1; [16384, 5120, 5120] 508.7 -> 501.2).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ Pack32 ld_stream32(const void *p, uint64_t pol) {
    Pack32 v;
    asm volatile(
        "ld.global.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
        : "=r"(v.a.x), "=r"(v.a.y), "=r"(v.a.z), "=r"(v.a.w), "=r"(v.b.x), "=r"(v.b.y),
          "=r"(v.b.z), "=r"(v.b.w)
        : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void st_global32(void *p, const uint4 &a, const uint4 &b,
                                            uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p),
                 "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w),
                 "l"(pol)
                 : "memory");
}

// L2 policy that keeps lines resident in preference to others (the GEMM's
// operands, re-read by every tile of a row or column of tiles).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int c0,
                                                 int c1, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(pol)
        : "memory");
}

// 2-D TMA tile store from shared memory (bulk group); rows and columns
// outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int c0, int c1, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// This thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's shared-memory writes visible to the TMA (async proxy).
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Barrier over the CTA's 128 threads (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void epi_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// BK * 2 = 128 (or 64) bytes, swizzled in 8-row atoms by the TMA
// (128-byte / 64-byte swizzle): start address, stride between 8-row groups
// (8 rows x row bytes), descriptor version 1, swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, int row_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;  // leading byte offset: unused for swizzled K-major
    d |= static_cast<uint64_t>((8 * row_bytes) >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(row_bytes == 128 ? 2 : 4) << 61;  // 128B / 64B swizzle
    return d;
}

// Instruction descriptor, kind::f16: binary32 accumulator, A and B of the same
// 16-bit type (bf16: 1, f16: 0), both K-major, M = 128, N = N_ (default 256).
template <typename T, int N_ = kMmaN>
__host__ __device__ constexpr uint32_t instr_desc() {
    static_assert(N_ % 16 == 0 && N_ >= 16 && N_ <= 256, "M = 128 takes N = 16 .. 256");
    constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4)                   // D: f32
           | (ab << 7) | (ab << 10)    // A, B type
           | (0u << 15) | (0u << 16)   // K-major A, B
           | ((uint32_t)(N_ >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM (this warp's lane quarter).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// One thread's share of a persistent kernel's epilogue for one tile: the
// NC accumulator columns at TMEM address `taddr` plus the residual row
// segment `rv` (prefetched), rounded once to h, stored back over the
// residual at `res`; returns the sum of squares of h in column order.
// Wide: 32-byte accesses (residual rows 32-byte aligned), else 16-byte.
template <typename T, int NC, bool Wide>
struct EpiRow {
    static constexpr int kPacks = Wide ? NC / 16 : NC / 8;
    using Pk = typename std::conditional<Wide, Pack32, uint4>::type;
    Pk rv[kPacks];

    __device__ __forceinline__ void load(const T *res) {
        [[maybe_unused]] const uint64_t pol = l2_evict_first_policy();
#pragma unroll
        for (int q = 0; q < kPacks; ++q) {
            if constexpr (Wide)
                rv[q] = ld_stream32(res + 16 * q, pol);
            else
                rv[q] = ld_stream(res + 8 * q);
        }
    }

    // h = RN(accumulator + residual) into rv, and the row's sum of squares
    // of h.  The sum of squares is formed per 64 columns and those sums
    // added in column order, so a 128-column slot has the same bits whether
    // one thread or two warp halves (64 columns each) computed it.  h is
    // stored by store_h, once the accumulator is released.
    __device__ __forceinline__ float run(uint32_t taddr, bool live) {
        static_assert(NC % 64 == 0, "64-column partial sums");
        float ss = 0.f, part = 0.f;
#pragma unroll
        for (int c = 0; c < NC; c += 32) {
            float v[32];
            tmem_ld32(taddr + c, v);
            if (live) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // 8 columns each, in column order
                    uint4 r;
                    if constexpr (Wide)
                        r = (q & 1) ? rv[c / 16 + q / 2].b : rv[c / 16 + q / 2].a;
                    else
                        r = rv[c / 8 + q];
                    float f[8];
                    DT<T>::unpack(r, f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        f[e] = DT<T>::round(v[8 * q + e] + f[e]);  // h: one rounding
                        part += f[e] * f[e];
                    }
                    if constexpr (Wide) {
                        if (q & 1)
                            rv[c / 16 + q / 2].b = DT<T>::pack(f);
                        else
                            rv[c / 16 + q / 2].a = DT<T>::pack(f);
                    } else {
                        rv[c / 8 + q] = DT<T>::pack(f);
                    }
                }
            }
            if (c % 64 == 32) {
                ss += part;
                part = 0.f;
            }
        }
        return ss;
    }

    // After run(): h back into the residual's row.
    __device__ __forceinline__ void store_h(T *res) const {
        [[maybe_unused]] const uint64_t pol = l2_evict_first_policy();
#pragma unroll
        for (int q = 0; q < kPacks; ++q) {
            if constexpr (Wide)
                st_global32(res + 16 * q, rv[q].a, rv[q].b, pol);
            else
                st_global(res + 8 * q, rv[q]);
        }
    }

    // After run(): y = RN((h * inv) * gamma) for the same columns.
    __device__ __forceinline__ static uint4 scale(const uint4 &h, float inv, const T *g) {
        float f[8], w[8];
        DT<T>::unpack(h, f);
        DT<T>::unpack(ld_keep(g), w);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = (f[e] * inv) * w[e];
        return DT<T>::pack(f);
    }

    __device__ __forceinline__ void store_y(float inv, const T *g, T *y) const {
        [[maybe_unused]] const uint64_t pol = l2_evict_first_policy();
#pragma unroll
        for (int q = 0; q < kPacks; ++q) {
            if constexpr (Wide)
                st_global32(y + 16 * q, scale(rv[q].a, inv, g + 16 * q),
                            scale(rv[q].b, inv, g + 16 * q + 8), pol);
            else
                st_global(y + 8 * q, scale(rv[q], inv, g + 8 * q));
        }
    }
};

// ---------------------------------------------------------------------------
// Kernel 1.  Grid: C x ceil(T / 128) CTAs (C = H / NS column tiles); CTA b
// owns rows [128 (b / C), +128) and columns [NS (b % C), +NS).
// ---------------------------------------------------------------------------
template <typename T, int BK>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_res(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
               const __grid_constant__ CUtensorMap map_r, Params p) {
    static_assert(BK == 64 || BK == 32, "K slab of 128 or 64 bytes");
    constexpr int kRowBytes = BK * 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzle atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages, NS = p.ns;
    const Layout L = layout(S, NS, BK);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.ctl_off);
    uint64_t *empty = full + S;
    uint64_t *accum = empty + S;
    uint64_t *chunk_bar = accum + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(chunk_bar + kMaxChunks);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const int ntile = (int)(blockIdx.x % C);  // consecutive CTAs share the A tile (L2)
    const int64_t m0 = (int64_t)(blockIdx.x / C) * kBM;
    const int n0 = ntile * NS;
    const uint32_t ncols = NS;  // TMEM columns (power of two >= 32)

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum), 1);
        for (int c = 0; c < kMaxChunks; ++c) mbar_init(smem_u32(&chunk_bar[c]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(ncols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = *tmem_slot;

    grid_dependency_wait();  // A, W and the residual may come from the previous kernel

    const uint32_t idesc = instr_desc<T>();
    const int KB = p.kblocks;
    int issued = 0;  // producer: fills issued
    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % S;
            if (kb >= S &&
                !wait_phase(smem_u32(&empty[s]), ((kb / S) - 1) & 1, abort_flag, p.watchdog,
                            p.wait_limit_ns))
                break;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, L.stage_bytes + (blockIdx.x == 0 && kb == p.stall_fill ? 16u : 0u));
            const uint32_t sa = smem_u32(smem + s * L.stage_bytes);
            const uint32_t sb = sa + L.a_bytes;
            tma_load_2d(sa, &map_a, kb * BK, (int)m0, fb);
            for (int h = 0; h < NS / kMmaN; ++h)
                tma_load_2d(sb + h * kMmaN * kRowBytes, &map_w, kb * BK, n0 + h * kMmaN, fb);
            issued = kb + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        int done = 0;
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % S;
            if (!wait_phase(smem_u32(&full[s]), (kb / S) & 1, abort_flag, p.watchdog,
                            p.wait_limit_ns))
                break;
            tmem_fence_after();
            const uint32_t sa = smem_u32(smem + s * L.stage_bytes);
            const uint32_t sb = sa + L.a_bytes;
#pragma unroll
            for (int kk = 0; kk < BK / kMmaK; ++kk) {
                const uint64_t ad = smem_desc(sa + kk * kMmaK * 2, kRowBytes);
                for (int h = 0; h < NS / kMmaN; ++h) {
                    const uint64_t bd = smem_desc(sb + h * kMmaN * kRowBytes + kk * kMmaK * 2,
                                                  kRowBytes);
                    mma_f16(tmem + h * kMmaN, ad, bd, idesc, (kb | kk) != 0);
                }
            }
            mma_commit(smem_u32(&empty[s]));  // frees the stage once these MMAs are done
            done = kb + 1;
        }
        mma_commit(smem_u32(accum));  // arrives once every MMA issued has completed
        (void)done;
    }
    __syncwarp();

    // ---- epilogue: all 128 threads, thread i = row m0 + i ----
    wait_phase(smem_u32(accum), 0, abort_flag, p.watchdog, p.wait_limit_ns, true);
    tmem_fence_after();
    __syncthreads();
    const bool ok = !*abort_flag;  // the same snapshot in every thread
    grid_launch_dependents();
    const int r = threadIdx.x;
    const uint32_t tbase = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int nchunks = NS / kChunkCols;
    const uint32_t ring = smem_u32(smem);  // every MMA has completed: the ring is free
    // byte offset of 16-byte piece q of row r within a chunk (64-byte swizzle:
    // the piece index is XORed with bits 1-2 of the row)
    const uint32_t row_off = static_cast<uint32_t>(r) * 64u;
    const uint32_t swz = (static_cast<uint32_t>(r) >> 1) & 3u;
    if (ok && threadIdx.x == 0) {
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t cb = smem_u32(&chunk_bar[c]);
            mbar_arrive_expect_tx(cb, kChunkBytes);
            tma_load_2d(ring + c * kChunkBytes, &map_r, n0 + c * kChunkCols, (int)m0, cb);
        }
    }
    float ss = 0.f;
    for (int c = 0; c < nchunks; ++c) {
        float v[32];
        tmem_ld32(tbase + c * kChunkCols, v);
        const uint32_t ca = ring + c * kChunkBytes + row_off;
        if (ok) {
            wait_phase(smem_u32(&chunk_bar[c]), 0, abort_flag, p.watchdog, p.wait_limit_ns, true);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float f[8];
                const uint32_t a = ca + ((q ^ swz) << 4);
                DT<T>::unpack(lds128(a), f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    f[e] = DT<T>::round(v[8 * q + e] + f[e]);  // h: one rounding of acc + r
                    ss += f[e] * f[e];
                }
                sts128(a, DT<T>::pack(f));
            }
            fence_async_shared();
        }
        epi_barrier();
        if (ok && threadIdx.x == 0) {
            tma_store_2d(&map_r, n0 + c * kChunkCols, (int)m0, ring + c * kChunkBytes);
            bulk_commit();
        }
    }
    if (ok && m0 + r < p.T) p.ss[(m0 + r) * C + ntile] = ss;
    if (threadIdx.x == 0) {
        bulk_wait_all();  // the stores have completed before this CTA's memory goes away
        if (*abort_flag) {
            // after an abort anywhere in the CTA, the operand fills and the
            // residual chunks issued land before its memory goes away (bounded)
            for (int kb = issued - S > 0 ? issued - S : 0; kb < issued; ++kb)
                wait_phase(smem_u32(&full[kb % S]), (kb / S) & 1, abort_flag, p.watchdog,
                           p.wait_limit_ns, true);
            for (int c = 0; ok && c < nchunks; ++c)
                wait_phase(smem_u32(&chunk_bar[c]), 0, abort_flag, p.watchdog, p.wait_limit_ns,
                           true);
        }
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(ncols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Kernel 1, persistent and warp-specialised (NT = 256- or 128-column tiles):
// one CTA per SM walks tiles b, b + G, ... (G = grid size).  Warp 0 lane 0
// feeds a ring of [128 + NT] x 64 operand slabs by TMA (4 stages for NT = 256,
// 6 for 128); warp 1 lane 0 issues the MMAs into one of two TMEM accumulators
// (2 x NT columns) while
// warps 2-9 drain the other: the next tile's main loop overlaps this tile's
// epilogue, and the whole shared memory serves the operand ring.  Epilogue
// warp w reads TMEM lane quarter w % 4 and half (w - 2) / 4 of the tile's
// columns; it reads the residual and writes h with 16-byte accesses of each
// thread's own row, the next chunk's residual in flight while this chunk is
// added.
// ---------------------------------------------------------------------------
constexpr int kWsEpiWarps = 8;

// Barrier over the persistent kernel's 8 epilogue warps (id 2).
__device__ __forceinline__ void epi_barrier_ws() {
    asm volatile("bar.sync 2, %0;" ::"n"(32 * kWsEpiWarps) : "memory");
}
constexpr int kWsThreads = 64 + 32 * kWsEpiWarps;

template <int NT, int BK = 64>
struct WsLayout {
    static constexpr int a_bytes = kBM * BK * 2;                 // 16 KB (BK = 64)
    static constexpr int b_bytes = NT * BK * 2;                  // 32 KB (NT = 256, BK = 64)
    static constexpr int stage_bytes = a_bytes + b_bytes;        // 48 KB
    // as many stages as fit next to 3 KB of barriers and slack (at most 9)
    static constexpr int stages =
        (227 * 1024 - 3 * 1024) / stage_bytes > 9 ? 9 : (227 * 1024 - 3 * 1024) / stage_bytes;
    static constexpr int ctl_off = stages * stage_bytes;
    // full[S], empty[S], tfull[2], tempty[2], mma_done, tmem slot, abort
    // word, the epilogue's half-row sums
    static constexpr int total =
        ctl_off + (2 * stages + 5) * 8 + 8 + kWsEpiWarps * 32 * 4 + 16 + 1024;
};

template <typename T, int NT, int BK, bool Wide>
__global__ void __launch_bounds__(kWsThreads, 1)
    k_gemm_res_ws(const __grid_constant__ CUtensorMap map_a,
                  const __grid_constant__ CUtensorMap map_w, void *residual, int64_t ldr,
                  Params p) {
    static_assert(BK == 64 || BK == 32, "K slab of 128 or 64 bytes");
    using WsLayout = rarn::gemm::WsLayout<NT, BK>;
    constexpr int S = WsLayout::stages;
    constexpr int NS = NT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + WsLayout::ctl_off);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *half_ss = reinterpret_cast<float *>(tmem_slot + 2);  // [8 warps][32]
    volatile int *tile_ok = reinterpret_cast<volatile int *>(half_ss + kWsEpiWarps * 32);
    volatile int *norm_ok = tile_ok + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const int64_t mtiles = (p.T + kBM - 1) / kBM;
    const int64_t ntiles = mtiles * C;
    const int KB = p.kblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 32 * kWsEpiWarps);  // every epilogue thread
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // A, W and the residual may come from the previous kernel

    int64_t kit = 0;  // producer: k-slabs issued so far (all tiles)
    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer ----
            // ring position kept incrementally (stage s, round parity ph): the
            // issuing threads' instruction latency is on the critical path
            bool stop = false;
            uint32_t s = 0, ph = 0;
            const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty), ring0 = smem_u32(smem);
            // the operands stay in L2 ahead of the residual and h streams
            const uint64_t pol = l2_evict_last_policy();
            for (int64_t tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
                const int m0 = (int)((tile / C) * kBM);
                const int n0 = (int)((tile % C) * NS);
                for (int kb = 0; kb < KB; ++kb, ++kit) {
                    // fill kit of round r waits for the release of round r - 1
                    if (kit >= S && !wait_phase(empty0 + 8 * s, ph ^ 1u, abort_flag, p.watchdog,
                                                p.wait_limit_ns)) {
                        stop = true;
                        break;
                    }
                    const uint32_t fb = full0 + 8 * s;
                    mbar_arrive_expect_tx(
                        fb, WsLayout::stage_bytes + (blockIdx.x == 0 && kit == p.stall_fill ? 16u : 0u));
                    const uint32_t sa = ring0 + s * WsLayout::stage_bytes;
                    tma_load_2d_hint(sa, &map_a, kb * BK, m0, fb, pol);
                    tma_load_2d_hint(sa + WsLayout::a_bytes, &map_w, kb * BK, n0, fb, pol);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer ----
            const uint32_t idesc = instr_desc<T, NT>();
            // descriptors of stage 0, advanced by adds (start address in
            // 16-byte units: a stage is stage_bytes / 16, a K step 2)
            const uint64_t adesc0 = smem_desc(smem_u32(smem), BK * 2);
            const uint64_t bdesc0 = smem_desc(smem_u32(smem) + WsLayout::a_bytes, BK * 2);
            constexpr uint32_t kStageDesc = WsLayout::stage_bytes >> 4;
            const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
            uint32_t s = 0, ph = 0;
            int it = 0;
            bool stop = false;
            for (int64_t tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                if (it >= 2 && !wait_phase(smem_u32(&tempty[acc]), (uint32_t)(((it >> 1) - 1) & 1),
                                           abort_flag, p.watchdog, p.wait_limit_ns))
                    break;
                tmem_fence_after();
                const uint32_t d = tmem + acc * NS;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase(full0 + 8 * s, ph, abort_flag, p.watchdog, p.wait_limit_ns)) {
                        stop = true;
                        break;
                    }
                    tmem_fence_after();
                    const uint64_t ad = adesc0 + s * kStageDesc, bd = bdesc0 + s * kStageDesc;
                    mma_f16(d, ad, bd, idesc, kb != 0);
#pragma unroll
                    for (int kk = 1; kk < BK / kMmaK; ++kk)
                        mma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
                    mma_commit(empty0 + 8 * s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!stop) mma_commit(smem_u32(&tfull[acc]));
            }
            // every MMA issued has completed before tensor memory is freed
            mma_commit(smem_u32(mma_done));
            wait_phase(smem_u32(mma_done), 0, abort_flag, p.watchdog, p.wait_limit_ns, true);
        }
        __syncwarp();
    } else {
        // ---- epilogue: warps 2-9, TMEM lane quarter warp % 4, column half ----
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int c0 = ((warp - 2) >> 2) * (NS / 2);
        int it = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const int64_t m0 = (tile / C) * kBM;
            const int ntile = (int)(tile % C);
            const int64_t t = m0 + row;
            const bool live = t < p.T;
            T *res = reinterpret_cast<T *>(residual) + (live ? t : 0) * ldr + ntile * NS + c0;
            // this thread's residual columns are loaded before the wait for
            // the accumulator, so they arrive while the tile's MMAs run
            EpiRow<T, NS / 2, Wide> er;
            if (live) er.load(res);
            // one thread waits (bounded) and the 8 warps leave together, so
            // none is left at the epilogue barrier
            if (warp == 2 && lane == 0)
                *tile_ok = wait_phase(smem_u32(&tfull[acc]), (uint32_t)((it >> 1) & 1), abort_flag,
                                      p.watchdog, p.wait_limit_ns)
                               ? 1
                               : 0;
            epi_barrier_ws();
            if (!*tile_ok) break;
            tmem_fence_after();
            if (tile + gridDim.x >= ntiles) grid_launch_dependents();
            const uint32_t taddr =
                tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * NS + c0;
            const float ss = er.run(taddr, live);
            tmem_fence_before();
            mbar_arrive(smem_u32(&tempty[acc]));  // the accumulator is free again
            // h stored only now, off the accumulator's critical path
            if (live) er.store_h(res);
            // each warp half's 128 columns are one partial-sum slot of the row
            const int slots = 2 * C;
            if (live && !*abort_flag) p.ss[t * slots + ntile * 2 + (c0 >> 7)] = ss;
            epi_barrier_ws();
            if (p.counters) {
                // publish this tile's two slots, then wait (bounded) for the
                // other column tiles of the 128-row block
                unsigned int *cnt = p.counters + (m0 / kBM);
                if (warp == 2 && lane == 0) {
                    __threadfence();
                    atomicAdd(cnt, 2u);
                    *norm_ok = wait_count(cnt, (unsigned int)slots, abort_flag, p.watchdog,
                                          p.wait_limit_ns)
                                   ? 1
                                   : 0;
                }
                epi_barrier_ws();
                if (!*norm_ok) break;
                // inv of each row, formed once (warp half 0) from the row's
                // partials in column order and shared through shared memory
                if (c0 == 0 && live)
                    half_ss[row] = rsqrtf(row_sum(p.ss + t * slots, slots) / (float)p.H + p.eps);
                epi_barrier_ws();
                if (live)
                    er.store_y(half_ss[row], reinterpret_cast<const T *>(p.gamma) + ntile * NS + c0,
                               reinterpret_cast<T *>(p.y) + t * p.ldy + ntile * NS + c0);
            }
        }
    }
    tmem_fence_before();
    __syncthreads();
    // after an abort anywhere in the CTA, the fills the producer issued land
    // before the CTA's memory goes away (bounded)
    if (warp == 0 && lane == 0 && *abort_flag) {
        for (int64_t k = kit - S > 0 ? kit - S : 0; k < kit; ++k)
            wait_phase(smem_u32(&full[k % S]), (uint32_t)((k / S) & 1), abort_flag, p.watchdog,
                       p.wait_limit_ns, true);
    }
    __syncthreads();
    tmem_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Kernel 1, persistent, two SMs per tile (a cluster of two CTAs, tcgen05
// cta_group::2).  The pair computes a [256 x 256] tile of P with M = 256,
// N = 256 MMAs issued by the even CTA (the leader): each CTA stages its own
// 128 rows of A and its own 128 of the tile's 256 columns of W, and the
// matrix unit of each SM reads the A rows of its own CTA and both CTAs'
// halves of W, accumulating its 128 rows x 256 columns in its own tensor
// memory.  Per SM that halves the W bytes written into and read out of
// shared memory (and fetched from L2) against the one-SM kernel above, where
// a 128 x 256 x 64 slab moves 48 KB through shared memory per 128 x 256 x 64
// of work; here it is 32 KB.
//
// Signalling: both CTAs' TMA fills complete on the leader's full barrier
// (cta_group::2 copies may signal the peer's barrier); the leader arms it
// with both halves' bytes.  The leader's MMA commits arrive on the empty
// barrier of both CTAs (multicast), and on both CTAs' accumulator-full
// barrier; every epilogue thread of both CTAs arrives on the leader's
// accumulator-empty barrier.  The epilogue is the one-SM persistent
// kernel's, on the CTA's own 128 rows.
// ---------------------------------------------------------------------------
constexpr int kPairBM = 2 * kBM;  // rows of a pair tile

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of the variable at shared::cta address `a` in the
// cluster's CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// Every thread of both CTAs (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// 2-D TMA tile load into this CTA's shared memory whose completion is
// signalled on `bar`, a shared::cluster address in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int c0,
                                                 int c1, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at shared::cta offset `bar` in every CTA of `mask`
// once all pair MMAs this thread issued so far complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// Instruction descriptor of the pair MMA: as instr_desc, M = 256.
template <typename T, int N_>
__host__ __device__ constexpr uint32_t instr_desc_pair() {
    static_assert(N_ % 16 == 0 && N_ >= 32 && N_ <= 256, "M = 256 takes N = 32 .. 256");
    constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(N_ >> 3) << 17) |
           ((uint32_t)(kPairBM >> 4) << 24);
}

// An item of the pair kernel: a whole 256 x 256 tile or, for the tiles of
// the last partial round, one 128-column half of a tile (so that round fills
// up to twice as many SM pairs for half as long).
struct PairItem {
    int64_t tile;
    int col0;   // first column within the tile
    int ncols;  // 256 or 128
};

__device__ __forceinline__ PairItem pair_item(int64_t item, int64_t full_items) {
    if (item < full_items) return PairItem{item, 0, kMmaN};
    const int64_t h = item - full_items;
    return PairItem{full_items + h / 2, (int)(h & 1) * (kMmaN / 2), kMmaN / 2};
}

// A whole item of the pair kernel whose y waits for the next round (its
// 256-row block has items there): its epilogue writes h and publishes its
// partial sums as usual, and its y is formed during the pair's next item, so
// that the wait for the rest of the row block does not hold up the next
// accumulator.  m0 < 0: none.
struct PairPending {
    int64_t m0;  // first row of this CTA's 128-row block
    int ntile;   // column tile
    int gbuf;    // shared-memory gamma buffer holding its columns
};

// Warp 2 copies the item's gamma columns (16 bytes a lane) into shared memory.
template <typename T>
__device__ __forceinline__ void stage_gamma(const Params &p, const PairItem &pi, int ntile,
                                            uint32_t dst) {
    static_assert(sizeof(T) == 2, "16-bit operands");
    const int lane = threadIdx.x & 31;
    if (lane * 8 < pi.ncols)
        sts128(dst + lane * 16,
               ld_keep(reinterpret_cast<const T *>(p.gamma) + ntile * kMmaN + pi.col0 + lane * 8));
}

// y = RN((h * inv) * gamma) for 8 columns, gamma from shared memory.
template <typename T>
__device__ __forceinline__ uint4 scale_smem(const uint4 &h, float inv, uint32_t g) {
    float f[8], w[8];
    DT<T>::unpack(h, f);
    DT<T>::unpack(lds128(g), w);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = (f[e] * inv) * w[e];
    return DT<T>::pack(f);
}

// y for NC columns of this thread's row from h held in `er` (after run()).
template <typename T, int NC, bool Wide>
__device__ __forceinline__ void store_y_smem(const EpiRow<T, NC, Wide> &er, float inv,
                                             uint32_t g, T *y) {
    [[maybe_unused]] const uint64_t pol = l2_evict_first_policy();
#pragma unroll
    for (int q = 0; q < EpiRow<T, NC, Wide>::kPacks; ++q) {
        if constexpr (Wide)
            st_global32(y + 16 * q, scale_smem<T>(er.rv[q].a, inv, g + 32 * q),
                        scale_smem<T>(er.rv[q].b, inv, g + 32 * q + 16), pol);
        else
            st_global(y + 8 * q, scale_smem<T>(er.rv[q], inv, g + 16 * q));
    }
}

// y for NC columns of this thread's row from h re-read from global memory
// (this thread's own earlier stores), a few packs in flight at a time.
template <typename T, int NC, bool Wide>
__device__ __forceinline__ void store_y_reload(const T *h, float inv, uint32_t g, T *y) {
    constexpr int kPacks = EpiRow<T, NC, Wide>::kPacks;
    constexpr int kGroup = Wide ? 4 : 8;
    static_assert(kPacks % kGroup == 0, "whole groups");
    [[maybe_unused]] const uint64_t pol = l2_evict_first_policy();
#pragma unroll
    for (int q0 = 0; q0 < kPacks; q0 += kGroup) {
        typename EpiRow<T, NC, Wide>::Pk v[kGroup];
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
            if constexpr (Wide)
                v[q] = ld_stream32(h + 16 * (q0 + q), pol);
            else
                v[q] = ld_stream(h + 8 * (q0 + q));
        }
#pragma unroll
        for (int q = 0; q < kGroup; ++q) {
            if constexpr (Wide)
                st_global32(y + 16 * (q0 + q), scale_smem<T>(v[q].a, inv, g + 32 * (q0 + q)),
                            scale_smem<T>(v[q].b, inv, g + 32 * (q0 + q) + 16), pol);
            else
                st_global(y + 8 * (q0 + q), scale_smem<T>(v[q], inv, g + 16 * (q0 + q)));
        }
    }
}

// Waits (bounded, one thread) until the counter of the 128-row block at m0
// shows every column published, then leaves inv of each of its rows in
// rinv[row] (warp half 0 forms it; both halves read it).  Returns false when
// the wait gave up.
__device__ __forceinline__ bool block_inv(const Params &p, int64_t m0, float *rinv,
                                          volatile int *norm_ok, volatile int *abort_flag) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slots = 2 * p.C;
    if (warp == 2 && lane == 0)
        *norm_ok = wait_count(p.counters + (m0 / kBM), (unsigned int)slots, abort_flag,
                              p.watchdog, p.wait_limit_ns)
                       ? 1
                       : 0;
    epi_barrier_ws();
    if (!*norm_ok) return false;
    const int row = (warp & 3) * 32 + lane;
    const int64_t t = m0 + row;
    if (warp < 2 + kWsEpiWarps / 2 && t < p.T)
        rinv[row] = rsqrtf(row_sum(p.ss + t * slots, slots) / (float)p.H + p.eps);
    epi_barrier_ws();
    return true;
}

// The pair kernel's epilogue for one item, in one CTA (8 warps): NC columns
// per warp half (128 for a whole tile, 64 for a half).  Order: the
// accumulator is read and released, the partial sums published (the rest of
// the row block may be waiting on them), h stored, the y of a deferred
// earlier item written, and then this item's y -- or, when its row block
// ends in the next round and the pair has a next item, this item is
// deferred in turn.  Returns 0 when a wait gave up (the epilogue stops), 1
// otherwise.
template <typename T, int NC, bool Wide>
__device__ __forceinline__ int pair_epilogue(const Params &p, void *residual, int64_t ldr,
                                             const PairItem &pi, int it, int64_t item,
                                             int64_t npairs, int64_t items, int64_t m0,
                                             uint32_t tbase, uint64_t *tfull, uint64_t *tempty,
                                             volatile int *tile_ok, volatile int *norm_ok,
                                             float *half_ss, uint32_t gam0, PairPending &pend,
                                             volatile int *abort_flag) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wh = (warp - 2) >> 2;  // warp half
    const int acc = it & 1;
    const int ntile = (int)(pi.tile % p.C);
    const int slots = 2 * p.C;  // 128-column partial sums per row
    const int row = (warp & 3) * 32 + lane;
    const int64_t t = m0 + row;
    const bool live = t < p.T;
    const int c0 = pi.col0 + wh * NC;  // this warp half's first column in the tile
    constexpr uint32_t kGamBytes = kMmaN * 2;
    // three gamma buffers: warp 2 stages this item's columns before the
    // item's first barrier, while the other warps may still be forming the
    // y of the two items before it (a deferred one among them)
    const uint32_t gam = gam0 + (uint32_t)(it % 3) * kGamBytes;
    T *res = reinterpret_cast<T *>(residual) + (live ? t : 0) * ldr + ntile * kMmaN + c0;
    if (p.counters && warp == 2) stage_gamma<T>(p, pi, ntile, gam);
    // this thread's residual columns are loaded before the wait for the
    // accumulator, so they arrive while the item's MMAs run
    EpiRow<T, NC, Wide> er;
    if (live) er.load(res);
    // one thread waits (bounded) and the 8 warps leave together
    if (warp == 2 && lane == 0)
        *tile_ok = wait_phase(smem_u32(&tfull[acc]), (uint32_t)((it >> 1) & 1), abort_flag,
                              p.watchdog, p.wait_limit_ns)
                       ? 1
                       : 0;
    epi_barrier_ws();
    if (!*tile_ok) return 0;
    tmem_fence_after();
    if (item + npairs >= items) grid_launch_dependents();
    const float ss = er.run(tbase + wh * NC, live);
    tmem_fence_before();
    // this CTA's half of the accumulator is read: tell the leader
    mbar_arrive_remote(map_to_rank(smem_u32(&tempty[acc]), 0));
    const int slot = ntile * 2 + (c0 >> 7);
    if (NC == 128) {
        if (live && !*abort_flag) p.ss[t * slots + slot] = ss;
    } else {
        // both warp halves fill one slot: added in column order
        half_ss[(warp - 2) * 32 + lane] = ss;
        epi_barrier_ws();
        if (wh == 0 && live && !*abort_flag)
            p.ss[t * slots + slot] = ss + half_ss[(warp + 2) * 32 + lane];
    }
    epi_barrier_ws();
    if (p.counters && warp == 2 && lane == 0) {
        // publish this item's slots (the counter of its 128-row block)
        __threadfence();
        atomicAdd(p.counters + (m0 / kBM), (unsigned int)(pi.ncols >> 7));
    }
    // h stored only now, off the accumulator's and the row block's paths
    if (live) er.store_h(res);
    if (!p.counters) return 1;
    if (pend.m0 >= 0) {
        // the deferred whole item: its row block ended in this round of tiles
        if (!block_inv(p, pend.m0, half_ss, norm_ok, abort_flag)) return 0;
        const int64_t tp = pend.m0 + row;
        if (tp < p.T) {
            const int64_t col = (int64_t)pend.ntile * kMmaN + wh * 128;
            store_y_reload<T, 128, Wide>(reinterpret_cast<const T *>(residual) + tp * ldr + col,
                                         half_ss[row],
                                         gam0 + (uint32_t)pend.gbuf * kGamBytes + wh * 256,
                                         reinterpret_cast<T *>(p.y) + tp * p.ldy + col);
        }
        pend.m0 = -1;
    }
    if (item + npairs < items) {
        // the item index of the last tile of this 256-row block; the
        // block's tiles of the last partial round run as two halves each
        const int64_t last = (pi.tile / p.C) * p.C + p.C - 1;
        const int64_t last_item =
            last < p.full_items ? last : p.full_items + 2 * (last - p.full_items) + 1;
        if (last_item / npairs > item / npairs) {
            pend = PairPending{m0, ntile, it % 3};
            return 1;
        }
    }
    if (!block_inv(p, m0, half_ss, norm_ok, abort_flag)) return 0;
    if (live)
        store_y_smem<T, NC, Wide>(er, half_ss[row], gam + (uint32_t)(wh * NC) * 2,
                                  reinterpret_cast<T *>(p.y) + t * p.ldy + ntile * kMmaN + c0);
    return 1;
}

// AT: K slabs of BK elements per ring stage (each a 128-byte-swizzled atom of
// the operand, the next atom 16 KB further on).
template <int BK = 64, int AT = 1>
struct PairLayout {
    static constexpr int atom_a = kBM * BK * 2;            // 16 KB: this CTA's 128 rows of A
    static constexpr int atom_b = (kMmaN / 2) * BK * 2;    // 16 KB: its 128 columns of W
    static constexpr int a_bytes = AT * atom_a;
    static constexpr int b_bytes = AT * atom_b;
    static constexpr int stage_bytes = a_bytes + b_bytes;  // AT x 32 KB
    // 192 KB of the 227 KB: with one K slab per stage, 6 stages measured
    // faster than the 7 that fit (T = K = H = 4096 98.5 -> 96.3 us,
    // [8192, 4096, 4096] 170.6 -> 167.5, [16384, 5120, 5120] 506 -> 499.6;
    // 5 stages: 97.3, 168, 505.5; 4: 104.5); with AT slabs, 6 / AT stages
    static constexpr int stages = 6 / AT;
    static constexpr int ctl_off = stages * stage_bytes;
    // full[S], empty[S], tfull[2], tempty[2], mma_done (8 B each); tmem slot,
    // abort word, the peer's fill count, tile_ok, norm_ok; the epilogue's
    // half-row sums (and each row's inv)
    static constexpr int words_off = ctl_off + (2 * stages + 5) * 8;
    static constexpr int half_off = words_off + 32;
    // three buffers of one tile's gamma columns (items rotate)
    static constexpr int gam_off = (half_off + kWsEpiWarps * 32 * 4 + 15) / 16 * 16;
    static constexpr int total = gam_off + 3 * kMmaN * 2 + 1024;
    static_assert(total <= 227 * 1024, "one CTA per SM");
};

template <typename T, int BK, bool Wide, int AT = 1>
__global__ void __launch_bounds__(kWsThreads, 1)
    k_gemm_res_pair(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ CUtensorMap map_w_half, void *residual, int64_t ldr,
                    Params p) {
    static_assert(BK == 64, "K slab of 128 bytes");
    using Lay = PairLayout<BK, AT>;
    constexpr int S = Lay::stages;
    constexpr int NS = kMmaN;  // columns of a tile
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::ctl_off);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *words = reinterpret_cast<uint32_t *>(smem + Lay::words_off);
    uint32_t *tmem_slot = words;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(words + 1);
    volatile uint32_t *peer_kit = words + 2;  // leader: fills the peer issued (set at the end)
    volatile int *tile_ok = reinterpret_cast<volatile int *>(words + 3);
    volatile int *norm_ok = reinterpret_cast<volatile int *>(words + 4);
    float *half_ss = reinterpret_cast<float *>(smem + Lay::half_off);  // [8 warps][32]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();  // 0: leader (issues the MMAs)
    const int C = p.C;
    const int64_t items = p.items;
    const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int KB = (p.kblocks + AT - 1) / AT;  // ring fills per item

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);   // the leader's producer arms it
            mbar_init(smem_u32(&empty[s]), 1);  // the leader's MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 2 * 32 * kWsEpiWarps);  // both CTAs' epilogues
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        *peer_kit = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {  // one warp of each CTA allocates, together, the same columns in both
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
    tmem_fence_after();
    // a pair allocation takes the same columns in both CTAs: both use the
    // address the leader's allocation reported
    const uint32_t tmem = ld_cluster_u32(map_to_rank(smem_u32(tmem_slot), 0));
    grid_dependency_wait();  // A, W and the residual may come from the previous kernel

    int64_t kit = 0;  // producer: k-slabs issued so far (all items)
    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer (both CTAs) ----
            bool stop = false;
            uint32_t s = 0, ph = 0;
            const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty), ring0 = smem_u32(smem);
            const uint32_t lead_full0 = map_to_rank(full0, 0);
            const uint64_t pol = l2_evict_last_policy();
            for (int64_t item = pair; item < items && !stop; item += npairs) {
                const PairItem pi = pair_item(item, p.full_items);
                const int m0 = (int)((pi.tile / C) * kPairBM + rank * kBM);
                // this CTA's W rows: its half of the item's columns
                const int n0 = (int)((pi.tile % C) * NS + pi.col0 + rank * (pi.ncols / 2));
                const CUtensorMap *mw = pi.ncols == NS ? &map_w : &map_w_half;
                const uint32_t bytes = 2 * AT * (Lay::atom_a + pi.ncols / 2 * BK * 2);
                for (int kb = 0; kb < KB; ++kb, ++kit) {
                    if (kit >= S && !wait_phase(empty0 + 8 * s, ph ^ 1u, abort_flag, p.watchdog,
                                                p.wait_limit_ns)) {
                        stop = true;
                        break;
                    }
                    if (rank == 0)
                        mbar_arrive_expect_tx(
                            full0 + 8 * s, bytes + (blockIdx.x == 0 && kit == p.stall_fill ? 16u : 0u));
                    const uint32_t lead_fb = lead_full0 + 8 * s;
                    const uint32_t sa = ring0 + s * Lay::stage_bytes;
#pragma unroll
                    for (int at = 0; at < AT; ++at) {  // K slabs past K read as zeros
                        const int kx = (kb * AT + at) * BK;
                        tma_load_2d_pair(sa + at * Lay::atom_a, &map_a, kx, m0, lead_fb, pol);
                        tma_load_2d_pair(sa + Lay::a_bytes + at * Lay::atom_b, mw, kx, n0,
                                         lead_fb, pol);
                    }
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---- MMA issuer (leader only) ----
            const uint32_t idesc_full = instr_desc_pair<T, NS>();
            const uint32_t idesc_half = instr_desc_pair<T, NS / 2>();
            const uint64_t adesc0 = smem_desc(smem_u32(smem), BK * 2);
            const uint64_t bdesc0 = smem_desc(smem_u32(smem) + Lay::a_bytes, BK * 2);
            constexpr uint32_t kStageDesc = Lay::stage_bytes >> 4;
            const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
            uint32_t s = 0, ph = 0;
            int it = 0;
            bool stop = false;
            for (int64_t item = pair; item < items && !stop; item += npairs, ++it) {
                const int acc = it & 1;
                const uint32_t idesc = item < p.full_items ? idesc_full : idesc_half;
                if (it >= 2 &&
                    !wait_phase<true>(smem_u32(&tempty[acc]), (uint32_t)(((it >> 1) - 1) & 1),
                                      abort_flag, p.watchdog, p.wait_limit_ns))
                    break;
                tmem_fence_after();
                const uint32_t d = tmem + acc * NS;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase(full0 + 8 * s, ph, abort_flag, p.watchdog, p.wait_limit_ns)) {
                        stop = true;
                        break;
                    }
                    tmem_fence_after();
                    const uint64_t ad = adesc0 + s * kStageDesc, bd = bdesc0 + s * kStageDesc;
                    mma_f16_pair(d, ad, bd, idesc, kb != 0);
#pragma unroll
                    for (int kk = 1; kk < BK / kMmaK; ++kk)
                        mma_f16_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
#pragma unroll
                    for (int at = 1; at < AT; ++at) {
                        const uint64_t aa = ad + (at * Lay::atom_a >> 4);
                        const uint64_t ba = bd + (at * Lay::atom_b >> 4);
#pragma unroll
                        for (int kk = 0; kk < BK / kMmaK; ++kk)
                            mma_f16_pair(d, aa + 2 * kk, ba + 2 * kk, idesc, 1u);
                    }
                    mma_commit_pair(empty0 + 8 * s, 3);  // frees the stage in both CTAs
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!stop) mma_commit_pair(smem_u32(&tfull[acc]), 3);
            }
            // every MMA issued has completed before tensor memory is freed
            mma_commit_pair(smem_u32(mma_done), 1);
            wait_phase(smem_u32(mma_done), 0, abort_flag, p.watchdog, p.wait_limit_ns, true);
        }
        __syncwarp();
    } else {
        // ---- epilogue: warps 2-9 of both CTAs, each on its CTA's 128 rows;
        // warp half (warp - 2) / 4 takes half of the item's columns ----
        int it = 0;
        PairPending pend{-1, 0, 0};
        const uint32_t gam0 = smem_u32(smem + Lay::gam_off);
        for (int64_t item = pair; item < items; item += npairs, ++it) {
            const PairItem pi = pair_item(item, p.full_items);
            const int64_t m0 = (pi.tile / C) * kPairBM + rank * kBM;
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + (it & 1) * NS;
            const int ok =
                pi.ncols == NS
                    ? pair_epilogue<T, NS / 2, Wide>(p, residual, ldr, pi, it, item, npairs, items,
                                                     m0, tbase, tfull, tempty, tile_ok, norm_ok,
                                                     half_ss, gam0, pend, abort_flag)
                    : pair_epilogue<T, NS / 4, Wide>(p, residual, ldr, pi, it, item, npairs, items,
                                                     m0, tbase, tfull, tempty, tile_ok, norm_ok,
                                                     half_ss, gam0, pend, abort_flag);
            if (!ok) break;
        }
    }
    tmem_fence_before();
    __syncthreads();
    // the peer's fill count reaches the leader before the cluster barrier
    if (warp == 0 && lane == 0 && rank == 1)
        st_cluster_u32(map_to_rank(smem_u32((const void *)peer_kit), 0), (uint32_t)kit);
    cluster_sync();
    // After an abort anywhere in the pair, every fill either CTA issued lands
    // before shared memory goes away: the leader's full barriers count both
    // halves, so the leader waits (bounded) on each fill still open, arming
    // with the peer's bytes any fill its own producer never reached.  Without
    // an abort every fill was consumed by a completed MMA and nothing waits.
    if (warp == 0 && lane == 0 && rank == 0) {
        const int64_t kp = *peer_kit;
        const int64_t kmax = kit > kp ? kit : kp;
        for (int64_t k = kmax - S > 0 ? kmax - S : 0; k < kmax; ++k) {
            const int s = (int)(k % S);
            if (k >= kit) {
                // the item of fill k: this pair's (k / KB)-th
                const PairItem pi = pair_item(pair + (k / KB) * npairs, p.full_items);
                mbar_arrive_expect_tx(smem_u32(&full[s]), AT * (Lay::atom_a + pi.ncols / 2 * BK * 2));
            }
            wait_phase(smem_u32(&full[s]), (uint32_t)((k / S) & 1), abort_flag, p.watchdog,
                       p.wait_limit_ns, true);
        }
    }
    tmem_fence_before();
    cluster_sync();
    tmem_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Split K for few rows (ceil(T / 128) row blocks whose tiles leave at least
// half of the SMs idle): with only M x H / 256 tiles the tiled kernels would
// stream the operands through as many SMs; here CTA (m, n, s) of an
// M x C x splits grid multiplies the K slabs of split s for row block m and
// column tile n (4-stage TMA ring, M = 128, N = 256 MMAs into TMEM, as
// k_gemm_res) and writes its binary32 partial products for the live rows.
// k_splitk_norm then adds the splits in order, adds the residual (one
// rounding), and normalises.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_splitk(const __grid_constant__ CUtensorMap map_a,
                  const __grid_constant__ CUtensorMap map_w, Params p) {
    constexpr int BK = 64, NS = kMmaN, S = 4;
    constexpr int kRowBytes = BK * 2;
    constexpr Layout L = layout(S, NS, BK);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.ctl_off);
    uint64_t *empty = full + S;
    uint64_t *accum = empty + S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1 + kMaxChunks);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mblocks = (int)((p.T + kBM - 1) / kBM);
    const int ntile = (int)(blockIdx.x % p.C);
    const int mblk = (int)((blockIdx.x / p.C) % mblocks);
    const int split = (int)(blockIdx.x / ((unsigned)p.C * mblocks));
    const int n0 = ntile * NS;
    const int kb0 = split * p.kb_per_split;
    const int kb1 = min(p.kblocks, kb0 + p.kb_per_split);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(accum), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(NS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // A and W may come from the previous kernel

    int issued = 0;  // producer: fills issued
    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        uint32_t s = 0, ph = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++issued) {
            if (issued >= S && !wait_phase(smem_u32(&empty[s]), ph ^ 1u, abort_flag, p.watchdog,
                                           p.wait_limit_ns))
                break;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(fb, (uint32_t)(p.a_rows * kRowBytes + L.b_bytes) +
                                          (blockIdx.x == 0 && issued == p.stall_fill ? 16u : 0u));
            const uint32_t sa = smem_u32(smem + s * L.stage_bytes);
            tma_load_2d(sa, &map_a, kb * BK, mblk * kBM, fb);
            tma_load_2d(sa + L.a_bytes, &map_w, kb * BK, n0, fb);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        const uint32_t idesc = instr_desc<T>();
        const uint64_t adesc0 = smem_desc(smem_u32(smem), kRowBytes);
        const uint64_t bdesc0 = smem_desc(smem_u32(smem) + L.a_bytes, kRowBytes);
        constexpr uint32_t kStageDesc = L.stage_bytes >> 4;
        uint32_t s = 0, ph = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_phase(smem_u32(&full[s]), ph, abort_flag, p.watchdog, p.wait_limit_ns))
                break;
            tmem_fence_after();
            const uint64_t ad = adesc0 + s * kStageDesc, bd = bdesc0 + s * kStageDesc;
            mma_f16(tmem, ad, bd, idesc, kb != kb0);
#pragma unroll
            for (int kk = 1; kk < BK / kMmaK; ++kk)
                mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
            mma_commit(smem_u32(&empty[s]));
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        mma_commit(smem_u32(accum));  // arrives once every MMA issued has completed
    }
    __syncwarp();

    // ---- epilogue: thread i = row i; live rows write their partial products ----
    wait_phase(smem_u32(accum), 0, abort_flag, p.watchdog, p.wait_limit_ns, true);
    tmem_fence_after();
    __syncthreads();
    const bool ok = !*abort_flag;
    grid_launch_dependents();
    const int64_t r = (int64_t)mblk * kBM + threadIdx.x;
    const uint32_t tbase = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float *dst = p.part + ((int64_t)split * p.T + r) * p.H + n0;
    for (int c = 0; c < NS; c += 32) {
        float v[32];
        tmem_ld32(tbase + c, v);  // warp-wide: every lane takes part
        if (ok && r < p.T) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 a = make_uint4(__float_as_uint(v[8 * q]), __float_as_uint(v[8 * q + 1]),
                                           __float_as_uint(v[8 * q + 2]),
                                           __float_as_uint(v[8 * q + 3]));
                const uint4 b = make_uint4(
                    __float_as_uint(v[8 * q + 4]), __float_as_uint(v[8 * q + 5]),
                    __float_as_uint(v[8 * q + 6]), __float_as_uint(v[8 * q + 7]));
                st_global32(dst + c + 8 * q, a, b);
            }
        }
    }
    if (threadIdx.x == 0 && *abort_flag) {
        // after an abort, the fills issued land before this CTA's memory goes
        // away (bounded)
        for (int k = issued - S > 0 ? issued - S : 0; k < issued; ++k)
            wait_phase(smem_u32(&full[k % S]), (uint32_t)((k / S) & 1), abort_flag, p.watchdog,
                       p.wait_limit_ns, true);
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NS)
                     : "memory");
    }
}

// The split-K sum and the fused residual-add RMSNorm: a CTA per row, VPT
// 8-column packs per thread.  P = ((p_0 + p_1) + ...) + p_{S-1} in binary32,
// h = RN(P + r) (one rounding), the residual updated, Σh² over the CTA, y from
// the h held in registers.
template <typename T, int VPT, int SMAX>
__global__ void __launch_bounds__(256) k_splitk_norm(NormParams q, const float *part, int splits,
                                                      void *residual) {
    __shared__ float red[32];
    const int nv = (int)(q.H / 8);
    const int64_t t = blockIdx.x;
    grid_dependency_wait();
    grid_launch_dependents();
    T *res = reinterpret_cast<T *>(residual) + t * q.ldh;
    uint4 hv[VPT];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = threadIdx.x + k * blockDim.x;
        if (j < nv) {
            float acc[8];
            const float *src = part + t * q.H + (int64_t)j * 8;
            // the pack's S <= SMAX partials loaded together (one round trip;
            // K = H = 4096: T = 1 11.3 -> 10.1 us, T = 16 9.7 -> 8.2, T = 128
            // 14.8 -> 13.3), then added in split order
            Pack32 v[SMAX];
#pragma unroll
            for (int s = 0; s < SMAX; ++s)
                if (s < splits) v[s] = ld_stream32(src + (int64_t)s * q.T * q.H);
            acc[0] = __uint_as_float(v[0].a.x), acc[1] = __uint_as_float(v[0].a.y);
            acc[2] = __uint_as_float(v[0].a.z), acc[3] = __uint_as_float(v[0].a.w);
            acc[4] = __uint_as_float(v[0].b.x), acc[5] = __uint_as_float(v[0].b.y);
            acc[6] = __uint_as_float(v[0].b.z), acc[7] = __uint_as_float(v[0].b.w);
#pragma unroll
            for (int s = 1; s < SMAX; ++s) {
                if (s < splits) {
                    acc[0] += __uint_as_float(v[s].a.x), acc[1] += __uint_as_float(v[s].a.y);
                    acc[2] += __uint_as_float(v[s].a.z), acc[3] += __uint_as_float(v[s].a.w);
                    acc[4] += __uint_as_float(v[s].b.x), acc[5] += __uint_as_float(v[s].b.y);
                    acc[6] += __uint_as_float(v[s].b.z), acc[7] += __uint_as_float(v[s].b.w);
                }
            }
            float f[8];
            DT<T>::unpack(ld_stream(res + (int64_t)j * 8), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                f[e] = DT<T>::round(acc[e] + f[e]);  // h: one rounding of P + r
                ss += f[e] * f[e];
            }
            hv[k] = DT<T>::pack(f);
            st_global(res + (int64_t)j * 8, hv[k]);
        }
    }
    const float inv = rsqrtf(block_sum(ss, red) / (float)q.H + q.eps);
    T *y = reinterpret_cast<T *>(q.y) + t * q.ldy;
    const T *g = reinterpret_cast<const T *>(q.gamma);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = threadIdx.x + k * blockDim.x;
        if (j < nv) {
            float f[8], w[8];
            DT<T>::unpack(hv[k], f);
            DT<T>::unpack(ld_keep(g + (int64_t)j * 8), w);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = (f[e] * inv) * w[e];
            st_global(y + (int64_t)j * 8, DT<T>::pack(f));
        }
    }
}

// The same for very few rows: a cluster of kSplitNormCS CTAs per row, CTA c
// taking the row's packs [c P, (c + 1) P), P = H / 8 / kSplitNormCS, one per
// thread; each CTA's sum of squares (block order) goes to its shared memory
// and every CTA adds the cluster's in rank order (distributed shared memory)
// before writing y.  With one row, one CTA would carry all of the row's
// S x H partials alone.
constexpr int kSplitNormCS = 8;

template <typename T, int SMAX>
__global__ void __launch_bounds__(256) k_splitk_norm_cluster(NormParams q, const float *part,
                                                              int splits, void *residual) {
    __shared__ float red[32];
    __shared__ float seg_ss;
    const uint32_t rank = cluster_rank();
    const int64_t t = blockIdx.x / kSplitNormCS;
    const int per = (int)(q.H / 8 / kSplitNormCS);  // packs per CTA
    const int j = (int)rank * per + (int)threadIdx.x;
    const bool act = (int)threadIdx.x < per;
    grid_dependency_wait();
    grid_launch_dependents();
    T *res = reinterpret_cast<T *>(residual) + t * q.ldh;
    uint4 hv = make_uint4(0u, 0u, 0u, 0u);
    float ss = 0.f;
    if (act) {
        const float *src = part + t * q.H + (int64_t)j * 8;
        Pack32 v[SMAX];
#pragma unroll
        for (int s = 0; s < SMAX; ++s)
            if (s < splits) v[s] = ld_stream32(src + (int64_t)s * q.T * q.H);
        float acc[8];
        acc[0] = __uint_as_float(v[0].a.x), acc[1] = __uint_as_float(v[0].a.y);
        acc[2] = __uint_as_float(v[0].a.z), acc[3] = __uint_as_float(v[0].a.w);
        acc[4] = __uint_as_float(v[0].b.x), acc[5] = __uint_as_float(v[0].b.y);
        acc[6] = __uint_as_float(v[0].b.z), acc[7] = __uint_as_float(v[0].b.w);
#pragma unroll
        for (int s = 1; s < SMAX; ++s) {
            if (s < splits) {
                acc[0] += __uint_as_float(v[s].a.x), acc[1] += __uint_as_float(v[s].a.y);
                acc[2] += __uint_as_float(v[s].a.z), acc[3] += __uint_as_float(v[s].a.w);
                acc[4] += __uint_as_float(v[s].b.x), acc[5] += __uint_as_float(v[s].b.y);
                acc[6] += __uint_as_float(v[s].b.z), acc[7] += __uint_as_float(v[s].b.w);
            }
        }
        float f[8];
        DT<T>::unpack(ld_stream(res + (int64_t)j * 8), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            f[e] = DT<T>::round(acc[e] + f[e]);  // h: one rounding of P + r
            ss += f[e] * f[e];
        }
        hv = DT<T>::pack(f);
        st_global(res + (int64_t)j * 8, hv);
    }
    const float mine = block_sum(ss, red);
    if (threadIdx.x == 0) seg_ss = mine;
    cluster_sync();  // every CTA's sum is in its shared memory
    float tot = 0.f;
#pragma unroll
    for (int c = 0; c < kSplitNormCS; ++c)
        tot += __uint_as_float(ld_cluster_u32(map_to_rank(smem_u32(&seg_ss), (uint32_t)c)));
    const float inv = rsqrtf(tot / (float)q.H + q.eps);
    if (act) {
        float f[8], w[8];
        DT<T>::unpack(hv, f);
        DT<T>::unpack(ld_keep(reinterpret_cast<const T *>(q.gamma) + (int64_t)j * 8), w);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = (f[e] * inv) * w[e];
        st_global(reinterpret_cast<T *>(q.y) + t * q.ldy + (int64_t)j * 8, DT<T>::pack(f));
    }
    cluster_sync();  // no CTA leaves while another still reads its sum
}

// Zeroes the row-block counters of the norm in the persistent kernels'
// epilogue, after the previous kernel on the stream (which may be the previous
// call's GEMM, still counting) has finished.  The GEMM may launch at once (its
// prologue overlaps this kernel): its own wait for this grid covers these
// stores, and this grid ends only after the previous kernel has.
static __global__ void __launch_bounds__(256) k_zero_counters(unsigned int *cnt, int64_t n) {
    grid_launch_dependents();
    grid_dependency_wait();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) cnt[i] = 0u;
}

// Kernel 2: y from the stored h and the column blocks' partial sums.  A warp
// per (row, slice of up to 32 * VPT 16-byte packs): it loads its slice of h
// and the row's C partials at once, forms inv from the partials summed in
// column order (the same value in every slice of the row) and writes its
// slice of y.  No barrier: every warp works alone, grid-stride over items.
constexpr int kNormVPT = 4;
constexpr int kNormThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kNormThreads) k_norm_ss(NormParams p) {
    constexpr int EPV = DT<T>::EPV;
    constexpr int SLICE = 32 * kNormVPT;  // packs per item
    const int nv = (int)(p.H / EPV);
    const int slices = (nv + SLICE - 1) / SLICE;
    const int64_t items = p.T * slices;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * kNormThreads) >> 5;
    const T *g = reinterpret_cast<const T *>(p.gamma);
    grid_dependency_wait();  // kernel 1's stores are visible
    for (int64_t item = ((int64_t)blockIdx.x * kNormThreads + threadIdx.x) >> 5; item < items;
         item += nwarps) {
        if (item + nwarps >= items) grid_launch_dependents();
        const int64_t t = item / slices;
        const int j0 = (int)(item % slices) * SLICE;
        const T *h = reinterpret_cast<const T *>(p.h) + t * p.ldh;
        uint4 hv[kNormVPT];
#pragma unroll
        for (int k = 0; k < kNormVPT; ++k) {
            const int j = j0 + lane + 32 * k;
            if (j < nv) hv[k] = ld_stream(h + (int64_t)j * EPV);
        }
        // lanes q and q + 32 hold partials q and q + 32 (C <= 64); every lane
        // adds them in column order
        const float part0 = lane < p.C ? p.ss[t * p.C + lane] : 0.f;
        const float part1 = lane + 32 < p.C ? p.ss[t * p.C + lane + 32] : 0.f;
        float tot = 0.f;
        for (int q = 0; q < p.C; ++q)
            tot += __shfl_sync(0xffffffffu, q < 32 ? part0 : part1, q & 31);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        T *y = reinterpret_cast<T *>(p.y) + t * p.ldy;
#pragma unroll
        for (int k = 0; k < kNormVPT; ++k) {
            const int j = j0 + lane + 32 * k;
            if (j < nv) {
                float f[EPV], w[EPV];
                DT<T>::unpack(hv[k], f);
                DT<T>::unpack(ld_keep(g + (int64_t)j * EPV), w);
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = (f[e] * inv) * w[e];
                st_global(y + (int64_t)j * EPV, DT<T>::pack(f));
            }
        }
    }
}

}  // namespace gemm

}  // namespace rarn
