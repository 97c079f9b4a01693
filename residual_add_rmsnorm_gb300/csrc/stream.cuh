// stream.cuh -- persistent, warp-specialised kernel fed by TMA bulk copies.
//
// One CTA per SM walks rows t = blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 0 is the producer: one elected lane issues cp.async.bulk copies of each
// row's input streams (x; or the R partials and the residual) in chunks of
// 256 x PPT x 16 bytes per stream into a ring of shared-memory stages, each stage
// guarded by a "full" mbarrier (completed by the copies' byte count) and an
// "empty" mbarrier (released by the consumer warps).  The producer runs ahead
// across row boundaries, so HBM reads stay in flight while the consumers
// reduce and normalise.
//
// Warps 1.. are the consumers: G groups of 8 warps (256 threads); group g
// takes the CTA's rows i = g, g + G, ... so that while one group reduces and
// normalises its row the next group already consumes the following row's
// chunks.  For chunk c of a row, thread j of the group takes pack
// p = c * 256 + j: it sums the streams' packs in stream order in
// binary32, rounds once, writes the residual pack to global memory, keeps the
// rounded pack in a shared-memory copy of the row and accumulates its
// squares.  After the row's last chunk a named barrier combines the group's
// warps' sums; each thread then normalises the packs it staged itself (same
// p, so no further synchronisation) with gamma and writes y.  HBM is read
// exactly once per input element.
//
// Every wait is bounded (see wait_bounded): on a timeout the kernel records a
// bit in the watchdog word, stops issuing copies, drains the copies already
// issued and returns.  Consumer warps keep executing the same named barriers
// so that none is left waiting, and release only stages whose fills they saw
// complete.
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rarn {
namespace stream {

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy primitives (inline PTX)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
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

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Global -> shared bulk copy, completion signalled on `bar` by byte count.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Wait for the phase of `bar` with parity `parity`.  Gives up after
// `limit_ns` (or at once if another thread of the CTA already gave up): sets
// the CTA's abort word and the watchdog bit, returns false.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int *abort_flag, unsigned int *watchdog,
                                             unsigned int bit, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    unsigned long long t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            const unsigned long long now = global_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(watchdog, bit);
                return false;
            }
        }
    }
}

// Drain wait used by the producer before it exits: ignores the abort word
// (copies already issued must land before the CTA's memory goes away) and
// gives up at `deadline` (one deadline for the whole drain).
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity,
                                           unsigned long long deadline, unsigned int *watchdog) {
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() > deadline) {
            atomicOr(watchdog, kWatchProducer);
            return false;
        }
    }
    return true;
}

// Barrier over one consumer group's 256 threads (ids 1.. ; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kConsumers) : "memory");
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Row k of this CTA (t = blockIdx.x + k * gridDim.x) goes to consumer group
// g = k % G and through g's own ring of `stages` stages.  Each ring has one
// producer and one consumer group taking its fills in the same order, so a
// parity wait is never more than one phase ahead of its barrier: fill n of a
// ring lands in stage n % stages during that stage's phase n / stages, and
// fill n - stages of the same stage was consumed before fill n is waited on.
//
// A chunk is 256 * PPT packs of every input stream; consumer thread j takes
// packs c * 256 * PPT + m * 256 + j (m < PPT), i.e. over the whole row the
// packs j, j + 256, j + 512, ... -- the same packs it normalises later.
template <typename T, int OP, int G, int PPT>
__global__ void __launch_bounds__(threads(G), 1) k_stream(Problem p, int stages) {
    constexpr int EPV = DT<T>::EPV;
    constexpr int CP = kConsumers * PPT;      // packs per chunk
    constexpr int CB = CP * kPackBytes;       // bytes per stream per chunk
    extern __shared__ __align__(128) unsigned char smem[];
    const int ns = OP == OP_PLAIN ? 1 : p.R + 1;  // input streams
    const int row_bytes = (int)(p.H * (int64_t)sizeof(T));
    const int nv = row_bytes / kPackBytes;        // packs per row
    const int nchunks = (nv + CP - 1) / CP;
    const Layout L = layout(stages, ns, row_bytes, G, CB);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.ctl_off);   // [G][stages]
    uint64_t *empty = full + kMaxStages;                                // [G][stages]
    float *red_all = reinterpret_cast<float *>(empty + kMaxStages);  // [G][2][kConsumerWarps]
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(red_all + G * 2 * kConsumerWarps);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the first row's streams prefetched into L2 before the wait (L2 is the
    // point of coherence: correct while the previous kernel still writes them)
    if (p.l2_rows > 0 && threadIdx.x < ns && (int64_t)blockIdx.x < p.T) {
        const int64_t t = blockIdx.x;
        const T *src = reinterpret_cast<const T *>(p.src);
        const void *row = threadIdx.x < ns - (OP == OP_PLAIN ? 0 : 1)
                              ? static_cast<const void *>(src + threadIdx.x * p.slice + t * p.ldx)
                              : static_cast<const void *>(reinterpret_cast<const T *>(p.residual) +
                                                          t * p.ldr);
        prefetch_l2(row, (uint32_t)row_bytes);
    }
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        for (int s = 0; s < G * stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), kConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        long long issued0 = 0, issued1 = 0;  // fills issued into ring 0 / ring 1
        const long long stall_at = blockIdx.x == 0 ? p.stall_fill : -1;
        bool ok = true;
        int g = 0;
        for (int64_t t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
            const int64_t xrow = t * p.ldx, rrow = t * p.ldr;
            long long &n = g == 0 ? issued0 : issued1;
            for (int c = 0; c < nchunks && ok; ++c, ++n) {
                const int packs = min(CP, nv - c * CP);
                const uint32_t bytes = (uint32_t)packs * kPackBytes;
                const int st = (int)(n % stages);
                const uint32_t ph = (uint32_t)((n / stages) & 1);
                const int b = g * stages + st;
                ok = wait_bounded(smem_addr(&empty[b]), ph ^ 1u, abort_flag, p.watchdog,
                                  kWatchProducer, p.wait_limit_ns);
                if (!ok) break;
                const uint32_t fb = smem_addr(&full[b]);
                // test hook: expect 16 bytes more than the copies bring, so that
                // this fill never completes and its consumers' wait runs out
                const uint32_t extra = issued0 + issued1 == stall_at ? 16u : 0u;
                mbar_arrive_expect_tx(fb, bytes * (uint32_t)ns + extra);
                const uint32_t dst =
                    smem_addr(smem + (size_t)g * L.ring_stride + (size_t)st * ns * CB);
                const int64_t off = (int64_t)c * CP * EPV;
                for (int s = 0; s < ns; ++s) {
                    const T *src;
                    if (OP != OP_PLAIN && s == ns - 1)
                        src = reinterpret_cast<const T *>(p.residual) + rrow + off;
                    else
                        src = reinterpret_cast<const T *>(p.src) + (int64_t)s * p.slice + xrow +
                              off;
                    bulk_g2s(dst + (uint32_t)(s * CB), src, bytes, fb);
                }
            }
            if (++g == G) g = 0;
        }
        grid_launch_dependents();
        // Drain: in every ring the last min(stages, issued) fills must land
        // before the CTA exits (one deadline for all of them; after it, each
        // remaining fill is still checked once).
        const unsigned long long deadline = global_ns() + p.wait_limit_ns;
        for (int r = 0; r < G; ++r) {
            const long long issued = r == 0 ? issued0 : issued1;
            const long long first = issued > stages ? issued - stages : 0;
            for (long long f = first; f < issued; ++f)
                wait_drain(smem_addr(&full[r * stages + (int)(f % stages)]),
                           (uint32_t)((f / stages) & 1), deadline, p.watchdog);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = (warp - 1) / kConsumerWarps;       // consumer group
    const int cw = (warp - 1) % kConsumerWarps;      // warp within the group
    const int j = threadIdx.x - 32 - g * kConsumers;  // 0..255 within the group
    unsigned char *ring = smem + (size_t)g * L.ring_stride;
    uint64_t *gfull = full + g * stages;
    uint64_t *gempty = empty + g * stages;
    uint4 *row_copy = reinterpret_cast<uint4 *>(smem + L.row_off + g * L.row_stride);
    float *red = red_all + g * 2 * kConsumerWarps;
    const T *gamma = reinterpret_cast<const T *>(p.gamma);
    T *residual = reinterpret_cast<T *>(p.residual);
    int stage = 0;
    uint32_t phase = 0;
    int par = 0;
    for (int64_t t = blockIdx.x + (int64_t)g * gridDim.x; t < p.T;
         t += (int64_t)G * gridDim.x, par ^= 1) {
        float ss = 0.f;
        if (t + (int64_t)G * gridDim.x >= p.T) grid_launch_dependents();
        for (int c = 0; c < nchunks; ++c) {
            const bool ok = wait_bounded(smem_addr(&gfull[stage]), phase, abort_flag, p.watchdog,
                                         kWatchConsumer, p.wait_limit_ns);
            const unsigned char *sbase = ring + (size_t)stage * ns * CB;
#pragma unroll
            for (int m = 0; m < PPT; ++m) {
                const int q = m * kConsumers + j;  // pack within the chunk
                const int pk = c * CP + q;         // pack within the row
                if (!ok || pk >= nv) continue;
                const unsigned char *sb = sbase + q * kPackBytes;
                uint4 hv;
                if (OP == OP_PLAIN) {
                    hv = *reinterpret_cast<const uint4 *>(sb);
                } else {
                    float acc[EPV];
                    DT<T>::unpack(*reinterpret_cast<const uint4 *>(sb), acc);
#pragma unroll 4
                    for (int s = 1; s < ns; ++s) {
                        float f2[EPV];
                        DT<T>::unpack(*reinterpret_cast<const uint4 *>(sb + s * CB), f2);
#pragma unroll
                        for (int e = 0; e < EPV; ++e) acc[e] = acc[e] + f2[e];
                    }
                    hv = DT<T>::pack(acc);  // the one rounding to the storage type
                    st_global(residual + t * p.ldr + (int64_t)pk * EPV, hv);
                }
                row_copy[pk] = hv;
                float h[EPV];
                DT<T>::unpack(hv, h);
#pragma unroll
                for (int e = 0; e < EPV; ++e) ss += h[e] * h[e];
            }
            __syncwarp();
            // Release the stage only if this warp saw its fill complete: after
            // an abort, a stage whose fill never completed stays held, so the
            // producer can never re-arm a full barrier inside an unfinished
            // phase (its own bounded wait then ends it).
            if (lane == 0 && ok) mbar_arrive(smem_addr(&gempty[stage]));
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // row sum of squares over the group's 8 warps
        ss = warp_sum(ss);
        if (lane == 0) red[par * kConsumerWarps + cw] = ss;
        named_barrier(1 + g);
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += red[par * kConsumerWarps + w];
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        if (*abort_flag) continue;
        T *y = reinterpret_cast<T *>(p.y) + t * p.ldy;
        for (int pk = j; pk < nv; pk += kConsumers) {
            float h[EPV], w[EPV];
            DT<T>::unpack(row_copy[pk], h);
            DT<T>::unpack(ld_keep(gamma + (int64_t)pk * EPV), w);
#pragma unroll
            for (int e = 0; e < EPV; ++e) h[e] = (h[e] * inv) * w[e];
            st_global(y + (int64_t)pk * EPV, DT<T>::pack(h));
        }
    }
}

}  // namespace stream

template <typename T, int OP, int G, int PPT>
static cudaError_t launch_stream_k(const Problem &p, const Plan &pl, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(stream::k_stream<T, OP, G, PPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    if (e != cudaSuccess) return e;
    e = launch_kernel(stream::k_stream<T, OP, G, PPT>, dim3(pl.grid), dim3(stream::threads(G)),
                      pl.smem, st, pl.pdl, 1, p, pl.stages);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, int OP, int G>
static cudaError_t launch_stream_g(const Problem &p, const Plan &pl, cudaStream_t st) {
    switch (pl.per_thread) {
    case 1: return launch_stream_k<T, OP, G, 1>(p, pl, st);
    case 2: return launch_stream_k<T, OP, G, 2>(p, pl, st);
    case 4: return launch_stream_k<T, OP, G, 4>(p, pl, st);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, int OP>
static cudaError_t launch_stream_op(const Problem &p, const Plan &pl, cudaStream_t st) {
    switch (pl.groups) {
    case 1: return launch_stream_g<T, OP, 1>(p, pl, st);
    case 2: return launch_stream_g<T, OP, 2>(p, pl, st);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_stream(const Problem &p, const Plan &pl, cudaStream_t st) {
    switch (p.op) {
    case OP_PLAIN: return launch_stream_op<T, OP_PLAIN>(p, pl, st);
    case OP_FUSED: return launch_stream_op<T, OP_FUSED>(p, pl, st);
    case OP_REDUCE: return launch_stream_op<T, OP_REDUCE>(p, pl, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rarn
