// stream.cuh -- persistent, warp-specialised kernel fed by TMA bulk copies.
//
// One CTA per SM walks rows t = blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 0 is the producer: one elected lane issues cp.async.bulk copies of each
// row's input streams (x; or the R partials and the residual) in chunks of
// 256 x 16 bytes per stream into a ring of shared-memory stages, each stage
// guarded by a "full" mbarrier (completed by the copies' byte count) and an
// "empty" mbarrier (released by the consumer warps).  The producer runs ahead
// across row boundaries, so HBM reads stay in flight while the consumers
// reduce and normalise.
//
// Warps 1..8 are the consumers (256 threads).  For chunk c of a row, thread j
// takes pack p = c * 256 + j: it sums the streams' packs in stream order in
// binary32, rounds once, writes the residual pack to global memory, keeps the
// rounded pack in a shared-memory copy of the row and accumulates its
// squares.  After the row's last chunk a named barrier combines the consumer
// warps' sums; each thread then normalises the packs it staged itself (same
// p, so no further synchronisation) with gamma and writes y.  HBM is read
// exactly once per input element.
//
// Every wait is bounded (see wait_bounded): on a timeout the kernel records a
// bit in the watchdog word, stops issuing copies, drains the copies already
// issued and returns.  Consumer warps keep executing the same named barriers
// so that none is left waiting.
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rarn {
namespace stream {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;  // packs per chunk
constexpr int kThreads = kConsumers + 32;        // + producer warp
constexpr int kChunkBytes = kConsumers * 16;     // per stream per stage
constexpr int kMaxStages = 32;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned int kWatchConsumer = 1u, kWatchProducer = 2u;

// Dynamic shared memory layout (all offsets 128-byte aligned):
//   [0, stages * NS * kChunkBytes)    stage ring
//   row copy: H * sizeof(T) bytes
//   control: full[kMaxStages], empty[kMaxStages] mbarriers, red[2][8], abort
struct Layout {
    int stages, ns, row_bytes;
    int ring_off, row_off, ctl_off, total;
};

__host__ __device__ inline int align128(int v) { return (v + 127) & ~127; }

__host__ __device__ inline Layout layout(int stages, int ns, int row_bytes) {
    Layout L;
    L.stages = stages;
    L.ns = ns;
    L.row_bytes = row_bytes;
    L.ring_off = 0;
    L.row_off = align128(stages * ns * kChunkBytes);
    L.ctl_off = align128(L.row_off + row_bytes);
    // 2 * kMaxStages mbarriers (8 B each), 2 x 8 floats, one abort word
    L.total = L.ctl_off + 2 * kMaxStages * 8 + 2 * kConsumerWarps * 4 + 16;
    return L;
}

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
// kWaitLimitNs (or at once if another thread already gave up): sets the
// block's abort word and the watchdog bit, returns false.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int *abort_flag, unsigned int *watchdog,
                                             unsigned int bit) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            const unsigned long long now = global_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(watchdog, bit);
                return false;
            }
        }
    }
}

// Drain wait used by the producer before it exits: bounded, ignores the abort
// word (copies already issued must land before the CTA's memory goes away).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned int *watchdog) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(watchdog, kWatchProducer);
            return;
        }
    }
}

__device__ __forceinline__ void named_barrier_consumers() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <typename T, int OP>
__global__ void __launch_bounds__(kThreads, 1) k_stream(Problem p, int stages) {
    constexpr int EPV = DT<T>::EPV;
    extern __shared__ __align__(128) unsigned char smem[];
    const int ns = OP == OP_PLAIN ? 1 : p.R + 1;  // input streams
    const int row_bytes = (int)(p.H * (int64_t)sizeof(T));
    const int nv = row_bytes / 16;                // packs per row
    const int nchunks = (nv + kConsumers - 1) / kConsumers;
    const Layout L = layout(stages, ns, row_bytes);
    unsigned char *ring = smem + L.ring_off;
    uint4 *row_copy = reinterpret_cast<uint4 *>(smem + L.row_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.ctl_off);
    uint64_t *empty = full + kMaxStages;
    float *red = reinterpret_cast<float *>(empty + kMaxStages);  // [2][kConsumerWarps]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 2 * kConsumerWarps);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
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
        int stage = 0;
        uint32_t phase = 0;
        long long issued = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
            const int64_t row_elem = t * p.H;
            for (int c = 0; c < nchunks && ok; ++c) {
                const int packs = min(kConsumers, nv - c * kConsumers);
                const uint32_t bytes = (uint32_t)packs * 16u;
                ok = wait_bounded(smem_addr(&empty[stage]), phase ^ 1u, abort_flag, p.watchdog,
                                  kWatchProducer);
                if (!ok) break;
                const uint32_t fb = smem_addr(&full[stage]);
                mbar_arrive_expect_tx(fb, bytes * (uint32_t)ns);
                const uint32_t dst = smem_addr(ring + (size_t)stage * ns * kChunkBytes);
                const int64_t off = row_elem + (int64_t)c * kConsumers * EPV;
                for (int s = 0; s < ns; ++s) {
                    const T *src;
                    if (OP != OP_PLAIN && s == ns - 1)
                        src = reinterpret_cast<const T *>(p.residual) + off;
                    else
                        src = reinterpret_cast<const T *>(p.src) + (int64_t)s * p.slice + off;
                    bulk_g2s(dst + (uint32_t)(s * kChunkBytes), src, bytes, fb);
                }
                ++issued;
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Drain: the last min(stages, issued) fills must land before exit.
        const long long first = issued > stages ? issued - stages : 0;
        for (long long f = first; f < issued; ++f)
            wait_drain(smem_addr(&full[f % stages]), (uint32_t)((f / stages) & 1), p.watchdog);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int j = threadIdx.x - 32;  // 0..255
    const int cw = warp - 1;          // consumer warp 0..7
    const T *gamma = reinterpret_cast<const T *>(p.gamma);
    int stage = 0;
    uint32_t phase = 0;
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        const int64_t row_elem = t * p.H;
        float ss = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const bool ok = wait_bounded(smem_addr(&full[stage]), phase, abort_flag, p.watchdog,
                                         kWatchConsumer);
            const int pk = c * kConsumers + j;
            if (ok && pk < nv) {
                const unsigned char *sb = ring + (size_t)stage * ns * kChunkBytes + j * 16;
                uint4 hv;
                if (OP == OP_PLAIN) {
                    hv = *reinterpret_cast<const uint4 *>(sb);
                } else {
                    float acc[EPV];
                    DT<T>::unpack(*reinterpret_cast<const uint4 *>(sb), acc);
#pragma unroll 4
                    for (int s = 1; s < ns; ++s) {
                        float f[EPV];
                        DT<T>::unpack(*reinterpret_cast<const uint4 *>(sb + s * kChunkBytes), f);
#pragma unroll
                        for (int e = 0; e < EPV; ++e) acc[e] = acc[e] + f[e];
                    }
                    hv = DT<T>::pack(acc);  // the one rounding to the storage type
                    st_global(reinterpret_cast<T *>(p.residual) + row_elem + (int64_t)pk * EPV,
                              hv);
                }
                row_copy[pk] = hv;
                float f[EPV];
                DT<T>::unpack(hv, f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) ss += f[e] * f[e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[stage]));
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // row sum of squares over the 8 consumer warps
        ss = warp_sum(ss);
        if (lane == 0) red[par * kConsumerWarps + cw] = ss;
        named_barrier_consumers();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += red[par * kConsumerWarps + w];
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        if (*abort_flag) continue;
        T *y = reinterpret_cast<T *>(p.y) + row_elem;
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

template <typename T>
cudaError_t launch_stream(const Problem &p, const Plan &pl, cudaStream_t st) {
    const int smem = pl.smem;
    cudaError_t e;
    switch (p.op) {
    case OP_PLAIN:
        e = cudaFuncSetAttribute(stream::k_stream<T, OP_PLAIN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        stream::k_stream<T, OP_PLAIN><<<pl.grid, stream::kThreads, smem, st>>>(p, pl.stages);
        break;
    case OP_FUSED:
        e = cudaFuncSetAttribute(stream::k_stream<T, OP_FUSED>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        stream::k_stream<T, OP_FUSED><<<pl.grid, stream::kThreads, smem, st>>>(p, pl.stages);
        break;
    case OP_REDUCE:
        e = cudaFuncSetAttribute(stream::k_stream<T, OP_REDUCE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        stream::k_stream<T, OP_REDUCE><<<pl.grid, stream::kThreads, smem, st>>>(p, pl.stages);
        break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace rarn
