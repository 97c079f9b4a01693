// tp.cuh -- tensor-parallel form: reduce-scatter, residual add + RMSNorm,
// all-gather over the N ranks' buffers.
//
// "Tokenweave fused-RMSNorm-AR kernel", Code walkthrough: every rank holds a
// partial [T, H] (the output of a row-parallel layer) in a buffer the other
// ranks can address; each rank reduces the rows of its own block of tokens
// over all ranks' buffers, adds its residual, stores it, normalises, and
// writes the normalised row into every rank's buffer, so that each rank ends
// with all T rows of y.  Here the reduction is N plain 16-byte loads per pack
// (one per rank, summed in binary32 in rank order 0 .. N-1, then the
// residual, one rounding) and the all-gather N plain 16-byte stores; no
// multimem / NVLS, no TMA copies (only a bulk L2 prefetch of the next row
// where that row is memory of this device).  Rank r owns rows floor(r T / N) ..
// floor((r + 1) T / N) - 1.
//
// Ordering between ranks: with signal pads, CTA b of every rank meets CTA b
// of every other rank in a barrier at entry (every rank's partial is
// complete) and at exit (every rank's rows of y are written), tokenweave's
// put / wait signal pair at system scope, every wait bounded; without them
// the caller orders the ranks (no device waits at all).
#pragma once

#include "common.cuh"

namespace rarn {
namespace tp {

constexpr int kMaxRanks = 8;
constexpr int kMaxCtas = 1024;             // signal slots per rank pair
constexpr unsigned int kWatchBarrier = 8u;  // watchdog bit 3
constexpr unsigned long long kWaitLimitNs = 10ull * 1000 * 1000 * 1000;
constexpr int kMaxPacks = 2048;            // 16-byte packs per row (32 KB rows)

struct Params {
    void *bufs[kMaxRanks];         // rank q's [T, H] buffer: partial in, y out
    uint32_t *signals[kMaxRanks];  // rank q's pad [kMaxCtas][kMaxRanks], or all null
    void *residual[kMaxRanks];     // rank q's residual rows [rows of q][H]
    const void *gamma;             // [H]
    int64_t T, H;
    int N;
    int rank;   // >= 0: this rank's CTAs only; -1: every rank, `ctas` CTAs each
    int ctas;   // CTAs per rank, the same on every rank
    float eps;
    unsigned int *watchdog;
    unsigned long long wait_limit_ns;  // bound on every barrier wait
    int stall_rank;  // test hook: this rank's CTA 0 never signals at entry (-1: off)
    // streams whose next row a CTA prefetches into L2 while it works on the
    // current one: bit q rank q's buffer, bit 8 + q rank q's residual; set
    // only for memory of the launching device
    uint32_t prefetch_mask;
};

// Rows [r0, r1) of rank r among N.
__host__ __device__ inline void rows_of(int64_t T, int N, int r, int64_t &r0, int64_t &r1) {
    r0 = T * r / N;
    r1 = T * (r + 1) / N;
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t cas_release_sys(uint32_t *p, uint32_t cmp, uint32_t val) {
    uint32_t old;
    asm volatile("atom.release.sys.global.cas.b32 %0, [%1], %2, %3;"
                 : "=r"(old)
                 : "l"(p), "r"(cmp), "r"(val)
                 : "memory");
    return old;
}

__device__ __forceinline__ uint32_t cas_acquire_sys(uint32_t *p, uint32_t cmp, uint32_t val) {
    uint32_t old;
    asm volatile("atom.acquire.sys.global.cas.b32 %0, [%1], %2, %3;"
                 : "=r"(old)
                 : "l"(p), "r"(cmp), "r"(val)
                 : "memory");
    return old;
}

// Barrier between CTA b of every rank.  Thread q < N sets slot [b][rank] of
// rank q's pad from 0 to 1 (release: what this CTA wrote before is visible to
// rank q once it takes the flag; while the slot still holds the previous
// barrier's flag the thread waits), then takes slot [b][q] of this rank's pad
// from 1 back to 0 (acquire: what rank q's CTA b wrote before its signal is
// visible here).  Each wait gives up after p.wait_limit_ns: the watchdog bit
// is set and the barrier returns false on every thread of the CTA.
__device__ __forceinline__ bool rank_barrier(const Params &p, int rank, int b, bool skip_put) {
    __syncthreads();
    bool ok = true;
    const int q = threadIdx.x;
    if (q < p.N) {
        const unsigned long long deadline = now_ns() + p.wait_limit_ns;
        uint32_t *put = p.signals[q] + (size_t)b * kMaxRanks + rank;
        uint32_t *take = p.signals[rank] + (size_t)b * kMaxRanks + q;
        __threadfence_system();
        if (!skip_put) {
            while (cas_release_sys(put, 0u, 1u) != 0u) {
                if (now_ns() > deadline) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
        }
        while (ok && cas_acquire_sys(take, 1u, 0u) != 1u) {
            if (now_ns() > deadline) {
                ok = false;
                break;
            }
            __nanosleep(32);
        }
        if (!ok) atomicOr(p.watchdog, kWatchBarrier);
    }
    return __syncthreads_and(ok) != 0;
}

// One CTA per row of this rank's block (rows r0 + b, r0 + b + ctas, ...);
// VPT 16-byte packs per thread, the rounded row held in registers.
template <typename T, int VPT>
__global__ void __launch_bounds__(512) k_tp_rows(Params p) {
    __shared__ float red[2][32];
    constexpr int EPV = DT<T>::EPV;
    const int nv = (int)(p.H / EPV);
    const bool world = p.rank < 0;
    const int rank = world ? (int)(blockIdx.x / p.ctas) : p.rank;
    const int b = world ? (int)(blockIdx.x % p.ctas) : (int)blockIdx.x;
    int64_t r0, r1;
    rows_of(p.T, p.N, rank, r0, r1);
    grid_dependency_wait();
    const bool sync = p.signals[0] != nullptr;
    bool ok = true;
    if (sync) ok = rank_barrier(p, rank, b, p.stall_rank == rank && b == 0);
    if (ok) {
        const T *gamma = reinterpret_cast<const T *>(p.gamma);
        uint4 gv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) gv[k] = ld_keep(gamma + (int64_t)j * EPV);
        }
        T *res = reinterpret_cast<T *>(p.residual[rank]);
        int par = 0;
        for (int64_t t = r0 + b; t < r1; t += p.ctas, par ^= 1) {
            // this CTA's next row into L2, one bulk prefetch per stream: one
            // CTA of 512 threads per SM holds one row in registers, so with
            // few ranks it has few loads in flight
            const int64_t tn = t + p.ctas;
            if (tn < r1 && (int)threadIdx.x <= p.N) {
                const uint32_t rb = (uint32_t)(p.H * (int64_t)sizeof(T));
                if ((int)threadIdx.x < p.N) {
                    if ((p.prefetch_mask >> threadIdx.x) & 1u)
                        prefetch_l2(reinterpret_cast<const T *>(p.bufs[threadIdx.x]) + tn * p.H, rb);
                } else if ((p.prefetch_mask >> (8 + rank)) & 1u) {
                    prefetch_l2(res + (tn - r0) * p.H, rb);
                }
            }
            // the residual row first: its loads are in flight with the
            // ranks' (8 ranks, [8192, 8192] on one GPU: 459.5 -> 372.5 us;
            // 4 ranks 292.7 -> 228.4; 2 ranks on [16384, 8192] 408 -> 306)
            T *rrow = res + (t - r0) * p.H;
            uint4 rres[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = threadIdx.x + k * blockDim.x;
                if (j < nv) rres[k] = ld_stream(rrow + (int64_t)j * EPV);
            }
            // reduce-scatter: this row of every rank's buffer, in rank order,
            // RB ranks' loads in flight at a time: all eight with two packs per
            // thread (8 ranks, [8192, 8192] on one GPU: 473 -> 462 us); four
            // with one (eight cost the second CTA per SM: [8192, 4096] 205 ->
            // 258 us); two with four (more spill)
            constexpr int RB = VPT == 2 ? 8 : VPT == 1 ? 4 : 2;
            float acc[VPT][EPV];
#pragma unroll
            for (int q0 = 0; q0 < kMaxRanks; q0 += RB) {
                if (q0 >= p.N) break;
                uint4 v[RB][VPT];
#pragma unroll
                for (int u = 0; u < RB; ++u) {
                    if (q0 + u >= p.N) break;
                    const T *src = reinterpret_cast<const T *>(p.bufs[q0 + u]) + t * p.H;
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        const int j = threadIdx.x + k * blockDim.x;
                        if (j < nv) v[u][k] = ld_stream(src + (int64_t)j * EPV);
                    }
                }
#pragma unroll
                for (int u = 0; u < RB; ++u) {
                    if (q0 + u >= p.N) break;
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        if (threadIdx.x + k * blockDim.x >= nv) continue;
                        float f[EPV];
                        DT<T>::unpack(v[u][k], f);
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            acc[k][e] = (q0 + u == 0) ? f[e] : __fadd_rn(acc[k][e], f[e]);
                    }
                }
            }
            // + residual, one rounding, stored; squares of the rounded row
            uint4 hv[VPT];
            float ss = 0.f;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = threadIdx.x + k * blockDim.x;
                if (j >= nv) continue;
                float f[EPV];
                DT<T>::unpack(rres[k], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = __fadd_rn(acc[k][e], f[e]);
                hv[k] = DT<T>::pack(f);
                st_global(rrow + (int64_t)j * EPV, hv[k]);
                DT<T>::unpack(hv[k], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) ss = fmaf(f[e], f[e], ss);
            }
            const float inv = rsqrtf(block_sum(ss, red[par]) / (float)p.H + p.eps);
            // all-gather: the normalised row into every rank's buffer
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = threadIdx.x + k * blockDim.x;
                if (j >= nv) continue;
                float f[EPV], g[EPV];
                DT<T>::unpack(hv[k], f);
                DT<T>::unpack(gv[k], g);
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = (f[e] * inv) * g[e];
                const uint4 yv = DT<T>::pack(f);
#pragma unroll
                for (int q = 0; q < kMaxRanks; ++q) {
                    if (q >= p.N) break;
                    st_global(reinterpret_cast<T *>(p.bufs[q]) + t * p.H + (int64_t)j * EPV, yv);
                }
            }
        }
    }
    grid_launch_dependents();
    if (sync && ok) rank_barrier(p, rank, b, false);
}

// Packs per thread and threads per CTA for a row of nv packs: the fewest
// packs per thread (1, 2, 4) that keep the CTA within 512 threads.
inline void tp_shape(int64_t nv, int &vpt, int &block) {
    vpt = nv <= 512 ? 1 : nv <= 1024 ? 2 : 4;
    block = (int)(((nv + vpt - 1) / vpt + 31) / 32 * 32);
}

// CTAs per rank (T > 0): every CTA of a rank resident at once (a CTA waits
// on its counterparts only), all ranks' in the one grid of the world launch;
// the rows of the largest block spread evenly; the same on every rank.
inline int ctas_per_rank(int64_t T, int N, int num_sms, int per_sm, bool world) {
    const int64_t rows_max = (T + N - 1) / N;
    int64_t slots = (int64_t)num_sms * per_sm / (world ? N : 1);
    if (slots > kMaxCtas) slots = kMaxCtas;
    if (slots < 1) slots = 1;
    const int64_t rounds = (rows_max + slots - 1) / slots;
    const int64_t c = (rows_max + rounds - 1) / rounds;
    return c < 1 ? 1 : (int)c;
}

// Whether each CTA prefetches its next row into L2.  A CTA holds its row's
// N + 1 loads (the residual and the N ranks', each a row of row_bytes) in
// flight before it reduces, so an SM has per_sm (N + 1) rows of loads out.
// Measured on a GB300, eight to two ranks' buffers on one GPU, prefetch off
// -> on: with one CTA per SM a gain up to 64 KB in flight (bf16 H = 8192, two
// ranks 160.5 -> 125.7 us; H = 5120, four ranks 188.5 -> 148.8; H = 8192,
// three ranks 194.4 -> 170.5), mostly a gain at 80 KB (four ranks at H =
// 8192: bf16 228.9 -> 214.0, f16 220.6 -> 213.0; f32 H = 4096 211.3 ->
// 213.2), a loss from 96 KB (eight ranks at H = 8192: 378 -> 436; f32 H =
// 8192, two ranks 244.4 -> 257.2); with two or four CTAs per SM a gain at
// 48 KB (bf16 H = 4096, two ranks 77.0 -> 71.2), none at 64 KB and a loss at
// 80 KB (H = 4096, four ranks 110.6 -> 117.8; H = 2048 111.0 -> 120.5).
inline bool prefetch_wanted(int per_sm, int N, int64_t row_bytes) {
    const int64_t inflight = (int64_t)per_sm * (N + 1) * row_bytes;
    return inflight <= 64 * 1024 || (per_sm == 1 && inflight <= 80 * 1024);
}

}  // namespace tp

// CTAs of k_tp_rows that fit on one SM for rows of H elements.
template <typename T>
cudaError_t tp_blocks_per_sm(int64_t H, int *blocks);

// Launch k_tp_rows for p (p.ctas already set) as `grid` CTAs; cooperative
// when every rank runs in this one grid and the ranks meet in barriers (all
// CTAs must then be resident at once).
template <typename T>
cudaError_t launch_tp(const tp::Params &p, int grid, bool cooperative, bool pdl,
                      cudaStream_t st);

}  // namespace rarn
