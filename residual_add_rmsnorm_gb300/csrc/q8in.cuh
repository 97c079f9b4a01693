// q8in.cuh -- reduce + residual-add + RMSNorm over R partials stored as 8-bit
// codes (e4m3 / e5m2) with one binary32 scale per partial buffer.
//
//   v_r = fl32(dec(c_r) * s_r)                 (each partial dequantised, one rounding)
//   acc = v_0; acc = fl32(acc + v_r), r = 1 .. R-1; acc = fl32(acc + residual)
//   h = RN(acc); residual <- h; inv = rsqrt(mean(h^2) + eps); y = RN((h * inv) * gamma)
//
// ("Block All Reduce", FP8 section: reductions over 8-bit inputs with a
// binary32 accumulator; "Tokenweave fused-RMSNorm-AR kernel", Code
// walkthrough: the reduce + residual + norm steps.)
//
// Two kernel forms.  Register kernels: a CTA per row, VPT packs of 8 (or 16)
// elements per thread: 8 (16) bytes of codes per partial (decoded exactly
// through binary16: every e4m3 / e5m2 value is a binary16 value), the
// residual, gamma and y in the storage type; the partial loop is unrolled so
// that a pack's loads are in flight together, and the rounded row stays in
// registers for the normalise pass.  The TMA-fed kernel (more than 4
// partials, many rows): a persistent CTA per SM whose producer warp streams
// the rows' code chunks and residual into a shared-memory ring with bulk
// copies while 16 consumer warps reduce and normalise.
#pragma once

#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "stream.cuh"  // mbarrier / bulk-copy primitives and bounded waits

namespace rarn {
namespace q8in {

struct Params {
    void *y;
    const uint8_t *codes;   // [R][T][H]
    const float *scales;    // [R]
    void *residual;         // [T][H], updated
    const void *gamma;      // [H]
    int64_t T, H;
    int R;
    int fmt;                // 0 e4m3, 1 e5m2
    float eps;
    int l2_rows;            // rows prefetched into L2 before the dependency wait
    // TMA-fed kernel only
    unsigned int *watchdog;          // device word for bounded-wait failures
    unsigned long long wait_limit_ns;  // bound on every shared-memory barrier wait
    long long stall_fill;            // test hook: in CTA 0 this fill never completes (-1: off)
    int max_smem;                    // dynamic shared memory a CTA may opt into, bytes
};

// 8 elements of the storage type: one 16-byte pack (16-bit) or two (binary32).
template <typename T>
struct Pack8 {
    static constexpr int W = sizeof(T) == 4 ? 2 : 1;  // 16-byte words
    uint4 w[W];
    __device__ __forceinline__ void load(const T *p) {
#pragma unroll
        for (int i = 0; i < W; ++i) w[i] = ld_stream(reinterpret_cast<const char *>(p) + 16 * i);
    }
    __device__ __forceinline__ void load_keep(const T *p) {
#pragma unroll
        for (int i = 0; i < W; ++i) w[i] = ld_keep(reinterpret_cast<const char *>(p) + 16 * i);
    }
    __device__ __forceinline__ void store(T *p) const {
#pragma unroll
        for (int i = 0; i < W; ++i) st_global(reinterpret_cast<char *>(p) + 16 * i, w[i]);
    }
    __device__ __forceinline__ void unpack(float (&f)[8]) const {
        if constexpr (W == 2) {
            DT<T>::unpack(w[0], *reinterpret_cast<float(*)[4]>(f));
            DT<T>::unpack(w[1], *reinterpret_cast<float(*)[4]>(f + 4));
        } else {
            DT<T>::unpack(w[0], f);
        }
    }
    __device__ __forceinline__ void pack(const float (&f)[8]) {
        if constexpr (W == 2) {
            w[0] = DT<T>::pack(*reinterpret_cast<const float(*)[4]>(f));
            w[1] = DT<T>::pack(*reinterpret_cast<const float(*)[4]>(f + 4));
        } else {
            w[0] = DT<T>::pack(f);
        }
    }
};

// 8 codes (8 bytes) -> 8 binary32 values, exact.
template <int FMT>
__device__ __forceinline__ void decode8(uint2 c, float (&f)[8]) {
    constexpr __nv_fp8_interpretation_t kind = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
    const uint32_t w[2] = {c.x, c.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __nv_fp8x2_storage_t two =
                static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * k)) & 0xffffu);
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, kind);
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            f[4 * i + 2 * k] = v.x;
            f[4 * i + 2 * k + 1] = v.y;
        }
    }
}

__device__ __forceinline__ uint2 ld_codes(const uint8_t *p) {
    uint2 v;
    asm volatile("ld.global.cs.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

template <typename T, int VPT, int RMAX, int FMT>
__global__ void __launch_bounds__(256) k_q8in(Params p) {
    __shared__ float red[2][32];
    const int nv = (int)(p.H / 8);
    const int64_t plane = p.T * p.H;
    // first row's codes prefetched into L2 before the wait (L2 is the point
    // of coherence: correct while the previous kernel still writes them);
    // the bulk prefetch needs a 16-byte aligned start and a multiple of 16
    // bytes, so only rows that satisfy both (H a multiple of 16)
    if ((int)threadIdx.x < p.R && (int)threadIdx.x < 32 && blockIdx.x < p.T && p.l2_rows > 0 &&
        p.H % 16 == 0) {
        const uint8_t *row = p.codes + threadIdx.x * plane + (int64_t)blockIdx.x * p.H;
        if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) prefetch_l2(row, (uint32_t)p.H);
    }
    grid_dependency_wait();
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        const uint8_t *crow = p.codes + t * p.H;
        T *res = reinterpret_cast<T *>(p.residual) + t * p.H;
        // the residual packs and partial 0 first, then one partial at a time
        // for all packs (its loads in flight together)
        Pack8<T> hv[VPT];
        float acc[VPT][8];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) hv[k].load(res + 8 * (int64_t)j);
        }
        // unrolled in steps of 4 partials: deeper unrolling lets the compiler
        // hoist every partial's loads and run out of registers
#pragma unroll 4
        for (int r = 0; r < RMAX; ++r) {
            if (r < p.R) {
                const float scr = __ldg(p.scales + r);
                uint2 c[VPT];
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = threadIdx.x + k * blockDim.x;
                    if (j < nv) c[k] = ld_codes(crow + r * plane + 8 * (int64_t)j);
                }
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = threadIdx.x + k * blockDim.x;
                    if (j < nv) {
                        float f[8];
                        decode8<FMT>(c[k], f);
                        // product and sum rounded separately (__fmul_rn /
                        // __fadd_rn are never contracted into one FMA)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float v = __fmul_rn(f[e], scr);
                            acc[k][e] = r == 0 ? v : __fadd_rn(acc[k][e], v);
                        }
                    }
                }
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) {
                float rv[8];
                hv[k].unpack(rv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    acc[k][e] = DT<T>::round(__fadd_rn(acc[k][e], rv[e]));  // h: one rounding
                    ss += acc[k][e] * acc[k][e];
                }
                hv[k].pack(acc[k]);
                hv[k].store(res + 8 * (int64_t)j);
            }
        }
        const float inv = rsqrtf(block_sum(ss, red[par]) / (float)p.H + p.eps);
        T *y = reinterpret_cast<T *>(p.y) + t * p.H;
        const T *g = reinterpret_cast<const T *>(p.gamma);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) {
                float h[8], w[8];
                hv[k].unpack(h);
                Pack8<T> gp;
                gp.load_keep(g + 8 * (int64_t)j);
                gp.unpack(w);
#pragma unroll
                for (int e = 0; e < 8; ++e) h[e] = (h[e] * inv) * w[e];
                Pack8<T> o;
                o.pack(h);
                o.store(y + 8 * (int64_t)j);
            }
        }
    }
}

// Grid: every row-CTA resident at once (the kernel's occupancy times the SMs),
// at most one per row.
template <typename K>
static dim3 resident_grid(K kernel, dim3 block, const Params &p, int num_sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, (int)block.x, 0) !=
            cudaSuccess ||
        per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    return dim3(static_cast<unsigned>(std::min<int64_t>(p.T, (int64_t)num_sms * per_sm)));
}

// 2 codes -> 2 binary32 values, exact (through binary16).
template <int FMT>
__device__ __forceinline__ float2 decode2(uint32_t two) {
    constexpr __nv_fp8_interpretation_t kind = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
    const __half2_raw hr =
        __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), kind);
    return __half22float2(*reinterpret_cast<const __half2 *>(&hr));
}

__device__ __forceinline__ uint4 ld_codes16(const uint8_t *p) { return ld_stream(p); }

// The same operation on packs of 16 elements (H a multiple of 16): one
// 16-byte load of codes per partial and pack, two 8-element packs of the
// storage type for the residual, gamma and y.  (Packed binary32 .f32x2
// multiply and add were tried: the compiler fuses a multiply with its single
// use in an add into one FMA, which skips the product's own rounding, so the
// scalar __fmul_rn / __fadd_rn are used.)
template <typename T, int VPT, int RMAX, int FMT>
__global__ void __launch_bounds__(256) k_q8in16(Params p) {
    __shared__ float red[2][32];
    const int nv = (int)(p.H / 16);
    const int64_t plane = p.T * p.H;
    if ((int)threadIdx.x < p.R && (int)threadIdx.x < 32 && blockIdx.x < p.T && p.l2_rows > 0) {
        const uint8_t *row = p.codes + threadIdx.x * plane + (int64_t)blockIdx.x * p.H;
        if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) prefetch_l2(row, (uint32_t)p.H);
    }
    grid_dependency_wait();
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        const uint8_t *crow = p.codes + t * p.H;
        T *res = reinterpret_cast<T *>(p.residual) + t * p.H;
        Pack8<T> hv[VPT][2];
        float2 acc[VPT][8];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) {
                hv[k][0].load(res + 16 * (int64_t)j);
                hv[k][1].load(res + 16 * (int64_t)j + 8);
            }
        }
        // partials unrolled 8 at a time (4 with four binary32 packs per thread:
        // deeper unrolling hoists more loads than the registers hold)
        constexpr int kUnroll = (VPT == 4 && sizeof(T) == 4) ? 4 : 8;
#pragma unroll kUnroll
        for (int r = 0; r < RMAX; ++r) {
            if (r < p.R) {
                // the scale through the read-only cache (a register array
                // indexed by the partly unrolled loop would live in memory)
                const float scr = __ldg(p.scales + r);
                uint4 c[VPT];
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = threadIdx.x + k * blockDim.x;
                    if (j < nv) c[k] = ld_codes16(crow + r * plane + 16 * (int64_t)j);
                }
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = threadIdx.x + k * blockDim.x;
                    if (j < nv) {
                        const uint32_t w[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float2 d = decode2<FMT>(w[q >> 1] >> (16 * (q & 1)));
                            const float2 v = make_float2(__fmul_rn(d.x, scr), __fmul_rn(d.y, scr));
                            acc[k][q] = r == 0 ? v
                                               : make_float2(__fadd_rn(acc[k][q].x, v.x),
                                                             __fadd_rn(acc[k][q].y, v.y));
                        }
                    }
                }
            }
        }
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float rv[8], h[8];
                    hv[k][hh].unpack(rv);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 s2 = make_float2(__fadd_rn(acc[k][4 * hh + q].x, rv[2 * q]),
                                                      __fadd_rn(acc[k][4 * hh + q].y, rv[2 * q + 1]));
                        h[2 * q] = DT<T>::round(s2.x);  // h: one rounding
                        h[2 * q + 1] = DT<T>::round(s2.y);
                        ss += h[2 * q] * h[2 * q] + h[2 * q + 1] * h[2 * q + 1];
                    }
                    hv[k][hh].pack(h);
                    hv[k][hh].store(res + 16 * (int64_t)j + 8 * hh);
                }
            }
        }
        const float inv = rsqrtf(block_sum(ss, red[par]) / (float)p.H + p.eps);
        T *y = reinterpret_cast<T *>(p.y) + t * p.H;
        const T *g = reinterpret_cast<const T *>(p.gamma);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = threadIdx.x + k * blockDim.x;
            if (j < nv) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float h[8], w[8];
                    hv[k][hh].unpack(h);
                    Pack8<T> gp;
                    gp.load_keep(g + 16 * (int64_t)j + 8 * hh);
                    gp.unpack(w);
#pragma unroll
                    for (int e = 0; e < 8; ++e) h[e] = (h[e] * inv) * w[e];
                    Pack8<T> o;
                    o.pack(h);
                    o.store(y + 16 * (int64_t)j + 8 * hh);
                }
            }
        }
    }
}

template <typename T, int VPT, int RMAX>
static cudaError_t launch_fmt16(const Params &p, int num_sms, dim3 block, bool pdl,
                                cudaStream_t st) {
    auto kernel = p.fmt == 0 ? k_q8in16<T, VPT, RMAX, 0> : k_q8in16<T, VPT, RMAX, 1>;
    return launch_kernel(kernel, resident_grid(kernel, block, p, num_sms), block, 0, st, pdl, 1, p);
}

template <typename T, int VPT>
static cudaError_t launch_r16(const Params &p, int num_sms, dim3 block, bool pdl,
                              cudaStream_t st) {
    if (p.R <= 2) return launch_fmt16<T, VPT, 2>(p, num_sms, block, pdl, st);
    if (p.R <= 4) return launch_fmt16<T, VPT, 4>(p, num_sms, block, pdl, st);
    if (p.R <= 8) return launch_fmt16<T, VPT, 8>(p, num_sms, block, pdl, st);
    return launch_fmt16<T, VPT, 16>(p, num_sms, block, pdl, st);
}

template <typename T, int VPT, int RMAX>
static cudaError_t launch_fmt(const Params &p, int num_sms, dim3 block, bool pdl,
                              cudaStream_t st) {
    auto kernel = p.fmt == 0 ? k_q8in<T, VPT, RMAX, 0> : k_q8in<T, VPT, RMAX, 1>;
    return launch_kernel(kernel, resident_grid(kernel, block, p, num_sms), block, 0, st, pdl, 1, p);
}

template <typename T, int VPT>
static cudaError_t launch_r(const Params &p, int num_sms, dim3 block, bool pdl,
                            cudaStream_t st) {
    if (p.R <= 2) return launch_fmt<T, VPT, 2>(p, num_sms, block, pdl, st);
    if (p.R <= 4) return launch_fmt<T, VPT, 4>(p, num_sms, block, pdl, st);
    if (p.R <= 8) return launch_fmt<T, VPT, 8>(p, num_sms, block, pdl, st);
    return launch_fmt<T, VPT, 16>(p, num_sms, block, pdl, st);
}

// ---------------------------------------------------------------------------
// TMA-fed persistent kernel (rows of a multiple of 16 elements, 16-byte
// aligned partials; T >= 2 x #SM)
// ---------------------------------------------------------------------------

// v[e] = fl32(dec(c_e) * s) for 8 codes (exact decode through binary16).
// (Measured on the TMA-fed kernel, R = 8, [8192, 8192]: the same speed or
// slower were an integer re-layout of each code into binary32 bits, and
// binary16 pairs widened by a mixed-precision add of -0.)
template <int FMT>
__device__ __forceinline__ void dequant8(uint2 c, float s, float (&v)[8]) {
    float f[8];
    decode8<FMT>(c, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(f[e], s);
}

// Consumer warps of the TMA-fed kernel (16 measured faster than 8: R = 8,
// [8192, 8192] bf16 157 vs 173 us; R = 4, [16384, 4096] 133 vs 161 us).
constexpr int kStreamWarps = 16;
// Units of 8 elements per row the TMA-fed kernel takes (H <= 16384; binary32
// storage H <= 8192).
template <typename T>
constexpr int max_units() { return sizeof(T) == 4 ? 1024 : 2048; }

// Shared-memory layout: `stages` stages, each R code chunks (8 bytes per
// 8-element unit) and one residual chunk (8 elements of T per unit); the
// rounded row; then the control words.  Offsets 128-byte aligned.
struct SLayout {
    int code_chunk, stage_bytes, row_off, ctl_off, total;
};

__host__ __device__ inline SLayout slayout(int stages, int R, int ppt, int s, int64_t H,
                                           int warps) {
    SLayout L;
    L.code_chunk = 32 * warps * ppt * 8;
    L.stage_bytes = stream::align128(R * L.code_chunk + L.code_chunk * s);
    L.row_off = stages * L.stage_bytes;
    L.ctl_off = L.row_off + stream::align128((int)(H * s));
    L.total = L.ctl_off + 2 * stream::kMaxStages * 8 + 2 * warps * 4 + 16;
    return L;
}

// One CTA per SM walks rows t = blockIdx.x, blockIdx.x + gridDim.x, ...
// Warp 0 is the producer: one lane issues, per chunk of CU = 512 * PPT units
// of 8 elements, R + 1 cp.async.bulk copies (the R partials' codes and the
// residual) into the next stage of a shared-memory ring, guarded by a "full"
// mbarrier (completed by the byte count) and an "empty" one (released by the
// 16 consumer warps); it runs ahead across rows, so HBM reads stay in flight
// while the consumers reduce and normalise.  Consumer thread j takes the
// units c * CU + m * 512 + j of chunk c: it dequantises and sums the partials
// in order, adds the residual (one rounding), writes the residual unit,
// keeps it in the shared-memory row and accumulates its squares; after the
// row a named barrier combines the warps' sums and each thread normalises
// its own units (the same units, no further synchronisation).  Every wait is
// bounded: on a timeout the kernel sets the watchdog word and the CTA's
// abort word, stops issuing copies, drains the ones issued and returns.
template <typename T, int PPT, int RMAX, int FMT>
__global__ void __launch_bounds__(32 + 32 * kStreamWarps, 1) k_q8in_stream(Params p, int stages) {
    using namespace stream;
    constexpr int kConsumerWarps = kStreamWarps;
    constexpr int kConsumers = 32 * kStreamWarps;
    constexpr int CU = kConsumers * PPT;       // units per chunk
    constexpr int UB = 8 * (int)sizeof(T);     // residual bytes per unit
    extern __shared__ __align__(128) unsigned char smem[];
    const int nu = (int)(p.H / 8);
    const int nchunks = (nu + CU - 1) / CU;
    const int64_t plane = p.T * p.H;
    const SLayout L = slayout(stages, p.R, PPT, (int)sizeof(T), p.H, kStreamWarps);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.ctl_off);  // [stages]
    uint64_t *empty = full + kMaxStages;                               // [stages]
    float *red = reinterpret_cast<float *>(empty + kMaxStages);        // [2][kConsumerWarps]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 2 * kConsumerWarps);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the first row's streams prefetched into L2 before the wait (L2 is the
    // point of coherence: correct while the previous kernel still writes them)
    if (p.l2_rows > 0 && (int)threadIdx.x <= p.R && (int64_t)blockIdx.x < p.T) {
        const int64_t t = blockIdx.x;
        if ((int)threadIdx.x < p.R)
            prefetch_l2(p.codes + threadIdx.x * plane + t * p.H, (uint32_t)p.H);
        else
            prefetch_l2(reinterpret_cast<const T *>(p.residual) + t * p.H,
                        (uint32_t)(p.H * (int64_t)sizeof(T)));
    }
    grid_dependency_wait();
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
        long long n = 0;  // fills issued
        const long long stall_at = blockIdx.x == 0 ? p.stall_fill : -1;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
            for (int c = 0; c < nchunks && ok; ++c, ++n) {
                const int units = min(CU, nu - c * CU);
                const uint32_t cb = (uint32_t)units * 8u, rb = (uint32_t)units * UB;
                const int st = (int)(n % stages);
                const uint32_t ph = (uint32_t)((n / stages) & 1);
                ok = wait_bounded(smem_addr(&empty[st]), ph ^ 1u, abort_flag, p.watchdog,
                                  kWatchProducer, p.wait_limit_ns);
                if (!ok) break;
                const uint32_t fb = smem_addr(&full[st]);
                // test hook: expect 16 bytes more than the copies bring, so that
                // this fill never completes and its consumers' wait runs out
                const uint32_t extra = n == stall_at ? 16u : 0u;
                mbar_arrive_expect_tx(fb, cb * (uint32_t)p.R + rb + extra);
                const uint32_t dst = smem_addr(smem + (size_t)st * L.stage_bytes);
                const int64_t off = t * p.H + (int64_t)c * CU * 8;  // element offset
                for (int r = 0; r < p.R; ++r)
                    bulk_g2s(dst + (uint32_t)(r * L.code_chunk), p.codes + r * plane + off, cb,
                             fb);
                bulk_g2s(dst + (uint32_t)(p.R * L.code_chunk),
                         reinterpret_cast<const T *>(p.residual) + off, rb, fb);
            }
        }
        grid_launch_dependents();
        // Drain: the last min(stages, issued) fills must land before the CTA
        // exits (one deadline for all of them).
        const unsigned long long deadline = global_ns() + p.wait_limit_ns;
        for (long long f = n > stages ? n - stages : 0; f < n; ++f)
            wait_drain(smem_addr(&full[(int)(f % stages)]), (uint32_t)((f / stages) & 1),
                       deadline, p.watchdog);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int j = (int)threadIdx.x - 32;
    Pack8<T> *row_copy = reinterpret_cast<Pack8<T> *>(smem + L.row_off);
    const T *gamma = reinterpret_cast<const T *>(p.gamma);
    T *residual = reinterpret_cast<T *>(p.residual);
    // the partials' scales and this thread's gamma units in registers, read
    // once (they were global loads inside the unit loops: long-scoreboard
    // stalls under ncu)
    float scale[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) scale[r] = r < p.R ? __ldg(p.scales + r) : 0.f;
    constexpr int GU = max_units<T>() / kConsumers;  // gamma units per thread
    Pack8<T> gk[GU];
#pragma unroll
    for (int k = 0; k < GU; ++k)
        if (j + k * kConsumers < nu) gk[k].load_keep(gamma + 8 * (int64_t)(j + k * kConsumers));
    int stage = 0;
    uint32_t phase = 0;
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        float ss = 0.f;
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        for (int c = 0; c < nchunks; ++c) {
            const bool ok = wait_bounded(smem_addr(&full[stage]), phase, abort_flag, p.watchdog,
                                         kWatchConsumer, p.wait_limit_ns);
            const unsigned char *sbase = smem + (size_t)stage * L.stage_bytes;
#pragma unroll
            for (int m = 0; m < PPT; ++m) {
                const int q = m * kConsumers + j;  // unit within the chunk
                const int u = c * CU + q;          // unit within the row
                if (!ok || u >= nu) continue;
                float acc[8];
#pragma unroll
                for (int r = 0; r < RMAX; ++r) {
                    if (r < p.R) {
                        const uint2 code =
                            *reinterpret_cast<const uint2 *>(sbase + r * L.code_chunk + q * 8);
                        float v[8];
                        dequant8<FMT>(code, scale[r], v);
                        // product and sum rounded separately (__fmul_rn /
                        // __fadd_rn are never contracted into one FMA)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] = r == 0 ? v[e] : __fadd_rn(acc[e], v[e]);
                    }
                }
                Pack8<T> hv =
                    *reinterpret_cast<const Pack8<T> *>(sbase + p.R * L.code_chunk + q * UB);
                float rv[8];
                hv.unpack(rv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    acc[e] = DT<T>::round(__fadd_rn(acc[e], rv[e]));  // h: one rounding
                    ss += acc[e] * acc[e];
                }
                hv.pack(acc);
                hv.store(residual + t * p.H + 8 * (int64_t)u);
                row_copy[u] = hv;
            }
            __syncwarp();
            // release the stage only if this warp saw its fill complete (after
            // an abort an unfinished fill's stage stays held)
            if (lane == 0 && ok) mbar_arrive(smem_addr(&empty[stage]));
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[par * kConsumerWarps + cw] = ss;
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += red[par * kConsumerWarps + w];
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        if (*abort_flag) continue;
        T *y = reinterpret_cast<T *>(p.y) + t * p.H;
#pragma unroll
        for (int k = 0; k < GU; ++k) {
            const int u = j + k * kConsumers;
            if (u >= nu) break;
            float h[8], w[8];
            row_copy[u].unpack(h);
            gk[k].unpack(w);
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = (h[e] * inv) * w[e];
            Pack8<T> o;
            o.pack(h);
            o.store(y + 8 * (int64_t)u);
        }
    }
}

// Units per consumer thread per chunk (up to two, while at least 4 stages
// fit) and the deepest ring that fits the shared memory.
struct StreamPlan {
    int ppt = 0, stages = 0, smem = 0;
};

inline StreamPlan plan_stream(int64_t H, int R, int s, int max_smem) {
    StreamPlan sp;
    const int64_t nu = H / 8;
    for (int ppt = nu > 32 * kStreamWarps ? 2 : 1; ppt >= 1; ppt >>= 1) {
        int stages = stream::kMaxStages;
        while (stages >= 2 && slayout(stages, R, ppt, s, H, kStreamWarps).total > max_smem)
            --stages;
        if (stages < 2 || (ppt > 1 && stages < 4)) continue;
        sp.ppt = ppt;
        sp.stages = stages;
        sp.smem = slayout(stages, R, ppt, s, H, kStreamWarps).total;
        return sp;
    }
    return StreamPlan{};
}

// Which kernel a call takes (pure host logic; the launcher and the plan query
// share it).  The TMA-fed kernel (ring = true) needs rows of a multiple of 16
// elements (16-byte code copies) and 16-byte aligned codes, and is chosen
// with at least 8 rows per SM: for more than 4 partials where H >= 4096 (8 or
// more where the rows are shorter), for 4 partials with H >= 4096 and for 3
// with H >= 8192.  Measured (CUDA-graph timing, bf16
// unless noted, register kernel / TMA-fed kernel, us): R = 8 [8192, 8192]
// 234.5 / 139.8 (f16 234 / 156 and binary32 [8192, 4096] 155 / 109 with an
// earlier ring); R = 16 [4096, 8192] 167.0 / 110.2; R = 6 [8192, 8192]
// 193.7 / 125.3; R = 4 [4096, 16384] 140.8 / 116.2, [8192, 8192] 146.6 /
// 115.2, [16384, 4096] 129.7 / 121.5, [32768, 2048] 124.4 / 196.6; R = 3
// [8192, 8192] 126.7 / 97.3, [16384, 4096] 113.2 / 116.2, [32768, 2048]
// 108.1 / 190.2, [4096, 16384] 125.7 / 104.7; R = 2 [32768, 4096] 186.8 /
// 222.1; at H = 2048, [32768, 2048]: R = 6 188.3 / 208.3, R = 8 230.6 /
// 224.6; R = 8 [304, 8192] 7.3 / 8.0.  Otherwise a register kernel: 16-element packs where H is a
// multiple of 16, else 8-element packs, `vpt` packs per thread so that a row
// takes at most 256 threads (vpt = 0: H too long for the type).
// ring_override = 0 / 1 switches the TMA-fed kernel off / takes it for any
// shape it can run; pack16 = false switches the 16-element packs off (the
// RARN_TUNE_FP8IN_RING / RARN_TUNE_FP8IN_PACK16 knobs).
struct KernelChoice {
    bool ring = false;
    StreamPlan sp;       // ring
    int pack = 0;        // register kernels: elements per pack (8 or 16)
    int vpt = 0;         // register kernels: packs per thread
    int block = 0;       // register kernels: threads per CTA
};

inline KernelChoice choose_kernel(int64_t T, int64_t H, int R, int s, bool codes_aligned16,
                                  int num_sms, int max_smem, int ring_override = -1,
                                  bool pack16 = true) {
    KernelChoice k;
    const int force = ring_override;
    if (force != 0 && H % 16 == 0 && codes_aligned16 &&
        (force == 1 || (T >= 8 * (int64_t)num_sms &&
                        ((R > 4 && (H >= 4096 || R >= 8)) || (R == 4 && H >= 4096) ||
                         (R == 3 && H >= 8192))))) {
        k.sp = plan_stream(H, R, s, max_smem);
        if (k.sp.ppt > 0) {
            k.ring = true;
            return k;
        }
    }
    k.pack = H % 16 == 0 && pack16 ? 16 : 8;
    const int64_t nv = H / k.pack;
    k.vpt = nv <= 256 ? 1 : nv <= 512 ? 2 : nv <= 1024 ? 4 : 8;
    if ((k.pack == 16 && k.vpt == 8) || (k.vpt == 8 && s == 4)) k.vpt = 0;
    if (k.vpt > 0) k.block = (int)(((nv + k.vpt - 1) / k.vpt + 31) / 32 * 32);
    return k;
}

inline KernelChoice choose_kernel(const Params &p, int s, int num_sms, int ring_override = -1,
                                  bool pack16 = true) {
    return choose_kernel(p.T, p.H, p.R, s, (reinterpret_cast<uintptr_t>(p.codes) & 15u) == 0,
                         num_sms, p.max_smem, ring_override, pack16);
}

template <typename T, int PPT, int RMAX>
static cudaError_t launch_stream_fmt(const Params &p, const StreamPlan &sp, int grid, bool pdl,
                                     cudaStream_t st) {
    auto kernel = p.fmt == 0 ? k_q8in_stream<T, PPT, RMAX, 0> : k_q8in_stream<T, PPT, RMAX, 1>;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sp.smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kernel, dim3(grid), dim3(32 + 32 * kStreamWarps), sp.smem, st, pdl, 1,
                         p, sp.stages);
}

template <typename T, int PPT>
static cudaError_t launch_stream_r(const Params &p, const StreamPlan &sp, int grid, bool pdl,
                                   cudaStream_t st) {
    if (p.R <= 8) return launch_stream_fmt<T, PPT, 8>(p, sp, grid, pdl, st);
    return launch_stream_fmt<T, PPT, 16>(p, sp, grid, pdl, st);
}

}  // namespace q8in

// Launch the kernel choose_kernel picked for p (H <= 16384; binary32 storage
// H <= 8192); the register kernels grid-stride over rows with every CTA
// resident, the TMA-fed kernel has one CTA per SM.
template <typename T>
cudaError_t launch_q8in(const q8in::Params &p, const q8in::KernelChoice &k, int num_sms, bool pdl,
                        cudaStream_t st) {
    using namespace q8in;
    cudaError_t e = cudaErrorInvalidValue;
    if (k.ring) {
        const int grid = (int)std::min<int64_t>(p.T, num_sms);
        e = k.sp.ppt == 2 ? launch_stream_r<T, 2>(p, k.sp, grid, pdl, st)
                          : launch_stream_r<T, 1>(p, k.sp, grid, pdl, st);
    } else if (k.pack == 16) {
        const dim3 block(static_cast<unsigned>(k.block));
        switch (k.vpt) {
        case 1: e = launch_r16<T, 1>(p, num_sms, block, pdl, st); break;
        case 2: e = launch_r16<T, 2>(p, num_sms, block, pdl, st); break;
        case 4: e = launch_r16<T, 4>(p, num_sms, block, pdl, st); break;
        default: break;
        }
    } else {
        const dim3 block(static_cast<unsigned>(k.block));
        switch (k.vpt) {
        case 1: e = launch_r<T, 1>(p, num_sms, block, pdl, st); break;
        case 2: e = launch_r<T, 2>(p, num_sms, block, pdl, st); break;
        case 4: e = launch_r<T, 4>(p, num_sms, block, pdl, st); break;
        case 8:
            if constexpr (sizeof(T) != 4) e = launch_r<T, 8>(p, num_sms, block, pdl, st);
            break;
        default: break;
        }
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rarn
