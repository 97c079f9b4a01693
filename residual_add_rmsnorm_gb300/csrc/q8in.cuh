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
// A CTA per row, VPT packs of 8 elements per thread: 8 bytes of codes per
// partial (decoded exactly through binary16: every e4m3 / e5m2 value is a
// binary16 value), the residual, gamma and y in the storage type.  The
// partial loop is unrolled to RMAX so that every load of a pack is in flight
// at once; the rounded row stays in registers for the normalise pass.
#pragma once

#include <cuda_fp8.h>

#include <algorithm>
#include <cstdlib>

#include "common.cuh"

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

}  // namespace q8in

// Packs per thread so that a row takes at most 256 threads (H <= 16384;
// binary32 storage H <= 8192); grid-stride over rows with a few CTAs per SM.
template <typename T>
cudaError_t launch_q8in(const q8in::Params &p, int num_sms, bool pdl, cudaStream_t st) {
    using namespace q8in;
    if (p.H % 16 == 0 && !(getenv("RARN_Q8IN_16") && atoi(getenv("RARN_Q8IN_16")) == 0)) {
        // 16-element packs (measurements can switch them off)
        const int64_t nv = p.H / 16;
        const int vpt = nv <= 256 ? 1 : nv <= 512 ? 2 : 4;
        const dim3 block(static_cast<unsigned>((nv + vpt - 1) / vpt + 31) / 32 * 32);
        cudaError_t e;
        switch (vpt) {
        case 1: e = launch_r16<T, 1>(p, num_sms, block, pdl, st); break;
        case 2: e = launch_r16<T, 2>(p, num_sms, block, pdl, st); break;
        default: e = launch_r16<T, 4>(p, num_sms, block, pdl, st); break;
        }
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t nv = p.H / 8;
    const int vpt = nv <= 256 ? 1 : nv <= 512 ? 2 : nv <= 1024 ? 4 : 8;
    if (vpt == 8 && sizeof(T) == 4) return cudaErrorInvalidValue;
    const dim3 block(static_cast<unsigned>((nv + vpt - 1) / vpt + 31) / 32 * 32);
    cudaError_t e;
    switch (vpt) {
    case 1: e = launch_r<T, 1>(p, num_sms, block, pdl, st); break;
    case 2: e = launch_r<T, 2>(p, num_sms, block, pdl, st); break;
    case 4: e = launch_r<T, 4>(p, num_sms, block, pdl, st); break;
    default:
        if constexpr (sizeof(T) == 4) {
            e = cudaErrorInvalidValue;
        } else {
            e = launch_r<T, 8>(p, num_sms, block, pdl, st);
        }
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rarn
