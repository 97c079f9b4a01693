// common.cuh -- problem description and device helpers shared by the kernels.
//
// Storage types: float (binary32), __half (binary16), __nv_bfloat16.  Every
// kernel moves rows in 16-byte vectors ("packs") of EPV elements when the row
// and every base pointer are 16-byte aligned, and element by element
// otherwise.  All arithmetic is binary32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rarn {

enum Op : int { OP_PLAIN = 0, OP_FUSED = 1, OP_REDUCE = 2 };

// 8-bit output: code format and where its scale comes from.
enum QFormat : int { Q_E4M3 = 0, Q_E5M2 = 1 };
enum QMode : int { Q_TENSOR = 0, Q_ROW = 1 };

// One call's arguments, passed to every kernel by value.  Strides are in
// elements of each buffer's own storage type.
struct Problem {
    void *y;               // [T, H] output
    const void *src;       // plain / fused: x [T, H]; reduce: partials [R, T, H]
    void *residual;        // [T, H] in/out (fused, reduce); unused for plain
    const void *gamma;     // [H]
    int64_t T, H;
    int64_t ldx;           // elements between rows of x / of each partial
    int64_t ldr;           // elements between rows of the residual
    int64_t ldy;           // elements between rows of y
    int64_t slice;         // elements between consecutive partial buffers
    int R;                 // partial buffers (reduce), 1 (fused), 0 (plain)
    int op;                // Op
    float eps;
    unsigned int *watchdog;  // device word for bounded-wait failures
    unsigned long long wait_limit_ns;  // bound on every shared-memory barrier wait
    long long stall_fill;    // test hook: in CTA 0 of the stream kernel this fill never
                             // completes (-1: never), so that its consumers' wait runs out
    // 8-bit output (kernels built for it): y holds one-byte codes, ldy in bytes
    float *qscale;           // Q_TENSOR: the one scale (read); Q_ROW: [T] scales (written)
    int qfmt;                // QFormat
    int qmode;               // QMode
    int l2_rows;             // rows each CTA (or warp) prefetches into L2 before waiting on
                             // the previous kernel (0: none; device-memory inputs only)
};

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel waits for the grids it depends
// on before its first global memory access (a no-op when it was launched
// without the programmatic-serialization attribute), and lets its dependents
// launch once each CTA has started its last row, so that their launch
// overlaps this grid's tail.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned address.
// It only warms L2, the GPU's point of coherence, so it may be issued before
// grid_dependency_wait() even where the preceding kernel is still writing
// those bytes: the loads after the wait then find them in L2 instead of
// paying the DRAM latency that otherwise opens every launch.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launch with the programmatic-serialization attribute (pdl) and an
// optional cluster shape.
template <typename... K, typename... A>
inline cudaError_t launch_kernel(void (*kernel)(K...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, int cluster, A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<A &&>(args)...);
}

// ---------------------------------------------------------------------------
// Storage-type traits: 16-byte packs <-> binary32, one rounding on the way out
// ---------------------------------------------------------------------------

template <typename T>
struct DT;

template <>
struct DT<float> {
    static constexpr int EPV = 4;
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
    __device__ __forceinline__ static void unpack(const uint4 &p, float (&f)[EPV]) {
        f[0] = __uint_as_float(p.x);
        f[1] = __uint_as_float(p.y);
        f[2] = __uint_as_float(p.z);
        f[3] = __uint_as_float(p.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[EPV]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ __forceinline__ static float round(float v) { return v; }
};

template <>
struct DT<__half> {
    static constexpr int EPV = 8;
    __device__ __forceinline__ static float to_f(__half v) { return __half2float(v); }
    __device__ __forceinline__ static __half from_f(float v) { return __float2half_rn(v); }
    __device__ __forceinline__ static float2 w2f(uint32_t w) {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        return __half22float2(h);
    }
    __device__ __forceinline__ static uint32_t f2w(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 &p, float (&f)[EPV]) {
        float2 a = w2f(p.x), b = w2f(p.y), c = w2f(p.z), d = w2f(p.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[EPV]) {
        return make_uint4(f2w(f[0], f[1]), f2w(f[2], f[3]), f2w(f[4], f[5]), f2w(f[6], f[7]));
    }
    __device__ __forceinline__ static float round(float v) {
        return __half2float(__float2half_rn(v));
    }
};

template <>
struct DT<__nv_bfloat16> {
    static constexpr int EPV = 8;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) {
        return __float2bfloat16_rn(v);
    }
    // bf16 -> f32 is exact: the pattern moves to the upper half of the word.
    __device__ __forceinline__ static float2 w2f(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ __forceinline__ static uint32_t f2w(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 &p, float (&f)[EPV]) {
        float2 a = w2f(p.x), b = w2f(p.y), c = w2f(p.z), d = w2f(p.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[EPV]) {
        return make_uint4(f2w(f[0], f[1]), f2w(f[2], f[3]), f2w(f[4], f[5]), f2w(f[6], f[7]));
    }
    __device__ __forceinline__ static float round(float v) {
        return __bfloat162float(__float2bfloat16_rn(v));
    }
};

// ---------------------------------------------------------------------------
// Global memory access with cache hints (inline PTX)
// ---------------------------------------------------------------------------

// Load of data read once (x, partials, residual): a plain weak load, which
// sees this thread's own earlier stores and everything the kernels before the
// dependency wait wrote (residual, y aliasing x).  Measured against the
// evict-first (.cs) form, CUDA-graph timing, cold L2: fused bf16 [4096, 4096]
// 20.94 -> 20.75 us, [32768, 5120] 201.7 -> 200.8 us.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Read-only, reused load (gamma: every row reads it).
__device__ __forceinline__ uint4 ld_keep(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_global(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

template <typename T>
__device__ __forceinline__ float ld_elem(const void *base, int64_t i) {
    return DT<T>::to_f(reinterpret_cast<const T *>(base)[i]);
}

template <typename T>
__device__ __forceinline__ void st_elem(void *base, int64_t i, float v) {
    reinterpret_cast<T *>(base)[i] = DT<T>::from_f(v);
}

// ---------------------------------------------------------------------------
// Reductions (xor butterfly within a warp; warp totals combined through
// shared memory).  "Tokenweave fused-RMSNorm-AR kernel", blockReduceSum, and
// "Block All Reduce", warp_reduce_sum_f32 / block_all_reduce: the same
// two-stage scheme.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Sum of v over the whole CTA, returned to every thread.  `red` holds one
// float per warp; callers alternate between two such buffers on consecutive
// rows so that one __syncthreads per row suffices.  Deterministic: fixed
// order for a fixed block size.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = lane < nwarps ? red[lane] : 0.f;
    return warp_sum(s);
}

// Sum of s and maximum of m over the whole CTA in one pass through shared
// memory (one barrier), returned to every thread; the sum in the same order
// as block_sum.
__device__ __forceinline__ float2 block_sum_max(float s, float m, float2 *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    s = warp_sum(s);
    m = warp_max(m);
    if (lane == 0) red[warp] = make_float2(s, m);
    __syncthreads();
    const float2 v = lane < nwarps ? red[lane] : make_float2(0.f, 0.f);
    return make_float2(warp_sum(v.x), warp_max(v.y));
}

// ---------------------------------------------------------------------------
// 8-bit output.  A value v becomes the code of u = (v * m1) * m2, rounded to
// nearest even and saturated to the format's largest finite value:
//   per tensor: m1 = 1 / scale, m2 = 1;
//   per row:    m1 = 1 / max|v|, m2 = maxf (448 for e4m3, 57344 for e5m2), so
//               the row's largest magnitude maps to maxf; the row's scale
//               max|v| / maxf is written out (1 and m1 = m2 = 1 for a row of
//               zeros).  Since inv > 0, max|v| is taken as inv * max|h * gamma|,
//               so the maximum joins the sum of squares in one row reduction.
// ("Block All Reduce", FP8 section: e4m3 and e5m2 codes, converted with
// saturation to the largest finite value.)
// ---------------------------------------------------------------------------
struct QMul {
    float m1, m2;
};

__device__ __forceinline__ float q_maxf(int fmt) { return fmt == Q_E5M2 ? 57344.f : 448.f; }

// Per-tensor multipliers; the scale is read after the grid dependency wait.
__device__ __forceinline__ QMul quant_tensor(const Problem &p) {
    return p.qmode == Q_TENSOR ? QMul{1.f / *p.qscale, 1.f} : QMul{1.f, 1.f};
}

// Per-row multipliers from the row's reduced max|v|; `writer` stores the scale.
// A subnormal max|v| is scaled by 2^24 first (exact), so that its reciprocal
// stays finite.
__device__ __forceinline__ QMul quant_row(const Problem &p, int64_t t, float amax, bool writer) {
    const float maxf = q_maxf(p.qfmt);
    if (writer) p.qscale[t] = amax > 0.f ? amax / maxf : 1.f;
    if (!(amax > 0.f)) return QMul{1.f, 1.f};
    const float k = amax < 1.17549435e-38f ? 16777216.f : 1.f;
    return QMul{1.f / (amax * k), maxf * k};
}

__device__ __forceinline__ uint32_t fp8x2(float a, float b, int fmt) {
    return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                    fmt == Q_E5M2 ? __NV_E5M2 : __NV_E4M3);
}

__device__ __forceinline__ uint8_t fp8x1(float a, int fmt) {
    return __nv_cvt_float_to_fp8(a, __NV_SATFINITE, fmt == Q_E5M2 ? __NV_E5M2 : __NV_E4M3);
}

// Store the codes of N = 4 or 8 values (element 0 at the lowest address).
template <int N>
__device__ __forceinline__ void st_codes(uint8_t *dst, const float (&u)[N], int fmt) {
    static_assert(N == 4 || N == 8, "4 or 8 codes per store");
    const uint32_t w0 = fp8x2(u[0], u[1], fmt) | (fp8x2(u[2], u[3], fmt) << 16);
    if constexpr (N == 4) {
        asm volatile("st.global.u32 [%0], %1;" ::"l"(dst), "r"(w0) : "memory");
    } else {
        const uint32_t w1 = fp8x2(u[4], u[5], fmt) | (fp8x2(u[6], u[7], fmt) << 16);
        asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(dst), "r"(w0), "r"(w1) : "memory");
    }
}

}  // namespace rarn
