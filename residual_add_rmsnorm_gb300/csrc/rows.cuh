// rows.cuh -- register-staged row kernels: a warp or a CTA per row.
//
// Each row is read once from HBM.  The first pass loads the row's input
// streams (x; or the R partial buffers and the residual), sums them in
// binary32 in stream order, rounds the sum once to the storage type, writes it
// back as the residual and keeps it in registers while it accumulates the sum
// of squares.  After the row reduction the second pass scales the values still
// held in registers by rsqrt(ss / H + eps) and by gamma and writes y: the
// normalise pass never goes back to HBM.  ("Tokenweave fused-RMSNorm-AR
// kernel", Code walkthrough: the same two passes, where the second pass
// re-reads the residual from global memory; here only the two-pass kernel for
// rows too long for registers does that.)
//
// Rows are spread over a grid that is capped at what the GPU holds at once;
// each CTA (or warp) walks its rows with a grid stride.
#pragma once

#include "common.cuh"
#include "plan.h"

namespace rarn {

// Input streams per element: plain 1 (x); fused 2 (x, residual); reduce R + 1
// (partials, residual).  Stream s < R is partial s (x for fused); the last
// stream is the residual.
__device__ __forceinline__ int n_streams(const Problem &p) {
    return p.op == OP_PLAIN ? 1 : p.R + 1;
}

template <typename T>
__device__ __forceinline__ const T *stream_row(const Problem &p, int s, int64_t row_off) {
    const bool is_res = (p.op != OP_PLAIN) && (s == p.R);
    const T *base = is_res ? reinterpret_cast<const T *>(p.residual)
                           : reinterpret_cast<const T *>(p.src) + (int64_t)s * p.slice;
    return base + row_off;
}

// ---------------------------------------------------------------------------
// Pass 1, 16-byte packs.  Thread owns packs j = j0 + k * js (k < VPT, j < nv).
// Loads RC streams at a time so that RC * VPT loads are in flight per thread.
// Returns this thread's share of the sum of squares; hv receives the rounded
// row values.
// ---------------------------------------------------------------------------
template <typename T, int VPT, int OP, int RC>
__device__ __forceinline__ float pass1_vec(const Problem &p, int64_t t, int j0, int js, int nv,
                                           uint4 (&hv)[VPT]) {
    constexpr int EPV = DT<T>::EPV;
    const int64_t row_off = t * p.H;
    float ss = 0.f;
    if (OP == OP_PLAIN) {
        const T *x = reinterpret_cast<const T *>(p.src) + row_off;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * js;
            if (j < nv) hv[k] = ld_stream(x + (int64_t)j * EPV);
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * js;
            if (j < nv) {
                float f[EPV];
                DT<T>::unpack(hv[k], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) ss += f[e] * f[e];
            }
        }
        return ss;
    }
    const int S = p.R + 1;
    float acc[VPT][EPV];
    for (int s0 = 0; s0 < S; s0 += RC) {
        uint4 buf[RC][VPT];
#pragma unroll
        for (int q = 0; q < RC; ++q) {
            if (s0 + q < S) {
                const T *base = stream_row<T>(p, s0 + q, row_off);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = j0 + k * js;
                    if (j < nv) buf[q][k] = ld_stream(base + (int64_t)j * EPV);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < RC; ++q) {
            if (s0 + q < S) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int j = j0 + k * js;
                    if (j < nv) {
                        float f[EPV];
                        DT<T>::unpack(buf[q][k], f);
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            acc[k][e] = (s0 + q == 0) ? f[e] : acc[k][e] + f[e];
                    }
                }
            }
        }
    }
    T *res = reinterpret_cast<T *>(p.residual) + row_off;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            hv[k] = DT<T>::pack(acc[k]);  // the one rounding to the storage type
            st_global(res + (int64_t)j * EPV, hv[k]);
            float f[EPV];
            DT<T>::unpack(hv[k], f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) ss += f[e] * f[e];
        }
    }
    return ss;
}

// This thread's gamma packs.  A thread owns the same packs of every row, so
// kernels that keep gamma in registers load it once, before their first row:
// its latency then overlaps the first row's loads instead of following the
// row reduction.
template <typename T, int VPT>
__device__ __forceinline__ void load_gamma_vec(const Problem &p, int j0, int js, int nv,
                                               uint4 (&gv)[VPT]) {
    constexpr int EPV = DT<T>::EPV;
    const T *g = reinterpret_cast<const T *>(p.gamma);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) gv[k] = ld_keep(g + (int64_t)j * EPV);
    }
}

// Pass 2, 16-byte packs: y = (h * inv) * gamma, one rounding.  With PG the
// gamma packs come from registers (gv), otherwise from memory (L1 / L2).
template <typename T, int VPT, bool PG = false>
__device__ __forceinline__ void pass2_vec(const Problem &p, int64_t t, int j0, int js, int nv,
                                          const uint4 (&hv)[VPT], float inv,
                                          const uint4 *gv = nullptr) {
    constexpr int EPV = DT<T>::EPV;
    const T *g = reinterpret_cast<const T *>(p.gamma);
    T *y = reinterpret_cast<T *>(p.y) + t * p.H;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            float h[EPV], w[EPV];
            DT<T>::unpack(hv[k], h);
            DT<T>::unpack(PG ? gv[k] : ld_keep(g + (int64_t)j * EPV), w);
#pragma unroll
            for (int e = 0; e < EPV; ++e) h[e] = (h[e] * inv) * w[e];
            st_global(y + (int64_t)j * EPV, DT<T>::pack(h));
        }
    }
}

// ---------------------------------------------------------------------------
// Pass 1 / pass 2, single elements (rows or pointers not 16-byte aligned).
// Thread owns elements i = i0 + k * is (k < NE, i < H); values held as
// binary32 (already rounded to the storage type).
// ---------------------------------------------------------------------------
template <typename T, int NE, int OP, int RC>
__device__ __forceinline__ float pass1_scalar(const Problem &p, int64_t t, int i0, int is,
                                              float (&h)[NE]) {
    const int64_t row_off = t * p.H;
    const int H = (int)p.H;
    float ss = 0.f;
    if (OP == OP_PLAIN) {
        const T *x = reinterpret_cast<const T *>(p.src) + row_off;
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int i = i0 + k * is;
            h[k] = i < H ? DT<T>::to_f(x[i]) : 0.f;
            ss += h[k] * h[k];
        }
        return ss;
    }
    const int S = p.R + 1;
    for (int s0 = 0; s0 < S; s0 += RC) {
        float buf[RC][NE];
#pragma unroll
        for (int q = 0; q < RC; ++q) {
            if (s0 + q < S) {
                const T *base = stream_row<T>(p, s0 + q, row_off);
#pragma unroll
                for (int k = 0; k < NE; ++k) {
                    const int i = i0 + k * is;
                    buf[q][k] = i < H ? DT<T>::to_f(base[i]) : 0.f;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < RC; ++q) {
            if (s0 + q < S) {
#pragma unroll
                for (int k = 0; k < NE; ++k) h[k] = (s0 + q == 0) ? buf[q][k] : h[k] + buf[q][k];
            }
        }
    }
    T *res = reinterpret_cast<T *>(p.residual) + row_off;
#pragma unroll
    for (int k = 0; k < NE; ++k) {
        const int i = i0 + k * is;
        if (i < H) {
            const T r = DT<T>::from_f(h[k]);
            res[i] = r;
            h[k] = DT<T>::to_f(r);
            ss += h[k] * h[k];
        }
    }
    return ss;
}

template <typename T, int NE>
__device__ __forceinline__ void pass2_scalar(const Problem &p, int64_t t, int i0, int is,
                                             const float (&h)[NE], float inv) {
    const T *g = reinterpret_cast<const T *>(p.gamma);
    T *y = reinterpret_cast<T *>(p.y) + t * p.H;
    const int H = (int)p.H;
#pragma unroll
    for (int k = 0; k < NE; ++k) {
        const int i = i0 + k * is;
        if (i < H) y[i] = DT<T>::from_f((h[k] * inv) * DT<T>::to_f(g[i]));
    }
}

template <int OP>
struct Chunk {  // streams loaded together in pass 1
    static constexpr int value = OP == OP_REDUCE ? 4 : 2;
};

// CTA size each register-staged kernel is compiled for (plan.h budget); a
// combination over budget is compiled for 128 threads and never planned.
template <typename T, int VPT, int OP, bool PG = false>
struct VecBound {
    static constexpr int b = rows_max_block(rows_regs_vec(VPT, DT<T>::EPV, OP, PG));
    static constexpr int value = b > 0 ? b : 128;
};

template <int NE, int OP>
struct ScalarBound {
    static constexpr int b = rows_max_block(rows_regs_scalar(NE, OP));
    static constexpr int value = b > 0 ? b : 128;
};

// ---------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------

// One CTA per row, packs.  PG: gamma held in registers for all rows.
template <typename T, int VPT, int OP, bool PG>
__global__ void __launch_bounds__(VecBound<T, VPT, OP, PG>::value) k_cta_vec(Problem p) {
    __shared__ float red[2][32];
    const int nv = (int)(p.H / DT<T>::EPV);
    grid_dependency_wait();
    uint4 gv[VPT];
    if (PG) load_gamma_vec<T, VPT>(p, threadIdx.x, blockDim.x, nv, gv);
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        uint4 hv[VPT];
        const float ss = pass1_vec<T, VPT, OP, Chunk<OP>::value>(p, t, threadIdx.x, blockDim.x,
                                                                nv, hv);
        const float tot = block_sum(ss, red[par]);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        pass2_vec<T, VPT, PG>(p, t, threadIdx.x, blockDim.x, nv, hv, inv, gv);
    }
}

// One CTA per row, packs, software-pipelined across rows (plain and fused
// forms: one or two input streams).  Before a CTA reduces and writes row t it
// issues the loads of its next row into a second register buffer, so the
// SM keeps reads in flight through the row reduction and the y stores instead
// of draining between rows.
template <typename T, int VPT, int OP>
struct RowLoads {
    static constexpr int S = OP == OP_PLAIN ? 1 : 2;  // x (, residual)
    uint4 v[S][VPT];
};

template <typename T, int VPT, int OP>
__device__ __forceinline__ void issue_row_loads(const Problem &p, int64_t t, int j0, int js,
                                                int nv, RowLoads<T, VPT, OP> &b) {
    constexpr int EPV = DT<T>::EPV;
    const int64_t row_off = t * p.H;
#pragma unroll
    for (int s = 0; s < RowLoads<T, VPT, OP>::S; ++s) {
        const T *base = s == 0 ? reinterpret_cast<const T *>(p.src) + row_off
                               : reinterpret_cast<const T *>(p.residual) + row_off;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * js;
            if (j < nv) b.v[s][k] = ld_stream(base + (int64_t)j * EPV);
        }
    }
}

// h from the loaded packs (fused: x + residual in binary32, one rounding,
// residual written back); returns this thread's share of the sum of squares.
template <typename T, int VPT, int OP>
__device__ __forceinline__ float consume_row_loads(const Problem &p, int64_t t, int j0, int js,
                                                   int nv, const RowLoads<T, VPT, OP> &b,
                                                   uint4 (&hv)[VPT]) {
    constexpr int EPV = DT<T>::EPV;
    T *res = reinterpret_cast<T *>(p.residual) + t * p.H;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            float h[EPV];
            DT<T>::unpack(b.v[0][k], h);
            if (OP == OP_FUSED) {
                float r[EPV];
                DT<T>::unpack(b.v[1][k], r);
#pragma unroll
                for (int e = 0; e < EPV; ++e) h[e] = h[e] + r[e];
                hv[k] = DT<T>::pack(h);  // the one rounding to the storage type
                st_global(res + (int64_t)j * EPV, hv[k]);
                DT<T>::unpack(hv[k], h);
            } else {
                hv[k] = b.v[0][k];
            }
#pragma unroll
            for (int e = 0; e < EPV; ++e) ss += h[e] * h[e];
        }
    }
    return ss;
}

template <typename T, int VPT, int OP>
struct PipeBound {
    static constexpr int b = rows_max_block(rows_regs_vec(VPT, DT<T>::EPV, OP, false) +
                                            VPT * 4 * RowLoads<T, VPT, OP>::S);
    static constexpr int value = b > 0 ? b : 128;
};

template <typename T, int VPT, int OP>
__global__ void __launch_bounds__(PipeBound<T, VPT, OP>::value) k_cta_pipe(Problem p) {
    __shared__ float red[2][32];
    const int nv = (int)(p.H / DT<T>::EPV);
    grid_dependency_wait();
    RowLoads<T, VPT, OP> next;
    int64_t t = blockIdx.x;
    if (t < p.T) issue_row_loads<T, VPT, OP>(p, t, threadIdx.x, blockDim.x, nv, next);
    int par = 0;
    for (; t < p.T; t += gridDim.x, par ^= 1) {
        const RowLoads<T, VPT, OP> cur = next;
        if (t + gridDim.x < p.T) {
            issue_row_loads<T, VPT, OP>(p, t + gridDim.x, threadIdx.x, blockDim.x, nv, next);
        } else {
            grid_launch_dependents();
        }
        uint4 hv[VPT];
        const float ss = consume_row_loads<T, VPT, OP>(p, t, threadIdx.x, blockDim.x, nv, cur, hv);
        const float tot = block_sum(ss, red[par]);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        pass2_vec<T, VPT, false>(p, t, threadIdx.x, blockDim.x, nv, hv, inv);
    }
}

// One warp per row, packs; blockDim.x / 32 rows per CTA at a time.  Gamma is
// held in registers (at most 4 packs per lane).
template <typename T, int VPT, int OP>
__global__ void __launch_bounds__(256) k_warp_vec(Problem p) {
    const int nv = (int)(p.H / DT<T>::EPV);
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int64_t first = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const int64_t step = (int64_t)gridDim.x * wpb;
    grid_dependency_wait();
    uint4 gv[VPT];
    load_gamma_vec<T, VPT>(p, lane, 32, nv, gv);
    for (int64_t t = first; t < p.T; t += step) {
        if (t + step >= p.T) grid_launch_dependents();
        uint4 hv[VPT];
        const float ss = pass1_vec<T, VPT, OP, Chunk<OP>::value>(p, t, lane, 32, nv, hv);
        const float tot = warp_sum(ss);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        pass2_vec<T, VPT, true>(p, t, lane, 32, nv, hv, inv, gv);
    }
}

// One CTA per row, single elements.
template <typename T, int NE, int OP>
__global__ void __launch_bounds__(ScalarBound<NE, OP>::value) k_cta_scalar(Problem p) {
    __shared__ float red[2][32];
    grid_dependency_wait();
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        float h[NE];
        const float ss =
            pass1_scalar<T, NE, OP, Chunk<OP>::value>(p, t, threadIdx.x, blockDim.x, h);
        const float tot = block_sum(ss, red[par]);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        pass2_scalar<T, NE>(p, t, threadIdx.x, blockDim.x, h, inv);
    }
}

// Rows too long for registers: pass 1 walks the row in tiles of blockDim
// packs (or elements); pass 2 re-reads the stored row (the residual, or x for
// the plain form) -- each thread re-reads only what it wrote itself.
template <typename T, int OP, bool VEC>
__global__ void __launch_bounds__(1024) k_two_pass(Problem p) {
    __shared__ float red[2][32];
    constexpr int EPV = VEC ? DT<T>::EPV : 1;
    const int n = (int)(p.H / EPV);
    grid_dependency_wait();
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        float ss = 0.f;
        for (int base = 0; base < n; base += blockDim.x) {
            if (VEC) {
                uint4 hv[1];
                ss += pass1_vec<T, 1, OP, Chunk<OP>::value>(p, t, base + threadIdx.x, 1 << 30,
                                                           n, hv);
            } else {
                float h[1];
                ss += pass1_scalar<T, 1, OP, Chunk<OP>::value>(p, t, base + threadIdx.x,
                                                              1 << 30, h);
            }
        }
        const float tot = block_sum(ss, red[par]);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        const void *stored = OP == OP_PLAIN ? p.src : p.residual;
        for (int base = 0; base < n; base += blockDim.x) {
            const int j = base + threadIdx.x;
            if (j >= n) break;
            if (VEC) {
                uint4 hv[1] = {ld_stream(reinterpret_cast<const T *>(stored) + t * p.H +
                                         (int64_t)j * EPV)};
                pass2_vec<T, 1>(p, t, j, 1 << 30, n, hv, inv);
            } else {
                float h[1] = {ld_elem<T>(stored, t * p.H + j)};
                pass2_scalar<T, 1>(p, t, j, 1 << 30, h, inv);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Launcher: plan -> template instance
// ---------------------------------------------------------------------------

template <typename T, int OP>
static cudaError_t launch_rows_op(const Problem &p, const Plan &pl, cudaStream_t st) {
    const dim3 g(pl.grid), b(pl.block);
    auto go = [&](auto kernel) { return launch_kernel(kernel, g, b, 0, st, pl.pdl, 1, p); };
    switch (pl.kind) {
    case KIND_WARP:
        switch (pl.per_thread) {
        case 1: return go(k_warp_vec<T, 1, OP>);
        case 2: return go(k_warp_vec<T, 2, OP>);
        case 4: return go(k_warp_vec<T, 4, OP>);
        default: return cudaErrorInvalidValue;
        }
    case KIND_CTA:
        if (pl.vec && pl.pipe && OP != OP_REDUCE) {
            switch (pl.per_thread) {
            case 1: return go(k_cta_pipe<T, 1, OP == OP_REDUCE ? OP_FUSED : OP>);
            case 2: return go(k_cta_pipe<T, 2, OP == OP_REDUCE ? OP_FUSED : OP>);
            case 4: return go(k_cta_pipe<T, 4, OP == OP_REDUCE ? OP_FUSED : OP>);
            case 8: return go(k_cta_pipe<T, 8, OP == OP_REDUCE ? OP_FUSED : OP>);
            default: return cudaErrorInvalidValue;
            }
        }
        if (pl.vec && pl.prefetch_gamma) {
            switch (pl.per_thread) {
            case 1: return go(k_cta_vec<T, 1, OP, true>);
            case 2: return go(k_cta_vec<T, 2, OP, true>);
            case 4: return go(k_cta_vec<T, 4, OP, true>);
            case 8: return go(k_cta_vec<T, 8, OP, true>);
            default: return cudaErrorInvalidValue;
            }
        }
        if (pl.vec) {
            switch (pl.per_thread) {
            case 1: return go(k_cta_vec<T, 1, OP, false>);
            case 2: return go(k_cta_vec<T, 2, OP, false>);
            case 4: return go(k_cta_vec<T, 4, OP, false>);
            case 8: return go(k_cta_vec<T, 8, OP, false>);
            default: return cudaErrorInvalidValue;
            }
        }
        switch (pl.per_thread) {
        case 1: return go(k_cta_scalar<T, 1, OP>);
        case 2: return go(k_cta_scalar<T, 2, OP>);
        case 4: return go(k_cta_scalar<T, 4, OP>);
        case 8: return go(k_cta_scalar<T, 8, OP>);
        case 16: return go(k_cta_scalar<T, 16, OP>);
        default: return cudaErrorInvalidValue;
        }
    case KIND_TWO_PASS:
        return pl.vec ? go(k_two_pass<T, OP, true>) : go(k_two_pass<T, OP, false>);
    default:
        return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_rows(const Problem &p, const Plan &pl, cudaStream_t st) {
    cudaError_t e;
    switch (p.op) {
    case OP_PLAIN: e = launch_rows_op<T, OP_PLAIN>(p, pl, st); break;
    case OP_FUSED: e = launch_rows_op<T, OP_FUSED>(p, pl, st); break;
    case OP_REDUCE: e = launch_rows_op<T, OP_REDUCE>(p, pl, st); break;
    default: return cudaErrorInvalidValue;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rarn
