// rows.cuh -- register-staged row kernels: a warp or a CTA per row.
//
// Each row is read once from HBM.  The first pass loads the row's input
// streams (x; or the R partial buffers and the residual), sums them in
// binary32 in stream order, rounds the sum once to the residual's storage
// type, writes it back as the residual and keeps it in registers while it
// accumulates the sum of squares.  After the row reduction the second pass
// scales the values still held in registers by rsqrt(ss / H + eps) and by
// gamma and writes y: the normalise pass never goes back to HBM.
// ("Tokenweave fused-RMSNorm-AR kernel", Code walkthrough: the same two
// passes, where the second pass re-reads the residual from global memory;
// here only the two-pass kernel for rows too long for registers does that.)
//
// T is the storage type of x / partials, gamma and y; TR that of the residual:
// either T, or binary32 with a 16-bit T (an fp32 residual stream), in which
// case the sum is kept in binary32 without rounding and staged as such.
// Every buffer has its own row stride (Problem::ldx, ldr, ldy).
//
// Rows are spread over a grid that is capped at what the GPU holds at once;
// each CTA (or warp) walks its rows with a grid stride.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "plan.h"

namespace rarn {

// ---------------------------------------------------------------------------
// Residual storage for one pack of T (EPV elements): N 16-byte words.
// ---------------------------------------------------------------------------
template <typename T, typename TR>
struct Res {
    static constexpr int EPV = DT<T>::EPV;
    static constexpr bool SAME = std::is_same<T, TR>::value;
    static_assert(SAME || std::is_same<TR, float>::value, "residual: T or binary32");
    static constexpr int N = SAME ? 1 : (EPV * 4) / 16;  // 16-byte words per pack
    static constexpr int EPW = 16 / (int)sizeof(TR);     // residual elements per word

    __device__ __forceinline__ static void to_f(const uint4 (&v)[N], float (&f)[EPV]) {
        if constexpr (SAME) {
            DT<T>::unpack(v[0], f);
        } else {
#pragma unroll
            for (int q = 0; q < N; ++q) {
                f[4 * q + 0] = __uint_as_float(v[q].x);
                f[4 * q + 1] = __uint_as_float(v[q].y);
                f[4 * q + 2] = __uint_as_float(v[q].z);
                f[4 * q + 3] = __uint_as_float(v[q].w);
            }
        }
    }
    // The one rounding of the sum to the residual's storage type (none for
    // binary32).
    __device__ __forceinline__ static void from_f(const float (&f)[EPV], uint4 (&v)[N]) {
        if constexpr (SAME) {
            v[0] = DT<T>::pack(f);
        } else {
#pragma unroll
            for (int q = 0; q < N; ++q)
                v[q] = make_uint4(__float_as_uint(f[4 * q + 0]), __float_as_uint(f[4 * q + 1]),
                                  __float_as_uint(f[4 * q + 2]), __float_as_uint(f[4 * q + 3]));
        }
    }
};

template <int OP>
struct Chunk {  // streams loaded together in pass 1 (same-type residual)
    static constexpr int value = OP == OP_REDUCE ? 4 : 2;
};

// ---------------------------------------------------------------------------
// Pass 1, 16-byte packs.  Thread owns packs j = j0 + k * js (k < VPT, j < nv).
// Returns this thread's share of the sum of squares; hv receives the row
// values as stored in the residual (or x for the plain form).
// ---------------------------------------------------------------------------
template <typename T, int VPT, int OP, typename TR>
__device__ __forceinline__ float pass1_vec(const Problem &p, int64_t t, int j0, int js, int nv,
                                           uint4 (&hv)[VPT][Res<T, TR>::N]) {
    using RS = Res<T, TR>;
    constexpr int EPV = DT<T>::EPV;
    constexpr int RC = Chunk<OP>::value;
    const int64_t xo = t * p.ldx;
    float ss = 0.f;
    if constexpr (OP == OP_PLAIN) {
        const T *x = reinterpret_cast<const T *>(p.src) + xo;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * js;
            if (j < nv) hv[k][0] = ld_stream(x + (int64_t)j * EPV);
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * js;
            if (j < nv) {
                float f[EPV];
                DT<T>::unpack(hv[k][0], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) ss += f[e] * f[e];
            }
        }
        return ss;
    } else {
        TR *res = reinterpret_cast<TR *>(p.residual) + t * p.ldr;
        float acc[VPT][EPV];
        if constexpr (RS::SAME) {
            // streams 0..R-1 are the partials (x for fused), stream R the
            // residual; RC streams are loaded together
            const int S = p.R + 1;
            for (int s0 = 0; s0 < S; s0 += RC) {
                uint4 buf[RC][VPT];
#pragma unroll
                for (int q = 0; q < RC; ++q) {
                    if (s0 + q < S) {
                        const T *base =
                            s0 + q == p.R
                                ? reinterpret_cast<const T *>(res)
                                : reinterpret_cast<const T *>(p.src) + (int64_t)(s0 + q) * p.slice +
                                      xo;
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
        } else {
            // binary32 residual: its words are loaded first and added last
            uint4 rv[VPT][RS::N];
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = j0 + k * js;
                if (j < nv) {
#pragma unroll
                    for (int q = 0; q < RS::N; ++q)
                        rv[k][q] = ld_stream(res + (int64_t)j * EPV + q * RS::EPW);
                }
            }
            constexpr int PC = RC > 2 ? RC : 1;  // partials loaded together
            for (int s0 = 0; s0 < p.R; s0 += PC) {
                uint4 buf[PC][VPT];
#pragma unroll
                for (int q = 0; q < PC; ++q) {
                    if (s0 + q < p.R) {
                        const T *base =
                            reinterpret_cast<const T *>(p.src) + (int64_t)(s0 + q) * p.slice + xo;
#pragma unroll
                        for (int k = 0; k < VPT; ++k) {
                            const int j = j0 + k * js;
                            if (j < nv) buf[q][k] = ld_stream(base + (int64_t)j * EPV);
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < PC; ++q) {
                    if (s0 + q < p.R) {
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
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int j = j0 + k * js;
                if (j < nv) {
                    float f[EPV];
                    RS::to_f(rv[k], f);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) acc[k][e] = acc[k][e] + f[e];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int j = j0 + k * js;
            if (j < nv) {
                RS::from_f(acc[k], hv[k]);  // the one rounding to the residual's type
#pragma unroll
                for (int q = 0; q < RS::N; ++q)
                    st_global(res + (int64_t)j * EPV + q * RS::EPW, hv[k][q]);
                float f[EPV];
                RS::to_f(hv[k], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) ss += f[e] * f[e];
            }
        }
        return ss;
    }
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
// Q8: y holds 8-bit codes of ((h * inv) * gamma * m1) * m2 instead (EPV bytes
// per pack).
template <typename T, int VPT, typename TR, bool PG = false, bool Q8 = false>
__device__ __forceinline__ void pass2_vec(const Problem &p, int64_t t, int j0, int js, int nv,
                                          const uint4 (&hv)[VPT][Res<T, TR>::N], float inv,
                                          const uint4 *gv = nullptr, QMul qm = QMul{1.f, 1.f}) {
    constexpr int EPV = DT<T>::EPV;
    const T *g = reinterpret_cast<const T *>(p.gamma);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            float h[EPV], w[EPV];
            Res<T, TR>::to_f(hv[k], h);
            DT<T>::unpack(PG ? gv[k] : ld_keep(g + (int64_t)j * EPV), w);
#pragma unroll
            for (int e = 0; e < EPV; ++e) h[e] = (h[e] * inv) * w[e];
            if constexpr (Q8) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) h[e] = (h[e] * qm.m1) * qm.m2;
                st_codes<EPV>(reinterpret_cast<uint8_t *>(p.y) + t * p.ldy + (int64_t)j * EPV, h,
                              p.qfmt);
            } else {
                st_global(reinterpret_cast<T *>(p.y) + t * p.ldy + (int64_t)j * EPV,
                          DT<T>::pack(h));
            }
        }
    }
}

// Per-row scale: this thread's max |h * gamma| over its packs (times inv > 0
// after the row reduction, the row's max |v|).
template <typename T, int VPT, typename TR, bool PG>
__device__ __forceinline__ float amax_vec(const Problem &p, int j0, int js, int nv,
                                          const uint4 (&hv)[VPT][Res<T, TR>::N],
                                          const uint4 *gv) {
    constexpr int EPV = DT<T>::EPV;
    const T *g = reinterpret_cast<const T *>(p.gamma);
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            float h[EPV], w[EPV];
            Res<T, TR>::to_f(hv[k], h);
            DT<T>::unpack(PG ? gv[k] : ld_keep(g + (int64_t)j * EPV), w);
#pragma unroll
            for (int e = 0; e < EPV; ++e) m = fmaxf(m, fabsf(h[e] * w[e]));
        }
    }
    return m;
}

// ---------------------------------------------------------------------------
// Pass 1 / pass 2, single elements (rows or pointers not 16-byte aligned).
// Thread owns elements i = i0 + k * is (k < NE, i < H); values held as
// binary32 (already rounded to the residual's storage type).
// ---------------------------------------------------------------------------
template <typename T, int NE, int OP, typename TR>
__device__ __forceinline__ float pass1_scalar(const Problem &p, int64_t t, int i0, int is,
                                              float (&h)[NE]) {
    constexpr int RC = Chunk<OP>::value;
    const int64_t xo = t * p.ldx;
    const int H = (int)p.H;
    float ss = 0.f;
    if constexpr (OP == OP_PLAIN) {
        const T *x = reinterpret_cast<const T *>(p.src) + xo;
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int i = i0 + k * is;
            h[k] = i < H ? DT<T>::to_f(x[i]) : 0.f;
            ss += h[k] * h[k];
        }
        return ss;
    } else {
        TR *res = reinterpret_cast<TR *>(p.residual) + t * p.ldr;
        float rv[NE];
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int i = i0 + k * is;
            rv[k] = i < H ? DT<TR>::to_f(res[i]) : 0.f;
        }
        for (int s0 = 0; s0 < p.R; s0 += RC) {
            float buf[RC][NE];
#pragma unroll
            for (int q = 0; q < RC; ++q) {
                if (s0 + q < p.R) {
                    const T *base =
                        reinterpret_cast<const T *>(p.src) + (int64_t)(s0 + q) * p.slice + xo;
#pragma unroll
                    for (int k = 0; k < NE; ++k) {
                        const int i = i0 + k * is;
                        buf[q][k] = i < H ? DT<T>::to_f(base[i]) : 0.f;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < RC; ++q) {
                if (s0 + q < p.R) {
#pragma unroll
                    for (int k = 0; k < NE; ++k)
                        h[k] = (s0 + q == 0) ? buf[q][k] : h[k] + buf[q][k];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int i = i0 + k * is;
            if (i < H) {
                const TR r = DT<TR>::from_f(h[k] + rv[k]);  // one rounding to TR
                res[i] = r;
                h[k] = DT<TR>::to_f(r);
                ss += h[k] * h[k];
            }
        }
        return ss;
    }
}

template <typename T, int NE, bool Q8 = false>
__device__ __forceinline__ void pass2_scalar(const Problem &p, int64_t t, int i0, int is,
                                             const float (&h)[NE], float inv,
                                             QMul qm = QMul{1.f, 1.f}) {
    const T *g = reinterpret_cast<const T *>(p.gamma);
    const int H = (int)p.H;
#pragma unroll
    for (int k = 0; k < NE; ++k) {
        const int i = i0 + k * is;
        if (i < H) {
            const float v = (h[k] * inv) * DT<T>::to_f(g[i]);
            if constexpr (Q8)
                reinterpret_cast<uint8_t *>(p.y)[t * p.ldy + i] =
                    fp8x1((v * qm.m1) * qm.m2, p.qfmt);
            else
                reinterpret_cast<T *>(p.y)[t * p.ldy + i] = DT<T>::from_f(v);
        }
    }
}

template <typename T, int NE>
__device__ __forceinline__ float amax_scalar(const Problem &p, int i0, int is,
                                             const float (&h)[NE]) {
    const T *g = reinterpret_cast<const T *>(p.gamma);
    const int H = (int)p.H;
    float m = 0.f;
#pragma unroll
    for (int k = 0; k < NE; ++k) {
        const int i = i0 + k * is;
        if (i < H) m = fmaxf(m, fabsf(h[k] * DT<T>::to_f(g[i])));
    }
    return m;
}

// The row's reciprocal RMS from this thread's share ss of the sum of squares
// (CTA-wide).  With a per-row 8-bit scale, am is this thread's share of
// max |h * gamma|: it is reduced in the same pass (one barrier) and qm
// receives the row's multipliers.  red / red2 alternate between rows.
template <bool Q8>
__device__ __forceinline__ float row_inv_cta(const Problem &p, int64_t t, float ss, float am,
                                             float *red, float2 *red2, QMul &qm) {
    if constexpr (Q8) {
        if (p.qmode == Q_ROW) {
            const float2 r = block_sum_max(ss, am, red2);
            const float inv = rsqrtf(r.x / (float)p.H + p.eps);
            qm = quant_row(p, t, r.y * inv, threadIdx.x == 0);
            return inv;
        }
    }
    return rsqrtf(block_sum(ss, red) / (float)p.H + p.eps);
}

// The same for a warp per row.
template <bool Q8>
__device__ __forceinline__ float row_inv_warp(const Problem &p, int64_t t, float ss, float am,
                                              QMul &qm) {
    const float inv = rsqrtf(warp_sum(ss) / (float)p.H + p.eps);
    if constexpr (Q8) {
        if (p.qmode == Q_ROW) qm = quant_row(p, t, warp_max(am) * inv, (threadIdx.x & 31) == 0);
    }
    return inv;
}

// CTA size each register-staged kernel is compiled for (plan.h budget); a
// combination over budget is compiled for 128 threads and never planned.
template <typename T, int VPT, int OP, bool PG, typename TR>
struct VecBound {
    static constexpr int b =
        rows_max_block(rows_regs_vec(VPT, DT<T>::EPV, OP, PG, Res<T, TR>::N));
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

// Row t's inputs (x, or the R partials, and the residual) prefetched into L2
// by one thread before grid_dependency_wait(); rows of the 16-byte kernels
// start on 16-byte boundaries and are multiples of 16 bytes long.
template <typename T, int OP, typename TR>
__device__ __forceinline__ void prefetch_row_l2(const Problem &p, int64_t t) {
    if (t >= p.T) return;
    const T *src = reinterpret_cast<const T *>(p.src);
    const uint32_t xb = static_cast<uint32_t>(p.H * sizeof(T));
    if constexpr (OP == OP_REDUCE) {
        for (int r = 0; r < p.R; ++r) prefetch_l2(src + r * p.slice + t * p.ldx, xb);
    } else {
        prefetch_l2(src + t * p.ldx, xb);
    }
    if constexpr (OP != OP_PLAIN)
        prefetch_l2(reinterpret_cast<const TR *>(p.residual) + t * p.ldr,
                    static_cast<uint32_t>(p.H * sizeof(TR)));
}

// Rows t0, t0 + step, ... (p.l2_rows of them, at most 32) of one CTA
// prefetched into L2 before grid_dependency_wait(), one row per thread.
template <typename T, int OP, typename TR>
__device__ __forceinline__ void prefetch_rows_l2(const Problem &p, int64_t t0, int64_t step) {
    if ((int)threadIdx.x < p.l2_rows && threadIdx.x < 32)
        prefetch_row_l2<T, OP, TR>(p, t0 + (int64_t)threadIdx.x * step);
}

// One CTA per row, packs.  PG: gamma held in registers for all rows.  Q8:
// 8-bit output; a per-row scale takes a second CTA reduction (max |v|).
template <typename T, int VPT, int OP, bool PG, typename TR, bool Q8>
__global__ void __launch_bounds__(VecBound<T, VPT, OP, PG, TR>::value) k_cta_vec(Problem p) {
    __shared__ float red[2][32];
    __shared__ float2 red2[Q8 ? 64 : 1];
    const int nv = (int)(p.H / DT<T>::EPV);
    prefetch_rows_l2<T, OP, TR>(p, blockIdx.x, gridDim.x);
    grid_dependency_wait();
    QMul qm{1.f, 1.f};
    if constexpr (Q8) qm = quant_tensor(p);
    const bool qrow = Q8 && p.qmode == Q_ROW;
    uint4 gv[VPT];
    if (PG) load_gamma_vec<T, VPT>(p, threadIdx.x, blockDim.x, nv, gv);
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        uint4 hv[VPT][Res<T, TR>::N];
        const float ss = pass1_vec<T, VPT, OP, TR>(p, t, threadIdx.x, blockDim.x, nv, hv);
        const float am =
            qrow ? amax_vec<T, VPT, TR, PG>(p, threadIdx.x, blockDim.x, nv, hv, gv) : 0.f;
        const float inv = row_inv_cta<Q8>(p, t, ss, am, red[par], red2 + 32 * par, qm);
        pass2_vec<T, VPT, TR, PG, Q8>(p, t, threadIdx.x, blockDim.x, nv, hv, inv, gv, qm);
    }
}

// One CTA per row, packs, software-pipelined across rows (plain and fused
// forms: one input stream plus the residual).  Before a CTA reduces and
// writes row t it issues the loads of its next row into a second register
// buffer, so the SM keeps reads in flight through the row reduction and the
// y stores instead of draining between rows.
template <typename T, int VPT, int OP, typename TR>
struct RowLoads {
    static constexpr int RN = OP == OP_PLAIN ? 0 : Res<T, TR>::N;  // residual words per pack
    uint4 x[VPT];
    uint4 r[VPT][RN > 0 ? RN : 1];
};

template <typename T, int VPT, int OP, typename TR>
__device__ __forceinline__ void issue_row_loads(const Problem &p, int64_t t, int j0, int js,
                                                int nv, RowLoads<T, VPT, OP, TR> &b) {
    constexpr int EPV = DT<T>::EPV;
    constexpr int RN = RowLoads<T, VPT, OP, TR>::RN;
    const T *x = reinterpret_cast<const T *>(p.src) + t * p.ldx;
    const TR *res = reinterpret_cast<const TR *>(p.residual) + t * p.ldr;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            b.x[k] = ld_stream(x + (int64_t)j * EPV);
#pragma unroll
            for (int q = 0; q < RN; ++q)
                b.r[k][q] = ld_stream(res + (int64_t)j * EPV + q * Res<T, TR>::EPW);
        }
    }
}

// h from the loaded packs (fused: x + residual in binary32, one rounding to
// the residual's type, residual written back); returns this thread's share of
// the sum of squares.
template <typename T, int VPT, int OP, typename TR>
__device__ __forceinline__ float consume_row_loads(const Problem &p, int64_t t, int j0, int js,
                                                   int nv, const RowLoads<T, VPT, OP, TR> &b,
                                                   uint4 (&hv)[VPT][Res<T, TR>::N]) {
    using RS = Res<T, TR>;
    constexpr int EPV = DT<T>::EPV;
    TR *res = reinterpret_cast<TR *>(p.residual) + t * p.ldr;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int j = j0 + k * js;
        if (j < nv) {
            float h[EPV];
            DT<T>::unpack(b.x[k], h);
            if constexpr (OP == OP_FUSED) {
                float r[EPV];
                RS::to_f(b.r[k], r);
#pragma unroll
                for (int e = 0; e < EPV; ++e) h[e] = h[e] + r[e];
                RS::from_f(h, hv[k]);  // the one rounding to the residual's type
#pragma unroll
                for (int q = 0; q < RS::N; ++q)
                    st_global(res + (int64_t)j * EPV + q * RS::EPW, hv[k][q]);
                RS::to_f(hv[k], h);
            } else {
                hv[k][0] = b.x[k];
            }
#pragma unroll
            for (int e = 0; e < EPV; ++e) ss += h[e] * h[e];
        }
    }
    return ss;
}

template <typename T, int VPT, int OP, typename TR>
struct PipeBound {
    static constexpr int streams = 1 + RowLoads<T, VPT, OP, TR>::RN;
    static constexpr int b = rows_max_block(
        rows_regs_vec(VPT, DT<T>::EPV, OP, false, Res<T, TR>::N) + VPT * 4 * streams);
    static constexpr int value = b > 0 ? b : 128;
};

template <typename T, int VPT, int OP, typename TR, bool Q8>
__global__ void __launch_bounds__(PipeBound<T, VPT, OP, TR>::value) k_cta_pipe(Problem p) {
    __shared__ float red[2][32];
    __shared__ float2 red2[Q8 ? 64 : 1];
    const int nv = (int)(p.H / DT<T>::EPV);
    prefetch_rows_l2<T, OP, TR>(p, blockIdx.x, gridDim.x);
    grid_dependency_wait();
    QMul qm{1.f, 1.f};
    if constexpr (Q8) qm = quant_tensor(p);
    const bool qrow = Q8 && p.qmode == Q_ROW;
    // gamma in registers (with an 8-bit output the row maximum uses it too),
    // up to 4 packs per thread with a residual of type T (measured: C3
    // 21.84 -> 21.64 us; with a binary32 residual the extra registers cost a
    // CTA per SM: 302 -> 352 us, so not there)
    constexpr bool PGP = Q8 || (VPT <= 4 && std::is_same<T, TR>::value);
    uint4 gv[VPT];
    if constexpr (PGP) load_gamma_vec<T, VPT>(p, threadIdx.x, blockDim.x, nv, gv);
    RowLoads<T, VPT, OP, TR> next;
    int64_t t = blockIdx.x;
    if (t < p.T) issue_row_loads<T, VPT, OP, TR>(p, t, threadIdx.x, blockDim.x, nv, next);
    int par = 0;
    for (; t < p.T; t += gridDim.x, par ^= 1) {
        const RowLoads<T, VPT, OP, TR> cur = next;
        if (t + gridDim.x < p.T) {
            issue_row_loads<T, VPT, OP, TR>(p, t + gridDim.x, threadIdx.x, blockDim.x, nv, next);
        } else {
            grid_launch_dependents();
        }
        uint4 hv[VPT][Res<T, TR>::N];
        const float ss =
            consume_row_loads<T, VPT, OP, TR>(p, t, threadIdx.x, blockDim.x, nv, cur, hv);
        const float am =
            qrow ? amax_vec<T, VPT, TR, PGP>(p, threadIdx.x, blockDim.x, nv, hv, gv) : 0.f;
        const float inv = row_inv_cta<Q8>(p, t, ss, am, red[par], red2 + 32 * par, qm);
        pass2_vec<T, VPT, TR, PGP, Q8>(p, t, threadIdx.x, blockDim.x, nv, hv, inv, gv, qm);
    }
}

// One warp per row, packs; blockDim.x / 32 rows per CTA at a time.  Gamma is
// held in registers (at most 4 packs per lane).
template <typename T, int VPT, int OP, typename TR, bool Q8>
__global__ void __launch_bounds__(256) k_warp_vec(Problem p) {
    const int nv = (int)(p.H / DT<T>::EPV);
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int64_t first = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const int64_t step = (int64_t)gridDim.x * wpb;
    if (lane == 0 && p.l2_rows > 0) prefetch_row_l2<T, OP, TR>(p, first);
    grid_dependency_wait();
    QMul qm{1.f, 1.f};
    if constexpr (Q8) qm = quant_tensor(p);
    const bool qrow = Q8 && p.qmode == Q_ROW;
    uint4 gv[VPT];
    load_gamma_vec<T, VPT>(p, lane, 32, nv, gv);
    for (int64_t t = first; t < p.T; t += step) {
        if (t + step >= p.T) grid_launch_dependents();
        uint4 hv[VPT][Res<T, TR>::N];
        const float ss = pass1_vec<T, VPT, OP, TR>(p, t, lane, 32, nv, hv);
        const float am = qrow ? amax_vec<T, VPT, TR, true>(p, lane, 32, nv, hv, gv) : 0.f;
        const float inv = row_inv_warp<Q8>(p, t, ss, am, qm);
        pass2_vec<T, VPT, TR, true, Q8>(p, t, lane, 32, nv, hv, inv, gv, qm);
    }
}

// One warp per row, pipelined like k_cta_pipe (plain and fused): the next
// row's loads are in flight while this row is reduced and written.
template <typename T, int VPT, int OP, typename TR, bool Q8>
__global__ void __launch_bounds__(256) k_warp_pipe(Problem p) {
    const int nv = (int)(p.H / DT<T>::EPV);
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int64_t first = (int64_t)blockIdx.x * wpb + (threadIdx.x >> 5);
    const int64_t step = (int64_t)gridDim.x * wpb;
    if (lane == 0 && p.l2_rows > 0) prefetch_row_l2<T, OP, TR>(p, first);
    grid_dependency_wait();
    QMul qm{1.f, 1.f};
    if constexpr (Q8) qm = quant_tensor(p);
    const bool qrow = Q8 && p.qmode == Q_ROW;
    uint4 gv[VPT];
    load_gamma_vec<T, VPT>(p, lane, 32, nv, gv);
    RowLoads<T, VPT, OP, TR> next;
    int64_t t = first;
    if (t < p.T) issue_row_loads<T, VPT, OP, TR>(p, t, lane, 32, nv, next);
    for (; t < p.T; t += step) {
        const RowLoads<T, VPT, OP, TR> cur = next;
        if (t + step < p.T) {
            issue_row_loads<T, VPT, OP, TR>(p, t + step, lane, 32, nv, next);
        } else {
            grid_launch_dependents();
        }
        uint4 hv[VPT][Res<T, TR>::N];
        const float ss = consume_row_loads<T, VPT, OP, TR>(p, t, lane, 32, nv, cur, hv);
        const float am = qrow ? amax_vec<T, VPT, TR, true>(p, lane, 32, nv, hv, gv) : 0.f;
        const float inv = row_inv_warp<Q8>(p, t, ss, am, qm);
        pass2_vec<T, VPT, TR, true, Q8>(p, t, lane, 32, nv, hv, inv, gv, qm);
    }
}

// One CTA per row, single elements.
template <typename T, int NE, int OP, typename TR, bool Q8>
__global__ void __launch_bounds__(ScalarBound<NE, OP>::value, 1) k_cta_scalar(Problem p) {
    __shared__ float red[2][32];
    __shared__ float2 red2[Q8 ? 64 : 1];
    grid_dependency_wait();
    QMul qm{1.f, 1.f};
    if constexpr (Q8) qm = quant_tensor(p);
    const bool qrow = Q8 && p.qmode == Q_ROW;
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        float h[NE];
        const float ss = pass1_scalar<T, NE, OP, TR>(p, t, threadIdx.x, blockDim.x, h);
        const float am = qrow ? amax_scalar<T, NE>(p, threadIdx.x, blockDim.x, h) : 0.f;
        const float inv = row_inv_cta<Q8>(p, t, ss, am, red[par], red2 + 32 * par, qm);
        pass2_scalar<T, NE, Q8>(p, t, threadIdx.x, blockDim.x, h, inv, qm);
    }
}

// The stored row (the residual, or x for the plain form): pack or element j.
template <typename T, int OP, typename TR>
__device__ __forceinline__ void reload_vec(const Problem &p, int64_t t, int j,
                                           uint4 (&hv)[1][Res<T, TR>::N]) {
    using RS = Res<T, TR>;
    constexpr int EPV = DT<T>::EPV;
    if constexpr (OP == OP_PLAIN) {
        hv[0][0] = ld_stream(reinterpret_cast<const T *>(p.src) + t * p.ldx + (int64_t)j * EPV);
    } else {
        const TR *res = reinterpret_cast<const TR *>(p.residual) + t * p.ldr;
#pragma unroll
        for (int q = 0; q < RS::N; ++q) hv[0][q] = ld_stream(res + (int64_t)j * EPV + q * RS::EPW);
    }
}

template <typename T, int OP, typename TR>
__device__ __forceinline__ float reload_scalar(const Problem &p, int64_t t, int j) {
    return OP == OP_PLAIN ? ld_elem<T>(p.src, t * p.ldx + j) : ld_elem<TR>(p.residual, t * p.ldr + j);
}

// Rows too long for registers: pass 1 walks the row in tiles of blockDim
// packs (or elements); pass 2 re-reads the stored row (the residual, or x for
// the plain form) -- each thread re-reads only what it wrote itself.  A
// per-row 8-bit scale takes max |h * gamma| in pass 1.
template <typename T, int OP, bool VEC, typename TR, bool Q8>
__global__ void __launch_bounds__(1024) k_two_pass(Problem p) {
    using RS = Res<T, TR>;
    __shared__ float red[2][32];
    __shared__ float2 red2[Q8 ? 64 : 1];
    constexpr int EPV = VEC ? DT<T>::EPV : 1;
    const int n = (int)(p.H / EPV);
    grid_dependency_wait();
    QMul qm{1.f, 1.f};
    if constexpr (Q8) qm = quant_tensor(p);
    const bool qrow = Q8 && p.qmode == Q_ROW;
    int par = 0;
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x, par ^= 1) {
        if (t + gridDim.x >= p.T) grid_launch_dependents();
        float ss = 0.f, am = 0.f;
        for (int base = 0; base < n; base += blockDim.x) {
            const int j = base + threadIdx.x;
            if constexpr (VEC) {
                uint4 hv[1][RS::N];
                ss += pass1_vec<T, 1, OP, TR>(p, t, j, 1 << 30, n, hv);
                if (qrow) am = fmaxf(am, amax_vec<T, 1, TR, false>(p, j, 1 << 30, n, hv, nullptr));
            } else {
                float h[1];
                ss += pass1_scalar<T, 1, OP, TR>(p, t, j, 1 << 30, h);
                if (qrow) am = fmaxf(am, amax_scalar<T, 1>(p, j, 1 << 30, h));
            }
        }
        const float inv = row_inv_cta<Q8>(p, t, ss, am, red[par], red2 + 32 * par, qm);
        for (int base = 0; base < n; base += blockDim.x) {
            const int j = base + threadIdx.x;
            if (j >= n) break;
            if constexpr (VEC) {
                uint4 hv[1][RS::N];
                reload_vec<T, OP, TR>(p, t, j, hv);
                pass2_vec<T, 1, TR, false, Q8>(p, t, j, 1 << 30, n, hv, inv, nullptr, qm);
            } else {
                const float h[1] = {reload_scalar<T, OP, TR>(p, t, j)};
                pass2_scalar<T, 1, Q8>(p, t, j, 1 << 30, h, inv, qm);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Launcher: plan -> template instance
// ---------------------------------------------------------------------------

template <typename T, int OP, typename TR, bool Q8>
static cudaError_t launch_rows_op(const Problem &p, const Plan &pl, cudaStream_t st) {
    const dim3 g(pl.grid), b(pl.block);
    auto go = [&](auto kernel) { return launch_kernel(kernel, g, b, 0, st, pl.pdl, 1, p); };
    // combinations over the register budget are never planned: not built
    auto go_vec = [&](auto vpt, auto pg) {
        constexpr int V = decltype(vpt)::value;
        constexpr bool G = decltype(pg)::value;
        if constexpr (VecBound<T, V, OP, G, TR>::b > 0)
            return go(k_cta_vec<T, V, OP, G, TR, Q8>);
        else
            return cudaErrorInvalidValue;
    };
    auto go_pipe = [&](auto vpt) {
        constexpr int V = decltype(vpt)::value;
        if constexpr (PipeBound<T, V, OP, TR>::b > 0)
            return go(k_cta_pipe<T, V, OP, TR, Q8>);
        else
            return cudaErrorInvalidValue;
    };
    using V1 = std::integral_constant<int, 1>;
    using V2 = std::integral_constant<int, 2>;
    using V4 = std::integral_constant<int, 4>;
    using V8 = std::integral_constant<int, 8>;
    using PGt = std::true_type;
    using PGf = std::false_type;
    switch (pl.kind) {
    case KIND_WARP:
        if constexpr (OP != OP_REDUCE) {
            if (pl.pipe) {
                switch (pl.per_thread) {
                case 1: return go(k_warp_pipe<T, 1, OP, TR, Q8>);
                case 2: return go(k_warp_pipe<T, 2, OP, TR, Q8>);
                case 4: return go(k_warp_pipe<T, 4, OP, TR, Q8>);
                default: return cudaErrorInvalidValue;
                }
            }
        }
        switch (pl.per_thread) {
        case 1: return go(k_warp_vec<T, 1, OP, TR, Q8>);
        case 2: return go(k_warp_vec<T, 2, OP, TR, Q8>);
        case 4: return go(k_warp_vec<T, 4, OP, TR, Q8>);
        default: return cudaErrorInvalidValue;
        }
    case KIND_CTA:
        if constexpr (OP != OP_REDUCE) {
            if (pl.vec && pl.pipe) {
                switch (pl.per_thread) {
                case 1: return go_pipe(V1{});
                case 2: return go_pipe(V2{});
                case 4: return go_pipe(V4{});
                case 8: return go_pipe(V8{});
                default: return cudaErrorInvalidValue;
                }
            }
        }
        if (pl.vec && pl.prefetch_gamma) {
            switch (pl.per_thread) {
            case 1: return go_vec(V1{}, PGt{});
            case 2: return go_vec(V2{}, PGt{});
            case 4: return go_vec(V4{}, PGt{});
            case 8: return go_vec(V8{}, PGt{});
            default: return cudaErrorInvalidValue;
            }
        }
        if (pl.vec) {
            switch (pl.per_thread) {
            case 1: return go_vec(V1{}, PGf{});
            case 2: return go_vec(V2{}, PGf{});
            case 4: return go_vec(V4{}, PGf{});
            case 8: return go_vec(V8{}, PGf{});
            default: return cudaErrorInvalidValue;
            }
        }
        switch (pl.per_thread) {
        case 1: return go(k_cta_scalar<T, 1, OP, TR, Q8>);
        case 2: return go(k_cta_scalar<T, 2, OP, TR, Q8>);
        case 4: return go(k_cta_scalar<T, 4, OP, TR, Q8>);
        case 8: return go(k_cta_scalar<T, 8, OP, TR, Q8>);
        case 16: return go(k_cta_scalar<T, 16, OP, TR, Q8>);
        default: return cudaErrorInvalidValue;
        }
    case KIND_TWO_PASS:
        return pl.vec ? go(k_two_pass<T, OP, true, TR, Q8>) : go(k_two_pass<T, OP, false, TR, Q8>);
    default:
        return cudaErrorInvalidValue;
    }
}

// TR = T: every form.  TR = float with a 16-bit T: the fused and reduce forms
// (the plain form has no residual).
template <typename T, typename TR>
cudaError_t launch_rows(const Problem &p, const Plan &pl, cudaStream_t st) {
    cudaError_t e;
    switch (p.op) {
    case OP_PLAIN:
        if constexpr (!std::is_same<T, TR>::value) {
            return cudaErrorInvalidValue;
        } else {
            e = launch_rows_op<T, OP_PLAIN, T, false>(p, pl, st);
        }
        break;
    case OP_FUSED: e = launch_rows_op<T, OP_FUSED, TR, false>(p, pl, st); break;
    case OP_REDUCE: e = launch_rows_op<T, OP_REDUCE, TR, false>(p, pl, st); break;
    default: return cudaErrorInvalidValue;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

// 8-bit output (codes in p.y, scale in p.qscale): every form, residual of
// type T.
template <typename T>
cudaError_t launch_rows_q8(const Problem &p, const Plan &pl, cudaStream_t st) {
    cudaError_t e;
    switch (p.op) {
    case OP_PLAIN: e = launch_rows_op<T, OP_PLAIN, T, true>(p, pl, st); break;
    case OP_FUSED: e = launch_rows_op<T, OP_FUSED, T, true>(p, pl, st); break;
    case OP_REDUCE: e = launch_rows_op<T, OP_REDUCE, T, true>(p, pl, st); break;
    default: return cudaErrorInvalidValue;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rarn
