// cluster.cuh -- a thread-block cluster per row for long rows.
//
// The row is cut into CS contiguous segments, one per CTA of a cluster of CS
// CTAs (2, 4 or 8).  Each CTA runs the register-staged passes of rows.cuh on
// its segment; the CTAs' partial sums of squares meet through distributed
// shared memory: each CTA publishes its partial in its own shared memory, a
// hardware cluster barrier orders the writes, and every CTA reads all CS
// partials in rank order (the same order in every CTA, so all of them get the
// same total).  The row is read from HBM once and never re-read, even when it
// is too long for one CTA's registers, and a short batch of long rows spreads
// over CS times more SMs.
#pragma once

#include "rows.cuh"

namespace rarn {

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Hardware cluster barrier: release this thread's prior writes (shared memory
// included) to the cluster, acquire everyone else's.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float from the same shared-memory variable in CTA `rank` of this
// cluster.
__device__ __forceinline__ float ld_peer(const float *local, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <typename T, int VPT, int OP, bool PG, typename TR>
__global__ void __launch_bounds__(VecBound<T, VPT, OP, PG, TR>::value, 1) k_cluster_vec(Problem p) {
    __shared__ float red[2][32];
    __shared__ float part[2];
    const uint32_t rank = cluster_ctarank(), cs = cluster_nctarank();
    const int nv = (int)(p.H / DT<T>::EPV);
    const int seg = (nv + (int)cs - 1) / (int)cs;
    const int j_begin = (int)rank * seg;
    const int j_end = min(nv, j_begin + seg);
    const int64_t first = blockIdx.x / cs, step = gridDim.x / cs;
    grid_dependency_wait();
    uint4 gv[VPT];  // PG: this thread's gamma packs, the same for every row
    if (PG) load_gamma_vec<T, VPT>(p, j_begin + threadIdx.x, blockDim.x, j_end, gv);
    int par = 0;
    for (int64_t t = first; t < p.T; t += step, par ^= 1) {
        if (t + step >= p.T) grid_launch_dependents();
        uint4 hv[VPT][Res<T, TR>::N];
        const float ss =
            pass1_vec<T, VPT, OP, TR>(p, t, j_begin + threadIdx.x, blockDim.x, j_end, hv);
        const float mine = block_sum(ss, red[par]);
        if (threadIdx.x == 0) part[par] = mine;
        cluster_sync();
        float tot = 0.f;
        for (uint32_t r = 0; r < cs; ++r) tot += ld_peer(&part[par], r);
        const float inv = rsqrtf(tot / (float)p.H + p.eps);
        pass2_vec<T, VPT, TR, PG>(p, t, j_begin + threadIdx.x, blockDim.x, j_end, hv, inv, gv);
    }
    // no CTA leaves while a peer may still read its partials
    cluster_sync();
}

template <typename T, int OP, typename TR>
static cudaError_t launch_cluster_op(const Problem &p, const Plan &pl, cudaStream_t st) {
    const dim3 g(pl.grid), b(pl.block);
    // combinations over the register budget are never planned: not built
    auto go = [&](auto vpt, auto pg) {
        constexpr int V = decltype(vpt)::value;
        constexpr bool G = decltype(pg)::value;
        if constexpr (VecBound<T, V, OP, G, TR>::b > 0)
            return launch_kernel(k_cluster_vec<T, V, OP, G, TR>, g, b, 0, st, pl.pdl, pl.cluster,
                                 p);
        else
            return cudaErrorInvalidValue;
    };
    using V1 = std::integral_constant<int, 1>;
    using V2 = std::integral_constant<int, 2>;
    using V4 = std::integral_constant<int, 4>;
    using V8 = std::integral_constant<int, 8>;
    if (pl.prefetch_gamma) {
        switch (pl.per_thread) {
        case 1: return go(V1{}, std::true_type{});
        case 2: return go(V2{}, std::true_type{});
        case 4: return go(V4{}, std::true_type{});
        case 8: return go(V8{}, std::true_type{});
        default: return cudaErrorInvalidValue;
        }
    }
    switch (pl.per_thread) {
    case 1: return go(V1{}, std::false_type{});
    case 2: return go(V2{}, std::false_type{});
    case 4: return go(V4{}, std::false_type{});
    case 8: return go(V8{}, std::false_type{});
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, typename TR>
cudaError_t launch_cluster(const Problem &p, const Plan &pl, cudaStream_t st) {
    cudaError_t e;
    switch (p.op) {
    case OP_PLAIN:
        if constexpr (!std::is_same<T, TR>::value) {
            return cudaErrorInvalidValue;
        } else {
            e = launch_cluster_op<T, OP_PLAIN, T>(p, pl, st);
        }
        break;
    case OP_FUSED: e = launch_cluster_op<T, OP_FUSED, TR>(p, pl, st); break;
    case OP_REDUCE: e = launch_cluster_op<T, OP_REDUCE, TR>(p, pl, st); break;
    default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace rarn
