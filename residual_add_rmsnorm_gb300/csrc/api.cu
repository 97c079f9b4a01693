// api.cu -- the C ABI: argument checks, kernel planning, dispatch by dtype.
//
// Every entry point validates its arguments before touching the GPU, picks a
// kernel family from the shape (or the forced path), and enqueues exactly one
// kernel launch on the caller's stream.  No memory is allocated.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>

#include <unordered_map>

#include "../../include/rarn.h"
#include "gemm_plan.h"
#include "plan.h"
#include "q8in.cuh"
#include "tp.cuh"

namespace rarn {
// instantiated in q8in_{bf16,f16,f32}.cu
extern template cudaError_t launch_q8in<__nv_bfloat16>(const q8in::Params &,
                                                       const q8in::KernelChoice &, int, bool,
                                                       cudaStream_t);
extern template cudaError_t launch_q8in<__half>(const q8in::Params &, const q8in::KernelChoice &,
                                                int, bool, cudaStream_t);
extern template cudaError_t launch_q8in<float>(const q8in::Params &, const q8in::KernelChoice &,
                                               int, bool, cudaStream_t);
// instantiated in tp_{bf16,f16,f32}.cu
extern template cudaError_t tp_blocks_per_sm<__nv_bfloat16>(int64_t, int *);
extern template cudaError_t tp_blocks_per_sm<__half>(int64_t, int *);
extern template cudaError_t tp_blocks_per_sm<float>(int64_t, int *);
extern template cudaError_t launch_tp<__nv_bfloat16>(const tp::Params &, int, bool, bool,
                                                    cudaStream_t);
extern template cudaError_t launch_tp<__half>(const tp::Params &, int, bool, bool, cudaStream_t);
extern template cudaError_t launch_tp<float>(const tp::Params &, int, bool, bool, cudaStream_t);
}  // namespace rarn

using namespace rarn;

static_assert(RARN_TP_MAX_RANKS == tp::kMaxRanks, "rank limit");
static_assert(RARN_TP_SIGNAL_BYTES == tp::kMaxCtas * tp::kMaxRanks * 4, "signal pad size");

// Watchdog word: kernels with bounded waits record a timeout here.
__device__ unsigned int g_rarn_watchdog = 0;

// Scratch of the workspace-free GEMM entry point (rarn_gemm_add_rms_norm_noalloc):
// 4 MB reserved with the module, so that entry point allocates nothing.  In
// host code this name is only a stand-in: the device address comes from
// cudaGetSymbolAddress (gemm_scratch below), once per device.
constexpr int64_t kGemmScratchFloats = int64_t(1) << 20;
static __device__ __align__(256) float g_rarn_gemm_scratch[kGemmScratchFloats];

// Launch floor (rarn_launch_floor): everything a row kernel does besides its
// row work -- one thread per CTA prefetches the CTA's first row into L2, the
// CTA waits for the previous grid and lets the next one launch.
__global__ void k_launch_floor(const char *rows, uint32_t row_bytes) {
    if (threadIdx.x == 0 && rows) prefetch_l2(rows + (size_t)blockIdx.x * row_bytes, row_bytes);
    grid_dependency_wait();
    grid_launch_dependents();
}

namespace {

thread_local int t_last_cuda_error = 0;
std::atomic<int> g_path{RARN_PATH_AUTO};
std::atomic<int> g_pdl{1};
// test hook (rarn_test_stall): consumed by the next launch of the stream
// kernel or of the GEMM form
std::atomic<long long> g_stall_fill{-1};
std::atomic<unsigned long long> g_stall_limit_ns{0};

// Planner overrides (rarn_set_tuning): -1 is the planner's own choice.
struct Tuning {
    std::atomic<long long> v[RARN_TUNE_COUNT];
    Tuning() { reset(); }
    void reset() {
        for (auto &x : v) x.store(-1);
    }
    long long operator[](rarn_tuning k) const { return v[k].load(std::memory_order_relaxed); }
};
Tuning g_tune;

// The values each knob accepts besides -1.
bool tuning_value_ok(rarn_tuning k, long long x) {
    switch (k) {
    case RARN_TUNE_ROWS_PER_THREAD: return x == 1 || x == 2 || x == 4 || x == 8 || x == 16;
    case RARN_TUNE_ROWS_GRID: return x >= 1 && x <= 0x7fffffffLL;
    case RARN_TUNE_L2_ROWS: return x >= 0 && x <= 8;
    case RARN_TUNE_STREAM_PACKS: return x == 1 || x == 2 || x == 4;
    case RARN_TUNE_STREAM_GROUPS: return x == 1 || x == 2;
    case RARN_TUNE_GEMM_COLS: return x == 256 || x == 512;
    case RARN_TUNE_GEMM_SLAB: return x == 32 || x == 64;
    case RARN_TUNE_GEMM_CTAS_PER_SM: return x == 1 || x == 2;
    case RARN_TUNE_GEMM_PERSISTENT:
    case RARN_TUNE_GEMM_PAIR:
    case RARN_TUNE_GEMM_NORM_IN_EPILOGUE:
    case RARN_TUNE_FP8IN_RING:
    case RARN_TUNE_TP_PREFETCH: return x == 0 || x == 1;
    case RARN_TUNE_ROWS_PIPELINE:
    case RARN_TUNE_GEMM_TAIL_SPLIT:
    case RARN_TUNE_GEMM_SPLIT_K:
    case RARN_TUNE_FP8IN_PACK16: return x == 0;
    default: return false;
    }
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned int *watchdog = nullptr;
    float *gemm_scratch = nullptr;  // looked up at first use on this device
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

rarn_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return RARN_ERR_CUDA;
}

// Device properties and the watchdog word's device address, once per device.
rarn_status device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return RARN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int sms = 0, smem = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return cuda_fail(e);
        void *wd = nullptr;
        if ((e = cudaGetSymbolAddress(&wd, g_rarn_watchdog)) != cudaSuccess) return cuda_fail(e);
        d.num_sms = sms;
        d.max_smem_optin = smem;
        d.watchdog = static_cast<unsigned int *>(wd);
        d.ready = true;
    }
    *out = &d;
    return RARN_OK;
}

// The static GEMM scratch's device address on the current device.
rarn_status gemm_scratch(float **out) {
    DeviceInfo *d = nullptr;
    rarn_status st = device_info(&d);
    if (st != RARN_OK) return st;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!d->gemm_scratch) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_rarn_gemm_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        d->gemm_scratch = static_cast<float *>(p);
    }
    *out = d->gemm_scratch;
    return RARN_OK;
}

int elem_size(rarn_dtype dt) { return dt == RARN_F32 ? 4 : 2; }

int pow2_at_least(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int round_up(int64_t a, int64_t b) { return (int)(ceil_div(a, b) * b); }

// Register-staged kernels: a warp per row for short rows, a CTA per row up to
// the register budget, two passes beyond it.
// rn: residual words per pack (1, or 2 for a binary32 residual with 16-bit
// inputs).
Plan plan_rows(int op, int64_t T, int64_t H, int s, bool vec, int num_sms, int rn = 1) {
    Plan pl;
    pl.vec = vec;
    const int epv = vec ? 16 / s : 1;
    const int64_t n = H / epv;  // packs (vec) or elements (scalar) per row
    const int resident_threads = 2048;
    if (vec && n <= 128) {
        pl.kind = KIND_WARP;
        pl.per_thread = n <= 32 ? 1 : n <= 64 ? 2 : 4;
        pl.block = 256;
        // one warp per row; balanced like the CTA grid below
        const int64_t slots = (int64_t)num_sms * (resident_threads / 32);
        const int64_t rounds = ceil_div(T, slots);
        pl.grid = (int)ceil_div(ceil_div(T, rounds), pl.block / 32);
        // pipelined across rows (plain / fused) when every warp has several
        pl.pipe = op != OP_REDUCE && rounds >= 2 && g_tune[RARN_TUNE_ROWS_PIPELINE] != 0;
        return pl;
    }
    // values per thread: aim at 256 threads per row, powers of two, within
    // the register budget of the kernel compiled for that count
    auto max_block = [&](int pt, bool pg) {
        return vec ? rows_max_block(rows_regs_vec(pt, epv, op, pg, rn))
                   : (pg ? 0 : rows_max_block(rows_regs_scalar(pt, op)));
    };
    const int max_pt = vec ? 8 : 16;
    // a binary32 residual doubles the registers per pack of a reduce row:
    // spread it over twice the threads (measured: 293 vs 366 us at R = 8,
    // [8192, 8192]); plain / fused rows with at most one CTA per SM (one
    // latency-bound wave) over up to 1024 threads, so each thread issues
    // fewer loads before the row reduction (measured, fused bf16, us:
    // [1, 5120] 2.25 -> 1.97, [128, 5120] 2.91 -> 2.45, [64, 16384] 3.72 ->
    // 3.56)
    const int target = (op == OP_REDUCE && rn == 2) ? 512
                       : (op != OP_REDUCE && T <= num_sms) ? 1024 : 256;
    int pt = std::min(max_pt, pow2_at_least(ceil_div(n, target)));
    if (const long long f = g_tune[RARN_TUNE_ROWS_PER_THREAD]; f >= 1 && f <= max_pt) pt = (int)f;
    while (pt < max_pt && ceil_div(n, pt) > max_block(pt, false)) pt <<= 1;
    if (ceil_div(n, pt) > max_block(pt, false)) {
        pl.kind = KIND_TWO_PASS;
        pl.per_thread = 1;
        pl.block = 1024;
    } else {
        pl.kind = KIND_CTA;
        pl.per_thread = pt;
        pl.block = round_up(ceil_div(n, pt), 32);
    }
    // Balanced grid: every CTA gets ceil(T / slots) or one fewer rows, so the
    // last round is not a ragged partial wave (T = 4096 on 1216 slots would
    // otherwise leave 3 full rounds and a 37 % fourth one).
    const int64_t slots = (int64_t)num_sms * std::max(1, resident_threads / pl.block);
    const int64_t rounds = ceil_div(T, slots);
    pl.grid = (int)ceil_div(T, rounds);
    if (const long long f = g_tune[RARN_TUNE_ROWS_GRID]; f > 0)
        pl.grid = (int)std::min<int64_t>(f, T);
    // Gamma in registers when every CTA has a single row (latency-bound: the
    // gamma load then overlaps the row's loads instead of following the row
    // reduction) and the kernel's register budget allows it.
    pl.prefetch_gamma =
        pl.kind == KIND_CTA && pl.vec && rounds == 1 && pl.block <= max_block(pl.per_thread, true);
    // Software pipelining across rows (plain / fused): worth it when every
    // CTA has several rows; it holds a second set of load buffers.
    if (pl.kind == KIND_CTA && pl.vec && op != OP_REDUCE && rounds >= 2) {
        const int streams = op == OP_PLAIN ? 1 : 1 + rn;
        const int pipe_max = rows_max_block(rows_regs_vec(pl.per_thread, epv, op, false, rn) +
                                            pl.per_thread * 4 * streams);
        pl.pipe = pl.block <= pipe_max && g_tune[RARN_TUNE_ROWS_PIPELINE] != 0;
    }
    return pl;
}

// Persistent TMA-fed kernel: 16-byte aligned rows whose staged copy fits in
// shared memory next to at least two pipeline stages.
constexpr int64_t kStreamMaxRowBytes = 96 * 1024;
constexpr int kDefaultMaxSmem = 232448;  // opt-in shared memory per CTA on sm_100 / sm_103

// Packs per consumer thread per chunk: up to two (fewer, larger copies per
// producer iteration) while at least 4 stages fit; RARN_TUNE_STREAM_PACKS
// overrides it.
Plan plan_stream(int op, int64_t T, int64_t H, int R, int s, bool vec, int num_sms,
                 int max_smem, int groups) {
    Plan pl;
    const int64_t row_bytes = H * s;
    if (!vec || row_bytes > kStreamMaxRowBytes) return pl;
    const int ns = op == OP_PLAIN ? 1 : R + 1;
    const int64_t nv = row_bytes / 16;
    // two packs per thread measured best or equal everywhere (4 only for tests)
    int ppt = std::min<int64_t>(2, pow2_at_least(ceil_div(nv, stream::kConsumers)));
    if (const long long f = g_tune[RARN_TUNE_STREAM_PACKS]; f > 0) ppt = (int)f;
    for (; ppt >= 1; ppt >>= 1) {
        const int chunk = stream::chunk_bytes(ppt);
        for (int g = groups; g >= 1; --g) {
            int stages = stream::kMaxStages / g;  // per group
            while (stages >= 2 &&
                   stream::layout(stages, ns, (int)row_bytes, g, chunk).total > max_smem)
                --stages;
            if (stages < 2 || (ppt > 1 && stages < 4)) continue;
            pl.kind = KIND_STREAM;
            pl.vec = true;
            pl.per_thread = ppt;
            pl.groups = g;
            pl.block = stream::threads(g);
            pl.grid = (int)std::min<int64_t>(T, num_sms);
            pl.stages = stages;
            pl.chunk = chunk;
            pl.smem = stream::layout(stages, ns, (int)row_bytes, g, chunk).total;
            return pl;
        }
    }
    return Plan{};
}

// Cluster per row: the smallest cluster (2, 4, 8 CTAs) whose segments fit the
// register budget and, where possible, puts a CTA on every SM.
Plan plan_cluster(int op, int64_t T, int64_t H, int s, bool vec, int num_sms, int rn = 1) {
    Plan pl;
    if (!vec) return pl;
    const int epv = 16 / s;
    const int64_t n = H / epv;
    for (int cs = 2; cs <= 8; cs <<= 1) {
        const int64_t seg = ceil_div(n, cs);
        auto max_block = [&](int p, bool pg) {
            return rows_max_block(rows_regs_vec(p, epv, op, pg, rn));
        };
        int pt = std::min(8, pow2_at_least(ceil_div(seg, 256)));
        while (pt < 8 && ceil_div(seg, pt) > max_block(pt, false)) pt <<= 1;
        if (ceil_div(seg, pt) > max_block(pt, false)) continue;
        const bool fills = T * cs >= num_sms;
        if (!fills && cs < 8) {
            // a larger cluster spreads the rows over more SMs; keep looking
            // unless the segments would become tiny
            if (ceil_div(n, cs * 2) >= 64) continue;
        }
        pl.kind = KIND_CLUSTER;
        pl.vec = true;
        pl.cluster = cs;
        pl.per_thread = pt;
        pl.block = round_up(ceil_div(seg, pt), 32);
        const int64_t resident =
            std::max<int64_t>(1, (int64_t)num_sms * std::max(1, 2048 / pl.block) / cs);
        const int64_t rounds = ceil_div(T, resident);
        pl.grid = (int)(ceil_div(T, rounds) * cs);
        pl.prefetch_gamma = rounds == 1 && pl.block <= max_block(pt, true);
        return pl;
    }
    return pl;
}

// Consumer groups of the stream kernel when it is forced (RARN_TUNE_STREAM_GROUPS).
int stream_groups(int fallback) {
    const long long g = g_tune[RARN_TUNE_STREAM_GROUPS];
    if (g < 1) return fallback;
    return g > stream::kMaxGroups ? stream::kMaxGroups : (int)g;
}

// The automatic choice, from measurements on GB300 (cold L2, CUDA-graph
// timing over rotating input copies):
//  * enough rows to give every SM several (T >= 2 x #SM) and 16-byte rows:
//      - reduce (R >= 2): the TMA-fed stream kernel; it keeps R + 1 input
//        streams in flight without spending registers on them (one consumer
//        group from R >= 4, two below);
//      - plain / fused rows too long for one CTA's registers (> 2048
//        packs): the stream kernel instead of the two-pass kernel;
//      - otherwise the software-pipelined register kernel, which beats the
//        stream kernel for one or two input streams up to 32 KB rows;
//  * few rows: the register kernels, with a cluster per row where one CTA's
//    registers cannot hold the row.
Plan plan_auto(int op, int64_t T, int64_t H, int R, int s, bool vec, int num_sms, int max_smem,
               int rn) {
    const bool many = vec && T >= 2 * (int64_t)num_sms && rn == 1;  // stream: same types only
    if (many && op == OP_REDUCE && R >= 2) {
        Plan st = plan_stream(op, T, H, R, s, vec, num_sms, max_smem, R >= 4 ? 1 : 2);
        if (st.kind != KIND_NONE) return st;
    }
    Plan r = plan_rows(op, T, H, s, vec, num_sms, rn);
    if (r.kind == KIND_TWO_PASS && vec) {
        if (many) {
            Plan st = plan_stream(op, T, H, R, s, vec, num_sms, max_smem, op == OP_PLAIN ? 2 : 1);
            if (st.kind != KIND_NONE) return st;
        }
        Plan c = plan_cluster(op, T, H, s, vec, num_sms, rn);
        if (c.kind != KIND_NONE) return c;
    }
    return r;
}

// rn: residual words per pack (2 for a binary32 residual with 16-bit
// inputs: register and cluster kernels only).  q8: 8-bit output, built for
// the register row kernels only (warp, CTA, pipelined, two-pass).
Plan make_plan(int op, int64_t T, int64_t H, int R, rarn_dtype dt, bool vec, int num_sms,
               int max_smem, int path, int rn = 1, bool q8 = false) {
    const int s = elem_size(dt);
    if (q8) {
        if (rn != 1 || (path != RARN_PATH_AUTO && path != RARN_PATH_ROWS)) return Plan{};
        return plan_rows(op, T, H, s, vec, num_sms, 1);
    }
    switch (path) {
    case RARN_PATH_ROWS: return plan_rows(op, T, H, s, vec, num_sms, rn);
    case RARN_PATH_STREAM:
        if (rn != 1) return Plan{};
        return plan_stream(op, T, H, R, s, vec, num_sms, max_smem, stream_groups(1));
    case RARN_PATH_CLUSTER: return plan_cluster(op, T, H, s, vec, num_sms, rn);
    case RARN_PATH_AUTO: return plan_auto(op, T, H, R, s, vec, num_sms, max_smem, rn);
    default: return Plan{};
    }
}

const char *kind_name(int k) {
    switch (k) {
    case KIND_WARP: return "rows.warp";
    case KIND_CTA: return "rows.cta";
    case KIND_TWO_PASS: return "rows.two_pass";
    case KIND_STREAM: return "stream";
    case KIND_CLUSTER: return "cluster";
    default: return "none";
    }
}

bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared body of the three entry points.
// Device view of a range of host memory for the *_host entry points.
// Pinned host memory (cudaMemoryTypeHost, first and last byte, one
// contiguous mapping) is used through its device pointer; pageable memory
// (unregistered) only where the device reads it through the host's page
// tables, at the same address.  Device and managed memory are refused, and so
// is pageable memory elsewhere: RARN_ERR_INVALID_ARG, nothing launched.
rarn_status host_view(const void *p, int64_t bytes, bool pageable_ok, void **view) {
    const char *first = static_cast<const char *>(p);
    const char *last = first + (bytes - 1);
    cudaPointerAttributes a{}, b{};
    if (cudaPointerGetAttributes(&a, first) != cudaSuccess ||
        cudaPointerGetAttributes(&b, last) != cudaSuccess) {
        cudaGetLastError();  // not a sticky error: clear it
        return RARN_ERR_INVALID_ARG;
    }
    if (a.type == cudaMemoryTypeHost && b.type == cudaMemoryTypeHost && a.devicePointer &&
        b.devicePointer &&
        static_cast<const char *>(b.devicePointer) - static_cast<const char *>(a.devicePointer) ==
            bytes - 1) {
        *view = a.devicePointer;
        return RARN_OK;
    }
    if (pageable_ok && a.type == cudaMemoryTypeUnregistered &&
        b.type == cudaMemoryTypeUnregistered) {
        *view = const_cast<char *>(first);
        return RARN_OK;
    }
    return RARN_ERR_INVALID_ARG;
}

// One call, in its most general form.
struct Call {
    int op = OP_PLAIN;
    void *y = nullptr;
    int64_t ldy = 0;
    const void *src = nullptr;  // x, or partial 0
    int64_t ldx = 0;
    int64_t slice = 0;          // elements between partials
    int32_t R = 0;
    void *residual = nullptr;
    int64_t ldr = 0;
    const void *gamma = nullptr;
    int64_t T = 0, H = 0;
    float eps = 0.f;
    rarn_dtype dt = RARN_F32;   // x / partials, gamma, y
    rarn_dtype rdt = RARN_F32;  // residual
    void *stream = nullptr;
    bool host_buffers = false;
    // 8-bit output: y holds codes (ldy in bytes)
    bool q8 = false;
    int qfmt = 0;
    int qmode = 0;
    float *qscale = nullptr;
};

bool dtype_ok(rarn_dtype d) { return d == RARN_F32 || d == RARN_F16 || d == RARN_BF16; }

// Bytes spanned by T rows of H elements with row stride ld.
int64_t span_bytes(int64_t T, int64_t H, int64_t ld, int s) { return ((T - 1) * ld + H) * s; }

rarn_status run_ex(Call c) {
    const int op = c.op;
    if (!dtype_ok(c.dt) || !dtype_ok(c.rdt)) return RARN_ERR_INVALID_ARG;
    if (c.T < 0 || c.H <= 0 || !(c.eps >= 0.f) || std::isinf(c.eps)) return RARN_ERR_INVALID_ARG;
    if (op == OP_REDUCE && c.R < 1) return RARN_ERR_INVALID_ARG;
    if (c.H > RARN_MAX_H || c.T > RARN_MAX_T || c.R > RARN_MAX_R) return RARN_ERR_UNSUPPORTED;
    if (c.ldx < c.H || c.ldy < c.H || (op != OP_PLAIN && c.ldr < c.H) || c.slice < 0)
        return RARN_ERR_INVALID_ARG;
    if (c.T == 0) return RARN_OK;
    if (!c.y || !c.src || !c.gamma || (op != OP_PLAIN && !c.residual)) return RARN_ERR_INVALID_ARG;
    // storage types: all one type, or a binary32 residual with 16-bit inputs
    const bool mixed = op != OP_PLAIN && c.rdt != c.dt;
    if (mixed && !(c.rdt == RARN_F32 && (c.dt == RARN_F16 || c.dt == RARN_BF16)))
        return RARN_ERR_UNSUPPORTED;
    if (op == OP_PLAIN) c.rdt = c.dt;
    if (c.q8) {
        if ((c.qfmt != Q_E4M3 && c.qfmt != Q_E5M2) || (c.qmode != Q_TENSOR && c.qmode != Q_ROW) ||
            !c.qscale || c.host_buffers)
            return RARN_ERR_INVALID_ARG;
        if (mixed) return RARN_ERR_UNSUPPORTED;
        const int path = g_path.load();
        if (path == RARN_PATH_STREAM || path == RARN_PATH_CLUSTER) return RARN_ERR_UNSUPPORTED;
    }

    const int s = elem_size(c.dt), rs = elem_size(c.rdt);
    const int ys = c.q8 ? 1 : s;  // bytes per element of y
    const int64_t row_bytes = c.H * s;
    const int nsrc = op == OP_REDUCE ? c.R : 1;
    const int64_t ybytes = span_bytes(c.T, c.H, c.ldy, ys);
    const int64_t xbytes = span_bytes(c.T, c.H, c.ldx, s);
    const int64_t srcbytes = (int64_t)(nsrc - 1) * c.slice * s + xbytes;
    const int64_t rbytes = op != OP_PLAIN ? span_bytes(c.T, c.H, c.ldr, rs) : 0;
    // y may coincide exactly with x / partial 0 (same row stride); nothing
    // else may overlap an output (overlaps are judged on the row spans)
    const bool y_is_src = !c.q8 && c.y == c.src && c.ldy == c.ldx;
    if (!y_is_src && overlaps(c.y, ybytes, c.src, srcbytes)) return RARN_ERR_ALIAS;
    if (y_is_src && nsrc > 1 &&
        overlaps(c.y, ybytes, static_cast<const char *>(c.src) + c.slice * s,
                 srcbytes - c.slice * s))
        return RARN_ERR_ALIAS;
    if (overlaps(c.y, ybytes, c.gamma, row_bytes)) return RARN_ERR_ALIAS;
    if (op != OP_PLAIN) {
        if (overlaps(c.residual, rbytes, c.y, ybytes) ||
            overlaps(c.residual, rbytes, c.src, srcbytes) ||
            overlaps(c.residual, rbytes, c.gamma, row_bytes))
            return RARN_ERR_ALIAS;
    }
    if (c.q8) {
        // the scale (one value read, or T values written) overlaps no output,
        // and a written scale no input either
        const int64_t qbytes = c.qmode == Q_ROW ? c.T * 4 : 4;
        if (overlaps(c.qscale, qbytes, c.y, ybytes) ||
            (op != OP_PLAIN && overlaps(c.qscale, qbytes, c.residual, rbytes)))
            return RARN_ERR_ALIAS;
        if (c.qmode == Q_ROW && (overlaps(c.qscale, qbytes, c.src, srcbytes) ||
                                 overlaps(c.qscale, qbytes, c.gamma, row_bytes)))
            return RARN_ERR_ALIAS;
    }

    DeviceInfo *d = nullptr;
    rarn_status st = device_info(&d);
    if (st != RARN_OK) return st;

    if (c.host_buffers) {
        // Every buffer lives in host memory; the kernels read and write it
        // through its device mapping (over NVLink-C2C on Grace systems), so
        // the transfers happen inside the kernel.
        int pageable = 0;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                                   dev) != cudaSuccess)
            pageable = 0;
        void *vy, *vs, *vg, *vr = nullptr;
        if ((st = host_view(c.y, ybytes, pageable, &vy)) != RARN_OK) return st;
        if ((st = host_view(c.src, srcbytes, pageable, &vs)) != RARN_OK) return st;
        if ((st = host_view(c.gamma, row_bytes, pageable, &vg)) != RARN_OK) return st;
        if (op != OP_PLAIN && (st = host_view(c.residual, rbytes, pageable, &vr)) != RARN_OK)
            return st;
        c.y = vy;
        c.src = vs;
        c.gamma = vg;
        c.residual = vr;
    }

    // 16-byte packs: one pack of EPV = 16 / s inputs gives EPV bytes of codes
    const int yalign = c.q8 ? 16 / s : 16;
    const bool y_ok = reinterpret_cast<uintptr_t>(c.y) % yalign == 0 && (c.ldy * ys) % yalign == 0;
    const bool vec = y_ok && aligned16(c.src) && aligned16(c.gamma) &&
                     (c.ldx * s) % 16 == 0 && row_bytes % 16 == 0 &&
                     (nsrc == 1 || (c.slice * s) % 16 == 0) &&
                     (op == OP_PLAIN || (aligned16(c.residual) && (c.ldr * rs) % 16 == 0));
    const int rn = mixed ? 2 : 1;

    // Host-resident data: the register kernels keep more requests in flight
    // over the host link than the single-producer stream kernel (measured).
    const int path = c.host_buffers && g_path.load() == RARN_PATH_AUTO ? RARN_PATH_ROWS
                                                                       : g_path.load();
    Plan pl =
        make_plan(op, c.T, c.H, c.R, c.dt, vec, d->num_sms, d->max_smem_optin, path, rn, c.q8);
    if (c.host_buffers && path == RARN_PATH_ROWS && pl.kind == KIND_TWO_PASS && vec) {
        const Plan cl = plan_cluster(op, c.T, c.H, s, vec, d->num_sms, rn);
        if (cl.kind != KIND_NONE) pl = cl;
    }
    if (pl.kind == KIND_NONE) return RARN_ERR_UNSUPPORTED;

    Problem p{};
    p.y = c.y;
    p.src = c.src;
    p.residual = c.residual;
    p.gamma = c.gamma;
    p.T = c.T;
    p.H = c.H;
    p.ldx = c.ldx;
    p.ldr = op != OP_PLAIN ? c.ldr : c.H;
    p.ldy = c.ldy;
    p.slice = c.slice;
    p.R = op == OP_PLAIN ? 0 : (op == OP_FUSED ? 1 : c.R);
    p.op = op;
    p.eps = c.eps;
    p.watchdog = d->watchdog;
    p.wait_limit_ns = stream::kWaitLimitNs;
    p.stall_fill = -1;
    p.qscale = c.qscale;
    p.qfmt = c.qfmt;
    p.qmode = c.qmode;
    // each CTA's (or warp's) first row prefetched into L2 before the
    // dependency wait.  Measured (same process, CUDA-graph timing, µs, rows
    // prefetched 0 / 1 / 2 / 4): fused [4096, 4096] 21.49 / 20.96-21.23 /
    // 21.81 / 23.00 (more rows compete with the previous kernel's tail);
    // plain fp32 [512, 2048] 3.06 / 2.77; fused [128, 5120] 3.51 / 2.90;
    // fused [64, 16384] 4.52 / 3.71; the stream kernel unchanged
    p.l2_rows = c.host_buffers ? 0 : 1;
    if (const long long f = g_tune[RARN_TUNE_L2_ROWS]; f >= 0 && !c.host_buffers) p.l2_rows = (int)f;
    if (pl.kind == KIND_STREAM) {
        const long long f = g_stall_fill.exchange(-1);
        if (f >= 0) {
            p.stall_fill = f;
            p.wait_limit_ns = g_stall_limit_ns.load();
        }
    }
    pl.pdl = g_pdl.load() != 0;

    cudaStream_t cs = static_cast<cudaStream_t>(c.stream);
    cudaError_t e = cudaErrorInvalidValue;
    const int key = (int)c.dt * 4 + (int)c.rdt;  // (inputs, residual) storage types
    const int F32F32 = RARN_F32 * 4 + RARN_F32, F16F16 = RARN_F16 * 4 + RARN_F16,
              BF16BF16 = RARN_BF16 * 4 + RARN_BF16, F16F32 = RARN_F16 * 4 + RARN_F32,
              BF16F32 = RARN_BF16 * 4 + RARN_F32;
    switch (c.q8 ? -pl.kind : pl.kind) {
    case -KIND_WARP:
    case -KIND_CTA:
    case -KIND_TWO_PASS:
        if (key == F32F32) e = launch_rows_q8<float>(p, pl, cs);
        else if (key == F16F16) e = launch_rows_q8<__half>(p, pl, cs);
        else if (key == BF16BF16) e = launch_rows_q8<__nv_bfloat16>(p, pl, cs);
        else return RARN_ERR_UNSUPPORTED;
        break;
    case KIND_WARP:
    case KIND_CTA:
    case KIND_TWO_PASS:
        if (key == F32F32) e = launch_rows<float, float>(p, pl, cs);
        else if (key == F16F16) e = launch_rows<__half, __half>(p, pl, cs);
        else if (key == BF16BF16) e = launch_rows<__nv_bfloat16, __nv_bfloat16>(p, pl, cs);
        else if (key == F16F32) e = launch_rows<__half, float>(p, pl, cs);
        else if (key == BF16F32) e = launch_rows<__nv_bfloat16, float>(p, pl, cs);
        break;
    case KIND_STREAM:
        if (key == F32F32) e = launch_stream<float>(p, pl, cs);
        else if (key == F16F16) e = launch_stream<__half>(p, pl, cs);
        else if (key == BF16BF16) e = launch_stream<__nv_bfloat16>(p, pl, cs);
        else return RARN_ERR_UNSUPPORTED;
        break;
    case KIND_CLUSTER:
        if (key == F32F32) e = launch_cluster<float, float>(p, pl, cs);
        else if (key == F16F16) e = launch_cluster<__half, __half>(p, pl, cs);
        else if (key == BF16BF16) e = launch_cluster<__nv_bfloat16, __nv_bfloat16>(p, pl, cs);
        else if (key == F16F32) e = launch_cluster<__half, float>(p, pl, cs);
        else if (key == BF16F32) e = launch_cluster<__nv_bfloat16, float>(p, pl, cs);
        break;
    default: return RARN_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return RARN_OK;
}

// Dense row-major form of one call: every row stride H, partials T * H apart.
rarn_status run(int op, void *y, const void *src, int32_t R, void *residual, const void *gamma,
                int64_t T, int64_t H, float eps, rarn_dtype dt, void *stream,
                bool host_buffers = false) {
    Call c;
    c.op = op;
    c.y = y;
    c.ldy = H;
    c.src = src;
    c.ldx = H;
    c.slice = T * H;
    c.R = R;
    c.residual = residual;
    c.ldr = H;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = dt;
    c.rdt = dt;
    c.stream = stream;
    c.host_buffers = host_buffers;
    return run_ex(c);
}

}  // namespace

extern "C" {

rarn_status rarn_rms_norm(void *y, const void *x, const void *gamma, int64_t T, int64_t H,
                          float eps, rarn_dtype dt, void *stream) {
    return run(OP_PLAIN, y, x, 0, nullptr, gamma, T, H, eps, dt, stream);
}

rarn_status rarn_fused_add_rms_norm(void *y, const void *x, void *residual, const void *gamma,
                                    int64_t T, int64_t H, float eps, rarn_dtype dt,
                                    void *stream) {
    return run(OP_FUSED, y, x, 1, residual, gamma, T, H, eps, dt, stream);
}

rarn_status rarn_reduce_add_rms_norm(void *y, const void *partials, int32_t R, void *residual,
                                     const void *gamma, int64_t T, int64_t H, float eps,
                                     rarn_dtype dt, void *stream) {
    return run(OP_REDUCE, y, partials, R, residual, gamma, T, H, eps, dt, stream);
}

rarn_status rarn_rms_norm_host(void *y, const void *x, const void *gamma, int64_t T, int64_t H,
                               float eps, rarn_dtype dt, void *stream) {
    return run(OP_PLAIN, y, x, 0, nullptr, gamma, T, H, eps, dt, stream, true);
}

rarn_status rarn_fused_add_rms_norm_host(void *y, const void *x, void *residual,
                                         const void *gamma, int64_t T, int64_t H, float eps,
                                         rarn_dtype dt, void *stream) {
    return run(OP_FUSED, y, x, 1, residual, gamma, T, H, eps, dt, stream, true);
}

rarn_status rarn_reduce_add_rms_norm_host(void *y, const void *partials, int32_t R,
                                          void *residual, const void *gamma, int64_t T,
                                          int64_t H, float eps, rarn_dtype dt, void *stream) {
    return run(OP_REDUCE, y, partials, R, residual, gamma, T, H, eps, dt, stream, true);
}

rarn_status rarn_rms_norm_ex(rarn_rows y, rarn_rows x, const void *gamma, int64_t T, int64_t H,
                             float eps, void *stream) {
    if (y.dtype != x.dtype) return RARN_ERR_UNSUPPORTED;
    Call c;
    c.op = OP_PLAIN;
    c.y = y.data;
    c.ldy = y.row_stride;
    c.src = x.data;
    c.ldx = x.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = c.rdt = x.dtype;
    c.stream = stream;
    return run_ex(c);
}

rarn_status rarn_fused_add_rms_norm_ex(rarn_rows y, rarn_rows x, rarn_rows residual,
                                       const void *gamma, int64_t T, int64_t H, float eps,
                                       void *stream) {
    if (y.dtype != x.dtype) return RARN_ERR_UNSUPPORTED;
    Call c;
    c.op = OP_FUSED;
    c.y = y.data;
    c.ldy = y.row_stride;
    c.src = x.data;
    c.ldx = x.row_stride;
    c.R = 1;
    c.residual = residual.data;
    c.ldr = residual.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = x.dtype;
    c.rdt = residual.dtype;
    c.stream = stream;
    return run_ex(c);
}

rarn_status rarn_reduce_add_rms_norm_ex(rarn_rows y, rarn_rows partials, int64_t partial_stride,
                                        int32_t R, rarn_rows residual, const void *gamma,
                                        int64_t T, int64_t H, float eps, void *stream) {
    if (y.dtype != partials.dtype) return RARN_ERR_UNSUPPORTED;
    Call c;
    c.op = OP_REDUCE;
    c.y = y.data;
    c.ldy = y.row_stride;
    c.src = partials.data;
    c.ldx = partials.row_stride;
    c.slice = partial_stride;
    c.R = R;
    c.residual = residual.data;
    c.ldr = residual.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = partials.dtype;
    c.rdt = residual.dtype;
    c.stream = stream;
    return run_ex(c);
}

// 8-bit output forms: the general forms with y replaced by a code matrix.
static bool fp8_desc(const rarn_fp8_rows *y, Call &c) {
    if (!y) return false;
    c.q8 = true;
    c.y = y->data;
    c.ldy = y->row_stride;
    c.qfmt = (int)y->format;
    c.qmode = (int)y->scale_mode;
    c.qscale = y->scale;
    return true;
}

rarn_status rarn_rms_norm_fp8(const rarn_fp8_rows *y, rarn_rows x, const void *gamma, int64_t T,
                              int64_t H, float eps, void *stream) {
    Call c;
    if (!fp8_desc(y, c)) return RARN_ERR_INVALID_ARG;
    c.op = OP_PLAIN;
    c.src = x.data;
    c.ldx = x.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = c.rdt = x.dtype;
    c.stream = stream;
    return run_ex(c);
}

rarn_status rarn_fused_add_rms_norm_fp8(const rarn_fp8_rows *y, rarn_rows x, rarn_rows residual,
                                        const void *gamma, int64_t T, int64_t H, float eps,
                                        void *stream) {
    Call c;
    if (!fp8_desc(y, c)) return RARN_ERR_INVALID_ARG;
    c.op = OP_FUSED;
    c.src = x.data;
    c.ldx = x.row_stride;
    c.R = 1;
    c.residual = residual.data;
    c.ldr = residual.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = x.dtype;
    c.rdt = residual.dtype;
    c.stream = stream;
    return run_ex(c);
}

rarn_status rarn_reduce_add_rms_norm_fp8(const rarn_fp8_rows *y, rarn_rows partials,
                                         int64_t partial_stride, int32_t R, rarn_rows residual,
                                         const void *gamma, int64_t T, int64_t H, float eps,
                                         void *stream) {
    Call c;
    if (!fp8_desc(y, c)) return RARN_ERR_INVALID_ARG;
    c.op = OP_REDUCE;
    c.src = partials.data;
    c.ldx = partials.row_stride;
    c.slice = partial_stride;
    c.R = R;
    c.residual = residual.data;
    c.ldr = residual.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.eps = eps;
    c.dt = partials.dtype;
    c.rdt = residual.dtype;
    c.stream = stream;
    return run_ex(c);
}

// GEMM producer + fused residual-add RMSNorm: every matrix 16-bit, one type;
// 16-byte aligned bases and row strides; the caller's workspace holds the
// column tiles' partial sums of squares.
static GemmPlan gemm_plan_tuned(int64_t T, int64_t H, int64_t K, int num_sms,
                                bool no_splitk = false) {
    auto knob = [](rarn_tuning k) { return (int)g_tune[k]; };
    const int bk = std::max(0, knob(RARN_TUNE_GEMM_SLAB));
    const int ns = std::max(0, knob(RARN_TUNE_GEMM_COLS));
    const int ctas = std::max(0, knob(RARN_TUNE_GEMM_CTAS_PER_SM));
    const int splitk = no_splitk ? 0 : knob(RARN_TUNE_GEMM_SPLIT_K);
    return plan_gemm(T, H, K, bk, ns, ctas, knob(RARN_TUNE_GEMM_PERSISTENT), num_sms,
                     knob(RARN_TUNE_GEMM_PAIR), knob(RARN_TUNE_GEMM_NORM_IN_EPILOGUE),
                     knob(RARN_TUNE_GEMM_TAIL_SPLIT), splitk);
}

int64_t rarn_gemm_workspace_bytes(int64_t T, int64_t H) {
    if (T < 0 || H <= 0) return -1;
    return gemm_workspace_bytes(T, H);
}

// Every check of the GEMM form that does not involve the workspace, over all
// T rows: types, sizes, alignment, and overlaps between the outputs (y, the
// residual) and every other matrix.  RARN_OK with T == 0 means "nothing to
// do"; the workspace form adds its own workspace checks.
static rarn_status gemm_check(const rarn_rows &y, const rarn_rows &a, const rarn_rows &w,
                              const rarn_rows &residual, const void *gamma, int64_t T, int64_t H,
                              int64_t K, float eps) {
    const rarn_dtype dt = a.dtype;
    if (!dtype_ok(dt) || !dtype_ok(w.dtype) || !dtype_ok(y.dtype) || !dtype_ok(residual.dtype))
        return RARN_ERR_INVALID_ARG;
    if (w.dtype != dt || y.dtype != dt || residual.dtype != dt) return RARN_ERR_UNSUPPORTED;
    if (T < 0 || H <= 0 || K <= 0 || !(eps >= 0.f) || std::isinf(eps)) return RARN_ERR_INVALID_ARG;
    if (a.row_stride < K || w.row_stride < K || residual.row_stride < H || y.row_stride < H)
        return RARN_ERR_INVALID_ARG;
    if (T == 0) return RARN_OK;
    if (!y.data || !a.data || !w.data || !residual.data || !gamma) return RARN_ERR_INVALID_ARG;
    if (dt == RARN_F32) return RARN_ERR_UNSUPPORTED;  // the tensor path takes 16-bit operands
    if (T > (int64_t(1) << 31) - 128 || K > (int64_t(1) << 31) - 64) return RARN_ERR_UNSUPPORTED;
    if (plan_gemm(T, H, K).ns == 0) return RARN_ERR_UNSUPPORTED;
    auto al16 = [](const void *ptr, int64_t ld) { return aligned16(ptr) && (ld * 2) % 16 == 0; };
    if (!al16(a.data, a.row_stride) || !al16(w.data, w.row_stride) ||
        !al16(residual.data, residual.row_stride) || !al16(y.data, y.row_stride) ||
        !aligned16(gamma))
        return RARN_ERR_UNSUPPORTED;
    const int64_t yb = span_bytes(T, H, y.row_stride, 2), rb = span_bytes(T, H, residual.row_stride, 2);
    const int64_t ab = span_bytes(T, K, a.row_stride, 2), wb = span_bytes(H, K, w.row_stride, 2);
    const void *ins[3] = {a.data, w.data, gamma};
    const int64_t inb[3] = {ab, wb, H * 2};
    for (int j = 0; j < 3; ++j)
        if (overlaps(y.data, yb, ins[j], inb[j]) || overlaps(residual.data, rb, ins[j], inb[j]))
            return RARN_ERR_ALIAS;
    if (overlaps(y.data, yb, residual.data, rb)) return RARN_ERR_ALIAS;
    return RARN_OK;
}

// One validated GEMM-form call over T rows with a workspace of ws_bytes.
static rarn_status gemm_launch(const rarn_rows &y, const rarn_rows &a, const rarn_rows &w,
                               const rarn_rows &residual, const void *gamma, int64_t T, int64_t H,
                               int64_t K, float eps, void *workspace, size_t workspace_bytes,
                               const DeviceInfo *d, void *stream) {
    GemmPlan gp = gemm_plan_tuned(T, H, K, d->num_sms);
    if (gp.ns == 0) return RARN_ERR_UNSUPPORTED;
    // split K only where the workspace holds its partial products
    if (gp.splitk && ((int64_t)workspace_bytes < gemm_splitk_bytes(T, H, gp.splitk) ||
                      (reinterpret_cast<uintptr_t>(workspace) & 31u)))
        gp = gemm_plan_tuned(T, H, K, d->num_sms, /*no_splitk=*/true);
    GemmCall c{};
    c.a = a.data;
    c.lda = a.row_stride;
    c.w = w.data;
    c.ldw = w.row_stride;
    c.residual = residual.data;
    c.ldr = residual.row_stride;
    c.y = y.data;
    c.ldy = y.row_stride;
    c.gamma = gamma;
    c.T = T;
    c.H = H;
    c.K = K;
    c.eps = eps;
    c.ns = gp.ns;
    c.stages = gp.stages;
    c.bk = gp.bk;
    c.workspace = static_cast<float *>(workspace);
    c.num_sms = d->num_sms;
    c.persistent = gp.persistent;
    c.pair = gp.pair;
    c.splitk = gp.splitk;
    c.part = gp.splitk ? static_cast<float *>(workspace) + gemm_splitk_offset(T, H) : nullptr;
    // y in the epilogue where the planner picks it (long K, or a knob); the
    // launcher confirms it, and the tail split, against the clusters that
    // fit on this GPU
    c.fuse_norm = gp.fuse_norm;
    c.tail_split = g_tune[RARN_TUNE_GEMM_TAIL_SPLIT] != 0;
    c.wait_limit_ns = 2000000000ull;
    c.stall_fill = -1;
    {
        const long long f = g_stall_fill.exchange(-1);
        if (f >= 0) {
            c.stall_fill = f;
            c.wait_limit_ns = g_stall_limit_ns.load();
        }
    }
    c.pdl = g_pdl.load() != 0;
    c.watchdog = d->watchdog;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const cudaError_t e = a.dtype == RARN_BF16 ? launch_gemm_norm<__nv_bfloat16>(c, cs)
                                               : launch_gemm_norm<__half>(c, cs);
    if (e != cudaSuccess) return cuda_fail(e);
    return RARN_OK;
}

rarn_status rarn_gemm_add_rms_norm(rarn_rows y, rarn_rows a, rarn_rows w, rarn_rows residual,
                                   const void *gamma, int64_t T, int64_t H, int64_t K, float eps,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    rarn_status st = gemm_check(y, a, w, residual, gamma, T, H, K, eps);
    if (st != RARN_OK || T == 0) return st;
    if (!workspace) return RARN_ERR_INVALID_ARG;
    // at least the non-split kernels' workspace (split K runs only where the
    // workspace also holds its partial products); the span checked for
    // overlaps is what any plan could use of the workspace given
    const int64_t base = gemm_workspace_bytes_for(T, H);
    if ((int64_t)workspace_bytes < base || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return RARN_ERR_INVALID_ARG;
    const int room = H % 256 == 0 && H / 256 <= kGemmMaxTilesN ? splitk_room(T, (int)(H / 256)) : 0;
    const int64_t most = room ? gemm_splitk_bytes(T, H, room) : base;
    const int64_t ws = std::min<int64_t>((int64_t)workspace_bytes, most);
    const void *others[5] = {y.data, residual.data, a.data, w.data, gamma};
    const int64_t ob[5] = {span_bytes(T, H, y.row_stride, 2),
                           span_bytes(T, H, residual.row_stride, 2),
                           span_bytes(T, K, a.row_stride, 2), span_bytes(H, K, w.row_stride, 2),
                           H * 2};
    for (int j = 0; j < 5; ++j)
        if (overlaps(workspace, ws, others[j], ob[j])) return RARN_ERR_ALIAS;
    DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != RARN_OK) return st;
    return gemm_launch(y, a, w, residual, gamma, T, H, K, eps, workspace, workspace_bytes, d,
                       stream);
}

// Rows one launch sequence of the allocation-free GEMM entry point covers:
// its scratch holds one partial sum per row and 128 columns plus a counter per
// 128-row block; -1 for an unsupported H.
static int64_t noalloc_rows(int64_t H) {
    if (H <= 0 || plan_gemm(1, H, 64).ns == 0) return -1;
    return (kGemmScratchFloats - 16) / (H / 128 + 1) / 128 * 128;
}

int64_t rarn_gemm_noalloc_rows(int64_t H) { return noalloc_rows(H); }

rarn_status rarn_gemm_add_rms_norm_noalloc(rarn_rows y, rarn_rows a, rarn_rows w,
                                           rarn_rows residual, const void *gamma, int64_t T,
                                           int64_t H, int64_t K, float eps, void *stream) {
    // the whole call is checked once, over all T rows, before anything runs:
    // an overlap between different chunks' rows is refused like any other,
    // and no chunk is launched unless every chunk would be
    rarn_status st = gemm_check(y, a, w, residual, gamma, T, H, K, eps);
    if (st != RARN_OK || T == 0) return st;
    DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != RARN_OK) return st;
    float *scratch = nullptr;
    if ((st = gemm_scratch(&scratch)) != RARN_OK) return st;
    // rows per launch sequence that the scratch holds (partial sums and
    // row-block counters); later chunks reuse it in stream order
    const int64_t chunk = noalloc_rows(H);
    for (int64_t t0 = 0; t0 < T; t0 += chunk) {
        const int64_t rows = std::min(chunk, T - t0);
        auto shift = [t0](rarn_rows m) {
            m.data = static_cast<char *>(m.data) + t0 * m.row_stride * 2;
            return m;
        };
        st = gemm_launch(shift(y), shift(a), w, shift(residual), gamma, rows, H, K, eps, scratch,
                         kGemmScratchFloats * 4, d, stream);
        if (st != RARN_OK) return st;
    }
    return RARN_OK;
}

rarn_status rarn_reduce_add_rms_norm_fp8in(void *y, const void *partials, int32_t R,
                                           rarn_fp8_format format, const float *scales,
                                           void *residual, const void *gamma, int64_t T,
                                           int64_t H, float eps, rarn_dtype dt, void *stream) {
    if (!dtype_ok(dt) || (format != RARN_E4M3 && format != RARN_E5M2)) return RARN_ERR_INVALID_ARG;
    if (T < 0 || H <= 0 || R < 1 || !(eps >= 0.f) || std::isinf(eps)) return RARN_ERR_INVALID_ARG;
    if (T == 0) return RARN_OK;
    if (!y || !partials || !scales || !residual || !gamma) return RARN_ERR_INVALID_ARG;
    const int s = elem_size(dt);
    if (R > 16 || H % 8 != 0 || H > (dt == RARN_F32 ? 8192 : 16384)) return RARN_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(partials) & 7u) || !aligned16(residual) ||
        !aligned16(gamma) || !aligned16(y) || (reinterpret_cast<uintptr_t>(scales) & 3u))
        return RARN_ERR_UNSUPPORTED;
    const int64_t rows = T * H * s;
    const void *ins[3] = {partials, scales, gamma};
    const int64_t inb[3] = {(int64_t)R * T * H, (int64_t)R * 4, H * s};
    if (overlaps(y, rows, residual, rows)) return RARN_ERR_ALIAS;
    for (int i = 0; i < 3; ++i)
        if (overlaps(y, rows, ins[i], inb[i]) || overlaps(residual, rows, ins[i], inb[i]))
            return RARN_ERR_ALIAS;
    DeviceInfo *d = nullptr;
    rarn_status st = device_info(&d);
    if (st != RARN_OK) return st;
    q8in::Params p{};
    p.y = y;
    p.codes = static_cast<const uint8_t *>(partials);
    p.scales = scales;
    p.residual = residual;
    p.gamma = gamma;
    p.T = T;
    p.H = H;
    p.R = R;
    p.fmt = format == RARN_E4M3 ? 0 : 1;
    p.eps = eps;
    p.l2_rows = 1;
    p.watchdog = d->watchdog;
    p.wait_limit_ns = stream::kWaitLimitNs;
    p.stall_fill = -1;
    p.max_smem = d->max_smem_optin;
    const q8in::KernelChoice kc =
        q8in::choose_kernel(p, s, d->num_sms, (int)g_tune[RARN_TUNE_FP8IN_RING],
                            g_tune[RARN_TUNE_FP8IN_PACK16] != 0);
    if (kc.ring) {
        const long long f = g_stall_fill.exchange(-1);
        if (f >= 0) {
            p.stall_fill = f;
            p.wait_limit_ns = g_stall_limit_ns.load();
        }
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool pdl = g_pdl.load() != 0;
    cudaError_t e;
    switch (dt) {
    case RARN_BF16: e = launch_q8in<__nv_bfloat16>(p, kc, d->num_sms, pdl, cs); break;
    case RARN_F16: e = launch_q8in<__half>(p, kc, d->num_sms, pdl, cs); break;
    default: e = launch_q8in<float>(p, kc, d->num_sms, pdl, cs); break;
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return RARN_OK;
}

rarn_status rarn_plan_fp8in(int64_t T, int64_t H, int32_t R, rarn_dtype dt, int codes_aligned16,
                            int32_t num_sms, int32_t max_smem, char *out, size_t cap) {
    if (!out || cap == 0) return RARN_ERR_INVALID_ARG;
    if (!dtype_ok(dt) || T < 0 || H <= 0 || R < 1 || num_sms < 1 || max_smem < 0)
        return RARN_ERR_INVALID_ARG;
    if (R > 16 || H % 8 != 0 || H > (dt == RARN_F32 ? 8192 : 16384)) {
        snprintf(out, cap, "none: unsupported shape or type");
        return RARN_ERR_UNSUPPORTED;
    }
    const int s = elem_size(dt);
    const q8in::KernelChoice k =
        q8in::choose_kernel(T, H, R, s, codes_aligned16 != 0, num_sms, max_smem,
                            (int)g_tune[RARN_TUNE_FP8IN_RING], g_tune[RARN_TUNE_FP8IN_PACK16] != 0);
    if (k.ring) {
        const q8in::SLayout L =
            q8in::slayout(k.sp.stages, R, k.sp.ppt, s, H, q8in::kStreamWarps);
        snprintf(out, cap,
                 "q8in.ring warps=%d ppt=%d chunk_elems=%d stages=%d stage_bytes=%d smem=%d "
                 "grid=%lld block=%d",
                 q8in::kStreamWarps, k.sp.ppt, 32 * q8in::kStreamWarps * k.sp.ppt * 8,
                 k.sp.stages, L.stage_bytes, k.sp.smem,
                 (long long)std::min<int64_t>(T, num_sms), 32 + 32 * q8in::kStreamWarps);
    } else {
        snprintf(out, cap, "q8in.rows pack=%d vpt=%d block=%d grid=occupancy", k.pack, k.vpt,
                 k.block);
    }
    return RARN_OK;
}

rarn_status rarn_plan_gemm(int64_t T, int64_t H, int64_t K, rarn_dtype dt, int32_t num_sms,
                           char *out, size_t cap) {
    if (!out || cap == 0) return RARN_ERR_INVALID_ARG;
    if (!dtype_ok(dt) || T < 0 || H <= 0 || K <= 0) return RARN_ERR_INVALID_ARG;
    if (num_sms <= 0) {
        DeviceInfo *d = nullptr;
        const rarn_status st = device_info(&d);
        if (st != RARN_OK) return st;
        num_sms = d->num_sms;
    }
    const GemmPlan gp = dt == RARN_F32 ? GemmPlan{} : gemm_plan_tuned(T, H, K, num_sms);
    if (gp.ns == 0) {
        snprintf(out, cap, "none: unsupported shape or type");
        return RARN_ERR_UNSUPPORTED;
    }
    if (gp.splitk) {
        snprintf(out, cap,
                 "gemm.tcgen05 cols_per_cta=%d col_tiles=%d bk=%d stages=%d smem=%d grid=%lld "
                 "kblocks=%lld splitk=%d + split-K sum and norm",
                 gp.ns, gp.tiles_n, gp.bk, gp.stages, gp.smem, (long long)gp.grid,
                 (long long)((K + gp.bk - 1) / gp.bk), gp.splitk);
        return RARN_OK;
    }
    snprintf(out, cap,
             "gemm.tcgen05 cols_per_cta=%d col_tiles=%d bk=%d stages=%d smem=%d grid=%lld "
             "kblocks=%lld persistent=%d pair=%d%s %s",
             gp.ns, gp.tiles_n, gp.bk, gp.stages, gp.smem, (long long)gp.grid,
             (long long)((K + gp.bk - 1) / gp.bk), (int)gp.persistent, (int)gp.pair,
             gp.tail_split ? " tail=halves" : "", gp.fuse_norm ? "norm in epilogue" : "+ norm");
    return RARN_OK;
}

const char *rarn_status_string(rarn_status s) {
    switch (s) {
    case RARN_OK: return "ok";
    case RARN_ERR_INVALID_ARG: return "invalid argument";
    case RARN_ERR_UNSUPPORTED: return "unsupported size or kernel path";
    case RARN_ERR_ALIAS: return "output overlaps an input";
    case RARN_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
    }
}

int rarn_last_cuda_error(void) { return t_last_cuda_error; }

rarn_status rarn_set_path(rarn_path p) {
    if (p < RARN_PATH_AUTO || p > RARN_PATH_CLUSTER) return RARN_ERR_INVALID_ARG;
    g_path.store(p);
    return RARN_OK;
}

rarn_path rarn_get_path(void) { return static_cast<rarn_path>(g_path.load()); }

rarn_status rarn_set_pdl(int enable) {
    g_pdl.store(enable ? 1 : 0);
    return RARN_OK;
}

int rarn_get_pdl(void) { return g_pdl.load(); }

rarn_status rarn_set_tuning(rarn_tuning knob, int64_t value) {
    if ((int)knob < 0 || (int)knob >= RARN_TUNE_COUNT) return RARN_ERR_INVALID_ARG;
    if (value != -1 && !tuning_value_ok(knob, value)) return RARN_ERR_INVALID_ARG;
    g_tune.v[knob].store(value);
    return RARN_OK;
}

rarn_status rarn_get_tuning(rarn_tuning knob, int64_t *value) {
    if (!value || (int)knob < 0 || (int)knob >= RARN_TUNE_COUNT) return RARN_ERR_INVALID_ARG;
    *value = g_tune[knob];
    return RARN_OK;
}

rarn_status rarn_reset_tuning(void) {
    g_tune.reset();
    return RARN_OK;
}

rarn_status rarn_test_stall(long long fill, unsigned long long wait_limit_ns) {
    if (fill < 0 || wait_limit_ns == 0 || wait_limit_ns > stream::kWaitLimitNs)
        return RARN_ERR_INVALID_ARG;
    g_stall_limit_ns.store(wait_limit_ns);
    g_stall_fill.store(fill);
    return RARN_OK;
}

rarn_status rarn_plan(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt, int vec_ok,
                      int num_sms, char *out, size_t cap) {
    return rarn_plan_ex(op, T, H, R, dt, dt, vec_ok, num_sms, out, cap);
}

static rarn_status plan_text(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt,
                             rarn_dtype rdt, int vec_ok, int num_sms, char *out, size_t cap,
                             bool q8) {
    if (!out || cap == 0) return RARN_ERR_INVALID_ARG;
    if (op < RARN_OP_RMS_NORM || op > RARN_OP_REDUCE_ADD_RMS_NORM) return RARN_ERR_INVALID_ARG;
    if (!dtype_ok(dt) || !dtype_ok(rdt)) return RARN_ERR_INVALID_ARG;
    if (T < 0 || H <= 0 || (op == RARN_OP_REDUCE_ADD_RMS_NORM && R < 1))
        return RARN_ERR_INVALID_ARG;
    const bool mixed = op != RARN_OP_RMS_NORM && rdt != dt;
    if (mixed && (q8 || !(rdt == RARN_F32 && (dt == RARN_F16 || dt == RARN_BF16)))) {
        snprintf(out, cap, "none: unsupported storage types");
        return RARN_ERR_UNSUPPORTED;
    }
    int max_smem = kDefaultMaxSmem;
    if (num_sms <= 0) {
        DeviceInfo *d = nullptr;
        rarn_status st = device_info(&d);
        if (st != RARN_OK) return st;
        num_sms = d->num_sms;
        max_smem = d->max_smem_optin;
    }
    const bool vec = vec_ok && (H * elem_size(dt)) % 16 == 0;
    const Plan pl = make_plan((int)op, T, H, R, dt, vec, num_sms, max_smem, g_path.load(),
                              mixed ? 2 : 1, q8);
    snprintf(out, cap,
             "%s %s per_thread=%d block=%d grid=%d cluster=%d smem=%d stages=%d chunk=%d "
             "groups=%d gamma_regs=%d pipe=%d",
             kind_name(pl.kind), pl.vec ? "vec16" : "scalar", pl.per_thread, pl.block, pl.grid,
             pl.cluster, pl.smem, pl.stages, pl.chunk, pl.groups, (int)pl.prefetch_gamma,
             (int)pl.pipe);
    return pl.kind == KIND_NONE ? RARN_ERR_UNSUPPORTED : RARN_OK;
}

rarn_status rarn_plan_ex(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt,
                         rarn_dtype rdt, int vec_ok, int num_sms, char *out, size_t cap) {
    return plan_text(op, T, H, R, dt, rdt, vec_ok, num_sms, out, cap, false);
}

rarn_status rarn_plan_fp8(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt, int vec_ok,
                          int num_sms, char *out, size_t cap) {
    return plan_text(op, T, H, R, dt, dt, vec_ok, num_sms, out, cap, true);
}

rarn_status rarn_watchdog(uint32_t *flags, int clear) {
    if (!flags) return RARN_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_rarn_watchdog, sizeof(v))) != cudaSuccess)
        return cuda_fail(e);
    *flags = v;
    if (clear) {
        const unsigned int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_rarn_watchdog, &zero, sizeof(zero))) != cudaSuccess)
            return cuda_fail(e);
    }
    return RARN_OK;
}

int rarn_host_access(void) {
    int dev = 0, pageable = 0, mapped = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&mapped, cudaDevAttrCanMapHostMemory, dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                               dev) != cudaSuccess)
        return -1;
    return pageable ? 2 : (mapped ? 1 : 0);
}


// ---------------------------------------------------------------------------
// Tensor-parallel form
// ---------------------------------------------------------------------------

rarn_status rarn_tp_rows(int64_t T, int32_t world_size, int32_t rank, int64_t *r0, int64_t *r1) {
    if (T < 0 || world_size < 1 || rank < 0 || rank >= world_size || !r0 || !r1)
        return RARN_ERR_INVALID_ARG;
    tp::rows_of(T, world_size, rank, *r0, *r1);
    return RARN_OK;
}

// Whether the tensor-parallel kernel prefetches each CTA's next row into L2:
// the knob, else tp::prefetch_wanted.
static bool tp_prefetch(int per_sm, int N, int64_t row_bytes) {
    const long long f = g_tune[RARN_TUNE_TP_PREFETCH];
    return f >= 0 ? f != 0 : tp::prefetch_wanted(per_sm, N, row_bytes);
}

rarn_status rarn_plan_tp(int64_t T, int64_t H, int32_t world_size, rarn_dtype dt, int world,
                         int32_t num_sms, int32_t blocks_per_sm, char *out, size_t cap) {
    if (!out || cap == 0) return RARN_ERR_INVALID_ARG;
    if (!dtype_ok(dt) || T <= 0 || H <= 0 || world_size < 1 || world_size > RARN_TP_MAX_RANKS)
        return RARN_ERR_INVALID_ARG;
    const int s = elem_size(dt);
    if ((H * s) % 16 || H * s / 16 > tp::kMaxPacks) {
        snprintf(out, cap, "none: rows of H * sizeof(dt) bytes must be 16-byte packs, at most %d",
                 tp::kMaxPacks);
        return RARN_ERR_UNSUPPORTED;
    }
    if (num_sms <= 0) {
        DeviceInfo *d = nullptr;
        const rarn_status st = device_info(&d);
        if (st != RARN_OK) return st;
        num_sms = d->num_sms;
    }
    if (blocks_per_sm <= 0) {
        const cudaError_t e = dt == RARN_BF16 ? tp_blocks_per_sm<__nv_bfloat16>(H, &blocks_per_sm)
                              : dt == RARN_F16 ? tp_blocks_per_sm<__half>(H, &blocks_per_sm)
                                               : tp_blocks_per_sm<float>(H, &blocks_per_sm);
        if (e != cudaSuccess) return cuda_fail(e);
        if (blocks_per_sm < 1) return RARN_ERR_UNSUPPORTED;
    }
    int vpt = 0, block = 0;
    tp::tp_shape(H * s / 16, vpt, block);
    const int N = world_size;
    const int ctas = tp::ctas_per_rank(T, N, num_sms, blocks_per_sm, world != 0);
    snprintf(out, cap, "tp.%s ranks=%d ctas=%d block=%d vpt=%d blocks_per_sm=%d prefetch=%d",
             world ? "world" : "rank", N, ctas, block, vpt, blocks_per_sm,
             tp_prefetch(blocks_per_sm, N, H * s) ? 1 : 0);
    return RARN_OK;
}

// Checks of a tensor-parallel call (every rank's in the world launch, else
// group->rank's): before any CUDA call.
static rarn_status tp_check(const rarn_tp_group *g, void *const *residuals, const void *gamma,
                            int64_t T, int64_t H, float eps, rarn_dtype dt, bool world) {
    if (!g || g->world_size < 1 || g->world_size > RARN_TP_MAX_RANKS) return RARN_ERR_INVALID_ARG;
    const int N = g->world_size;
    if (!world && (g->rank < 0 || g->rank >= N)) return RARN_ERR_INVALID_ARG;
    if (!dtype_ok(dt) || T < 0 || H <= 0 || !(eps >= 0.f) || std::isinf(eps))
        return RARN_ERR_INVALID_ARG;
    if (T == 0) return RARN_OK;
    const int nsig = (int)std::count_if(g->signals, g->signals + N, [](uint32_t *s) { return s; });
    if (nsig != 0 && nsig != N) return RARN_ERR_INVALID_ARG;
    if (!gamma) return RARN_ERR_INVALID_ARG;
    // the residual of every rank this call runs that owns rows
    bool has_res[RARN_TP_MAX_RANKS] = {};
    for (int q = 0; q < N; ++q) {
        int64_t r0, r1;
        tp::rows_of(T, N, q, r0, r1);
        has_res[q] = (world || q == g->rank) && r1 > r0;
        if (!g->buffers[q]) return RARN_ERR_INVALID_ARG;
        if (has_res[q] && !residuals[q]) return RARN_ERR_INVALID_ARG;
    }
    const int s = elem_size(dt);
    if ((H * s) % 16 || H * s / 16 > tp::kMaxPacks) return RARN_ERR_UNSUPPORTED;
    if (!aligned16(gamma)) return RARN_ERR_UNSUPPORTED;
    for (int q = 0; q < N; ++q) {
        if (!aligned16(g->buffers[q])) return RARN_ERR_UNSUPPORTED;
        if (nsig && (reinterpret_cast<uintptr_t>(g->signals[q]) & 3u)) return RARN_ERR_UNSUPPORTED;
        if (has_res[q] && !aligned16(residuals[q])) return RARN_ERR_UNSUPPORTED;
    }
    // buffers, residual rows, gamma and pads: no two overlap
    const int64_t bb = T * H * s;
    std::vector<std::pair<const void *, int64_t>> spans;
    for (int q = 0; q < N; ++q) {
        spans.push_back({g->buffers[q], bb});
        if (has_res[q]) {
            int64_t r0, r1;
            tp::rows_of(T, N, q, r0, r1);
            spans.push_back({residuals[q], (r1 - r0) * H * s});
        }
        if (nsig) spans.push_back({g->signals[q], RARN_TP_SIGNAL_BYTES});
    }
    spans.push_back({gamma, H * s});
    for (size_t i = 0; i < spans.size(); ++i)
        for (size_t j = i + 1; j < spans.size(); ++j)
            if (overlaps(spans[i].first, spans[i].second, spans[j].first, spans[j].second))
                return RARN_ERR_ALIAS;
    return RARN_OK;
}

// Bit q: rank q's buffer, bit 8 + q: rank q's residual, for the streams that
// are memory of the current device (the prefetch is only issued for those).
static uint32_t tp_local_mask(const tp::Params &p, int N) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0u;
    }
    auto local = [dev](const void *ptr) {
        if (!ptr) return false;
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
            cudaGetLastError();  // not a sticky error: clear it
            return false;
        }
        return a.type == cudaMemoryTypeDevice && a.device == dev;
    };
    uint32_t m = 0;
    for (int q = 0; q < N; ++q) {
        if (local(p.bufs[q])) m |= 1u << q;
        if (local(p.residual[q])) m |= 1u << (8 + q);
    }
    return m;
}

static rarn_status tp_run(const rarn_tp_group *g, void *const *residuals, const void *gamma,
                          int64_t T, int64_t H, float eps, rarn_dtype dt, void *stream,
                          bool world) {
    rarn_status st = tp_check(g, residuals, gamma, T, H, eps, dt, world);
    if (st != RARN_OK || T == 0) return st;
    DeviceInfo *d = nullptr;
    if ((st = device_info(&d)) != RARN_OK) return st;
    const int N = g->world_size;
    if (!world && g->signals[0]) {
        // ranks that meet in the barrier run on different GPUs: two ranks'
        // launches on one GPU that wait on each other may never run at the
        // same time (the world launch is the one-GPU form)
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e);
        for (int q = 0; q < N; ++q) {
            if (q == g->rank) continue;
            cudaPointerAttributes a{};
            if (cudaPointerGetAttributes(&a, g->buffers[q]) != cudaSuccess) {
                cudaGetLastError();  // not a sticky error: clear it
                return RARN_ERR_INVALID_ARG;
            }
            if (a.type == cudaMemoryTypeDevice && a.device == dev) return RARN_ERR_UNSUPPORTED;
        }
    }
    int per_sm = 0;
    cudaError_t e = dt == RARN_BF16 ? tp_blocks_per_sm<__nv_bfloat16>(H, &per_sm)
                    : dt == RARN_F16 ? tp_blocks_per_sm<__half>(H, &per_sm)
                                     : tp_blocks_per_sm<float>(H, &per_sm);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm < 1) return RARN_ERR_UNSUPPORTED;
    const int ctas = tp::ctas_per_rank(T, N, d->num_sms, per_sm, world);
    tp::Params p{};
    const bool sync = g->signals[0] != nullptr;
    for (int q = 0; q < N; ++q) {
        p.bufs[q] = g->buffers[q];
        p.signals[q] = sync ? g->signals[q] : nullptr;
        p.residual[q] = (world || q == g->rank) ? residuals[q] : nullptr;
    }
    p.gamma = gamma;
    p.T = T;
    p.H = H;
    p.N = N;
    p.rank = world ? -1 : g->rank;
    p.ctas = ctas;
    p.eps = eps;
    p.watchdog = d->watchdog;
    p.wait_limit_ns = tp::kWaitLimitNs;
    p.stall_rank = -1;
    p.prefetch_mask =
        tp_prefetch(per_sm, N, H * elem_size(dt)) ? tp_local_mask(p, N) : 0u;
    if (sync) {
        const long long f = g_stall_fill.exchange(-1);
        if (f >= 0) {
            p.stall_rank = (int)(f % N);
            p.wait_limit_ns = g_stall_limit_ns.load();
        }
    }
    const int grid = world ? ctas * N : ctas;
    const bool coop = world && sync;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool pdl = g_pdl.load() != 0;
    e = dt == RARN_BF16 ? launch_tp<__nv_bfloat16>(p, grid, coop, pdl, cs)
        : dt == RARN_F16 ? launch_tp<__half>(p, grid, coop, pdl, cs)
                         : launch_tp<float>(p, grid, coop, pdl, cs);
    if (e != cudaSuccess) return cuda_fail(e);
    return RARN_OK;
}

rarn_status rarn_tp_reduce_add_rms_norm(const rarn_tp_group *group, void *residual,
                                        const void *gamma, int64_t T, int64_t H, float eps,
                                        rarn_dtype dt, void *stream) {
    void *res[RARN_TP_MAX_RANKS] = {};
    if (group && group->rank >= 0 && group->rank < RARN_TP_MAX_RANKS) res[group->rank] = residual;
    return tp_run(group, res, gamma, T, H, eps, dt, stream, false);
}

rarn_status rarn_tp_reduce_add_rms_norm_world(const rarn_tp_group *group, void *const *residuals,
                                              const void *gamma, int64_t T, int64_t H, float eps,
                                              rarn_dtype dt, void *stream) {
    if (!residuals) return RARN_ERR_INVALID_ARG;
    return tp_run(group, residuals, gamma, T, H, eps, dt, stream, true);
}

// IPC handles: a magic word, the CUDA handle of the allocation holding the
// pointer, and the pointer's offset in it.
namespace {
constexpr uint64_t kIpcMagic = 0x52524e4950433031ull;  // "RRNIPC01"
struct IpcHandle {
    uint64_t magic;
    cudaIpcMemHandle_t mem;
    uint64_t offset;
};
static_assert(sizeof(IpcHandle) <= RARN_IPC_HANDLE_BYTES, "handle size");
std::mutex g_ipc_mu;
std::unordered_map<uintptr_t, void *> g_ipc_open;  // returned pointer -> mapping base

using AddressRangeFn = CUresult (*)(CUdeviceptr *, size_t *, CUdeviceptr);
}  // namespace

rarn_status rarn_ipc_export(const void *ptr, void *handle) {
    if (!ptr || !handle) return RARN_ERR_INVALID_ARG;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!fn || q != cudaDriverEntryPointSuccess) return cuda_fail(cudaErrorNotSupported);
    CUdeviceptr base = 0;
    size_t size = 0;
    if (reinterpret_cast<AddressRangeFn>(fn)(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) !=
        CUDA_SUCCESS)
        return RARN_ERR_INVALID_ARG;  // not device memory of this context
    IpcHandle h{};
    h.magic = kIpcMagic;
    h.offset = reinterpret_cast<uintptr_t>(ptr) - (uintptr_t)base;
    if ((e = cudaIpcGetMemHandle(&h.mem, reinterpret_cast<void *>(base))) != cudaSuccess)
        return cuda_fail(e);
    memset(handle, 0, RARN_IPC_HANDLE_BYTES);
    memcpy(handle, &h, sizeof(h));
    return RARN_OK;
}

rarn_status rarn_ipc_import(const void *handle, void **ptr) {
    if (!handle || !ptr) return RARN_ERR_INVALID_ARG;
    IpcHandle h;
    memcpy(&h, handle, sizeof(h));
    if (h.magic != kIpcMagic) return RARN_ERR_INVALID_ARG;
    void *base = nullptr;
    const cudaError_t e = cudaIpcOpenMemHandle(&base, h.mem, cudaIpcMemLazyEnablePeerAccess);
    if (e != cudaSuccess) return cuda_fail(e);
    *ptr = static_cast<char *>(base) + h.offset;
    std::lock_guard<std::mutex> lock(g_ipc_mu);
    g_ipc_open[reinterpret_cast<uintptr_t>(*ptr)] = base;
    return RARN_OK;
}

rarn_status rarn_ipc_close(void *ptr) {
    if (!ptr) return RARN_ERR_INVALID_ARG;
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_ipc_mu);
        auto it = g_ipc_open.find(reinterpret_cast<uintptr_t>(ptr));
        if (it == g_ipc_open.end()) return RARN_ERR_INVALID_ARG;
        base = it->second;
        g_ipc_open.erase(it);
    }
    const cudaError_t e = cudaIpcCloseMemHandle(base);
    return e == cudaSuccess ? RARN_OK : cuda_fail(e);
}

rarn_status rarn_launch_floor(const void *rows, int64_t row_bytes, int32_t grid, int32_t block,
                              void *stream) {
    if (grid < 1 || block < 1 || block > 1024) return RARN_ERR_INVALID_ARG;
    if (rows && (row_bytes < 16 || row_bytes % 16 || row_bytes > (1 << 20) || !aligned16(rows)))
        return RARN_ERR_INVALID_ARG;
    const cudaError_t e =
        launch_kernel(k_launch_floor, dim3((unsigned)grid), dim3((unsigned)block), 0,
                      static_cast<cudaStream_t>(stream), g_pdl.load() != 0, 1,
                      static_cast<const char *>(rows), static_cast<uint32_t>(rows ? row_bytes : 0));
    if (e != cudaSuccess) return cuda_fail(e);
    return RARN_OK;
}

int rarn_version(void) { return (1 << 16) | 2; }

}  // extern "C"
