/*
 * rarn.h -- C ABI of the GB300 (sm_103a) row-wise RMSNorm library.
 *
 * Three operations on row-major [T, H] problems, one row per token:
 *
 *   rarn_rms_norm             y = x * rsqrt(mean(x^2) + eps) * gamma
 *   rarn_fused_add_rms_norm   h = x + residual; residual <- h; y = rmsnorm(h)
 *   rarn_reduce_add_rms_norm  h = p_0 + ... + p_{R-1} + residual;
 *                             residual <- h; y = rmsnorm(h)
 *
 * Definitions followed (page title, section):
 *   "RMSNorm kernel", 1 Background and 2 Analytics & Implementation
 *   (Abstraction): y_i = x_i * gamma_i / RMS(x), RMS taken over the last
 *   (hidden) dimension only; the shape [..., hidden] is flattened to
 *   [rows, hidden].
 *   "Tokenweave fused-RMSNorm-AR kernel", Code walkthrough: the first pass
 *   reduces the partial-sum buffers, adds the residual, writes the sum back as
 *   the residual and accumulates the squares of that stored value in fp32; the
 *   reciprocal RMS is rsqrt(variance / hidden_size + eps); the second pass
 *   scales by it and by the weight.
 *
 * Arithmetic contract:
 *   - h is summed in binary32 in the fixed order p_0, p_1, ..., p_{R-1}, then
 *     the residual, and rounded once (nearest-even) to the storage type.  The
 *     updated residual is that rounded h, bit for bit.
 *   - The sum of squares of the rounded h is accumulated in binary32; the
 *     reciprocal RMS is rsqrtf(ss / H + eps).
 *   - y_i = (h_i * inv) * gamma_i in binary32, rounded once to the storage
 *     type.  fp32 storage: within 1e-5 relative of the exact value; fp16 and
 *     bf16: within 2 units in the last place.
 *   - Results are deterministic: the same inputs give the same bits on every
 *     call.
 *   - Limitation: the sum of squares is binary32, so a row whose sum of
 *     squares exceeds FLT_MAX (|h| around 1e19 and above for H = 4096)
 *     normalises to zero.
 *
 * Common conventions for every compute entry point:
 *   - Pointers are DEVICE pointers owned by the caller (y, x, partials,
 *     residual, gamma); the *_host forms below take pinned host pointers
 *     instead.  The library allocates no memory and keeps no pointer after
 *     the call returns.
 *   - Layout: dense row-major.  x, residual and y are [T, H] with row stride H
 *     elements; partials is [R, T, H], partial r starting at element r*T*H;
 *     gamma is [H].  All share one storage type `dt`.  eps is binary32.
 *   - Alignment: any element-aligned pointer is accepted.  When every pointer
 *     is 16-byte aligned and H * sizeof(dt) is a multiple of 16 the 128-bit
 *     vector kernels run; otherwise a scalar kernel does.
 *   - Aliasing: y may equal x (rms_norm, fused) or partials (reduce: y then
 *     overwrites partial 0).  Any other overlap between an output (y,
 *     residual) and any other buffer returns RARN_ERR_ALIAS.
 *   - Streams: the work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) on the current device and the call returns
 *     without synchronising.  Results are ready when the stream reaches that
 *     point.
 *   - Errors: argument errors are returned synchronously, before any work is
 *     enqueued (nothing is written).  T == 0 is a no-op returning RARN_OK.  A
 *     failed launch returns RARN_ERR_CUDA; rarn_last_cuda_error() then gives
 *     the CUDA error code.  No C++ exception crosses this interface.
 */
#ifndef RARN_H
#define RARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rarn_dtype {
    RARN_F32 = 0,  /* IEEE binary32 */
    RARN_F16 = 1,  /* IEEE binary16 */
    RARN_BF16 = 2  /* bfloat16 */
} rarn_dtype;

typedef enum rarn_status {
    RARN_OK = 0,
    RARN_ERR_INVALID_ARG = 1, /* null pointer with T > 0, T < 0, H <= 0, R < 1,
                                 eps negative or NaN, unknown dtype or op */
    RARN_ERR_UNSUPPORTED = 2, /* sizes beyond the limits below, or a forced
                                 kernel path that cannot run this shape */
    RARN_ERR_ALIAS = 3,       /* outputs overlap inputs other than as allowed */
    RARN_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
} rarn_status;

/* Size limits: 1 <= H <= RARN_MAX_H, 0 <= T <= RARN_MAX_T, 1 <= R <= RARN_MAX_R. */
#define RARN_MAX_H (1 << 24)
#define RARN_MAX_T ((int64_t)1 << 40)
#define RARN_MAX_R 64

/* Operation codes used by the planning query. */
typedef enum rarn_op {
    RARN_OP_RMS_NORM = 0,
    RARN_OP_FUSED_ADD_RMS_NORM = 1,
    RARN_OP_REDUCE_ADD_RMS_NORM = 2
} rarn_op;

/* Kernel families.  RARN_PATH_AUTO picks per shape; the others force one
 * family (for tests and measurements) and return RARN_ERR_UNSUPPORTED from a
 * compute call whose shape that family cannot run. */
typedef enum rarn_path {
    RARN_PATH_AUTO = 0,
    RARN_PATH_ROWS = 1,    /* a warp or a CTA per row, row held in registers;
                              a two-pass CTA kernel when the row is too long */
    RARN_PATH_STREAM = 2,  /* persistent CTAs, one per SM, fed by TMA bulk
                              copies into a shared-memory pipeline */
    RARN_PATH_CLUSTER = 3  /* a thread-block cluster per row, sum of squares
                              combined through distributed shared memory */
} rarn_path;

/*
 * y[T,H] = RMSNorm(x[T,H]) * gamma[H].
 * ("RMSNorm kernel", 1 Background; 2 Abstraction.)
 * In: x, gamma.  Out: y (may equal x).
 */
rarn_status rarn_rms_norm(void *y, const void *x, const void *gamma, int64_t T, int64_t H,
                          float eps, rarn_dtype dt, void *stream);

/*
 * h = x + residual (binary32 add, one rounding); residual <- h;
 * y = RMSNorm(h) * gamma.
 * ("Tokenweave fused-RMSNorm-AR kernel", Code walkthrough, with one input
 * buffer in place of the cross-GPU reduction.)
 * In: x, gamma.  In/out: residual.  Out: y (may equal x, not residual).
 */
rarn_status rarn_fused_add_rms_norm(void *y, const void *x, void *residual, const void *gamma,
                                    int64_t T, int64_t H, float eps, rarn_dtype dt,
                                    void *stream);

/*
 * h = ((p_0 + p_1) + ... + p_{R-1}) + residual, each add in binary32, one
 * rounding; residual <- h; y = RMSNorm(h) * gamma.
 * ("Tokenweave fused-RMSNorm-AR kernel", Code walkthrough: the reduce of the
 * partial buffers, here R buffers in this GPU's memory, summed in a fixed
 * order.)
 * In: partials [R,T,H], gamma.  In/out: residual.  Out: y (may equal
 * partials, i.e. overwrite partial 0).
 */
rarn_status rarn_reduce_add_rms_norm(void *y, const void *partials, int32_t R, void *residual,
                                     const void *gamma, int64_t T, int64_t H, float eps,
                                     rarn_dtype dt, void *stream);

/*
 * Host-buffer forms of the three operations: the same arguments, layout,
 * aliasing and stream rules, but every buffer (y, x / partials, residual,
 * gamma) is PINNED HOST memory that the current device can address:
 * allocated with cudaHostAlloc / cudaMallocHost, or registered with
 * cudaHostRegister and mapped.  The kernels read the inputs and write the
 * outputs through that mapping, so the host<->device transfer happens inside
 * the one kernel launch (over NVLink-C2C on Grace systems) and no device
 * memory is needed.  The first and last byte of every buffer are checked
 * with cudaPointerGetAttributes before anything is enqueued: pinned host
 * memory is accepted; pageable host memory only where the device reads it
 * through the host's page tables (rarn_host_access() == 2, e.g. Grace);
 * device or managed memory, or pageable memory elsewhere, returns
 * RARN_ERR_INVALID_ARG.  As with the device forms, the caller guarantees
 * that each buffer really spans its full size.  Results are in
 * host memory once the stream reaches the call.  These forms have no
 * counterpart on the pages: they are how a caller with data in host memory
 * runs the path without staging copies.
 */
rarn_status rarn_rms_norm_host(void *y, const void *x, const void *gamma, int64_t T, int64_t H,
                               float eps, rarn_dtype dt, void *stream);
rarn_status rarn_fused_add_rms_norm_host(void *y, const void *x, void *residual,
                                         const void *gamma, int64_t T, int64_t H, float eps,
                                         rarn_dtype dt, void *stream);
rarn_status rarn_reduce_add_rms_norm_host(void *y, const void *partials, int32_t R,
                                          void *residual, const void *gamma, int64_t T,
                                          int64_t H, float eps, rarn_dtype dt, void *stream);

/*
 * General forms: per-buffer row strides and an fp32 residual stream.
 *
 * A rarn_rows names a [T, H] matrix inside a larger allocation: row t starts
 * at element t * row_stride of `data` (row_stride >= H, in elements of
 * `dtype`); only the first H elements of each row are read or written.
 * Partials are R such matrices `partial_stride` elements apart (from the
 * start of one to the start of the next).  gamma is [H] of the inputs' type.
 *
 * Storage types: y, x / partials and gamma share one type; the residual has
 * either that type or RARN_F32 with 16-bit inputs (the sum of the partials and
 * the residual is then kept in binary32 with no rounding, and y is rounded
 * once to the 16-bit type).  Other combinations return RARN_ERR_UNSUPPORTED.
 *
 * Aliasing is judged on the row spans ((T - 1) * row_stride + H elements):
 * y may equal x / partial 0 exactly (same data and row stride); any other
 * overlap of an output with another buffer returns RARN_ERR_ALIAS, even where
 * the rows themselves would interleave without touching.  The 16-byte kernels
 * run when every base pointer is 16-byte aligned and every row stride and the
 * partial stride are multiples of 16 bytes.  Everything else is as for the
 * dense forms above; those are these forms with every row stride H and the
 * partials T * H apart.  ("RMSNorm kernel", 1 Background: the norm runs over
 * the last dimension of [..., hidden]; a row stride lets that last dimension
 * be a slice of a wider one.)
 */
typedef struct rarn_rows {
    void *data;
    int64_t row_stride;
    rarn_dtype dtype;
} rarn_rows;

rarn_status rarn_rms_norm_ex(rarn_rows y, rarn_rows x, const void *gamma, int64_t T, int64_t H,
                             float eps, void *stream);
rarn_status rarn_fused_add_rms_norm_ex(rarn_rows y, rarn_rows x, rarn_rows residual,
                                       const void *gamma, int64_t T, int64_t H, float eps,
                                       void *stream);
rarn_status rarn_reduce_add_rms_norm_ex(rarn_rows y, rarn_rows partials, int64_t partial_stride,
                                        int32_t R, rarn_rows residual, const void *gamma,
                                        int64_t T, int64_t H, float eps, void *stream);

/*
 * 8-bit output forms: the general forms above with y replaced by a matrix of
 * one-byte codes in e4m3 or e5m2 and a scale ("Block All Reduce", FP8
 * section: both formats, converted with saturation to the largest finite
 * value).  For each row, with h, inv and v_i = (h_i * inv) * gamma_i computed
 * as for the 16-bit output (binary32), the code is u_i = v_i / s rounded to
 * nearest even and saturated to +-maxf (448 for e4m3, 57344 for e5m2):
 *   RARN_SCALE_TENSOR: s = scale[0], a binary32 value the kernel reads
 *                      (in device memory, so an earlier kernel may write it);
 *                      u_i = v_i * (1 / s);
 *   RARN_SCALE_ROW:    s = max_i |v_i| / maxf, written to scale[t] (T binary32
 *                      values); u_i = (v_i * (1 / max|v|)) * maxf, so the
 *                      row's largest magnitude maps to maxf; a row of zeros
 *                      gets s = 1 and zero codes.  max|v| is computed as
 *                      inv * max_i |h_i * gamma_i| (inv > 0), which equals it
 *                      up to binary32 rounding and joins the row reduction.
 * Dequantised, code value * s approximates v.  Row t of the codes starts at
 * byte t * row_stride of `data` (row_stride >= H); only the first H bytes of
 * each row are written.  The residual (fused / reduce) has the inputs'
 * storage type and is updated as in the other forms.
 *
 * Errors: a NULL descriptor or scale, an unknown format or mode:
 * RARN_ERR_INVALID_ARG; a residual of another type than the inputs, or the
 * stream / cluster path forced (the 8-bit output is built for the register
 * row kernels only): RARN_ERR_UNSUPPORTED; the codes or a written scale
 * overlapping any other buffer, or a read scale overlapping an output:
 * RARN_ERR_ALIAS.  Everything else as for the general forms.  The packed
 * kernels need, besides the inputs' 16-byte conditions, codes aligned to and
 * a row stride a multiple of 16 / sizeof(input element) bytes.
 */
typedef enum rarn_fp8_format { RARN_E4M3 = 0, RARN_E5M2 = 1 } rarn_fp8_format;
typedef enum rarn_scale_mode { RARN_SCALE_TENSOR = 0, RARN_SCALE_ROW = 1 } rarn_scale_mode;

typedef struct rarn_fp8_rows {
    void *data;                 /* codes: T rows of H bytes, device memory */
    int64_t row_stride;         /* bytes between rows, >= H */
    rarn_fp8_format format;
    rarn_scale_mode scale_mode;
    float *scale;               /* device memory: 1 value (read) or T values (written) */
} rarn_fp8_rows;

rarn_status rarn_rms_norm_fp8(const rarn_fp8_rows *y, rarn_rows x, const void *gamma, int64_t T,
                              int64_t H, float eps, void *stream);
rarn_status rarn_fused_add_rms_norm_fp8(const rarn_fp8_rows *y, rarn_rows x, rarn_rows residual,
                                        const void *gamma, int64_t T, int64_t H, float eps,
                                        void *stream);
rarn_status rarn_reduce_add_rms_norm_fp8(const rarn_fp8_rows *y, rarn_rows partials,
                                         int64_t partial_stride, int32_t R, rarn_rows residual,
                                         const void *gamma, int64_t T, int64_t H, float eps,
                                         void *stream);

/*
 * Reduce + residual add + RMSNorm over R partials stored as 8-bit codes, with
 * one binary32 scale per partial buffer ("Block All Reduce", FP8 section:
 * reductions over e4m3 / e5m2 inputs with a binary32 accumulator;
 * "Tokenweave fused-RMSNorm-AR kernel", Code walkthrough, for the reduce,
 * residual and norm steps):
 *
 *   v_r = fl32(dec(c_r) * scales[r])      each partial dequantised, one rounding
 *   acc = v_0; acc = fl32(acc + v_r) for r = 1 .. R-1; acc = fl32(acc + residual)
 *   h = RN(acc); residual <- h; y = RN((h * rsqrt(mean(h^2) + eps)) * gamma)
 *
 * partials: R x T x H bytes of codes in `format`, dense (partial r starts at
 * byte r * T * H), 8-byte aligned; scales: R binary32 values in device memory;
 * residual (updated in place), gamma [H] and y [T, H] in `dt`, dense, 16-byte
 * aligned.  All device memory owned by the caller; asynchronous on `stream`.
 * With H a multiple of 16, 16-byte aligned codes, at least 8 rows per SM and
 * either R >= 4 with H >= 4096, R >= 8, or R = 3 with H >= 8192, a persistent
 * kernel streams the codes and the residual through shared memory with bulk
 * copies; otherwise a CTA per row holds it in registers.  Both give the same residual bits (y may differ in the last
 * place: the row's sum of squares is reduced in another order).  The
 * persistent kernel's waits are bounded; one that runs out sets the
 * watchdog word (rarn_watchdog) and that CTA's outputs are invalid.
 *
 * Errors: NULL pointers with T > 0, T < 0, H <= 0, R < 1, a NaN / negative /
 * infinite eps, an unknown type or format: RARN_ERR_INVALID_ARG; R > 16, H not
 * a multiple of 8, H > 16384 (binary32: 8192) or misaligned pointers:
 * RARN_ERR_UNSUPPORTED; y or the residual overlapping each other or an input:
 * RARN_ERR_ALIAS.  T = 0 returns RARN_OK.
 */
rarn_status rarn_reduce_add_rms_norm_fp8in(void *y, const void *partials, int32_t R,
                                           rarn_fp8_format format, const float *scales,
                                           void *residual, const void *gamma, int64_t T,
                                           int64_t H, float eps, rarn_dtype dt, void *stream);

/*
 * GEMM producer with the fused residual-add RMSNorm as its epilogue: the
 * partial that the fused form adds to the residual is the product of the
 * activations A [T, K] and a linear layer's weight W [H, K]:
 *   P = A W^T                      (binary32 accumulation on the tensor cores)
 *   h = RN(P + residual)           residual <- h (the accumulator plus the
 *                                  residual, rounded once; P is never written)
 *   y = RN((h * inv) * gamma),     inv = rsqrt(mean(h^2) + eps)
 * ("sm80 GEMM + ReduceScatter": the flux epilogue consumes the accumulator
 * tile before anything is written; "Tokenweave fused-RMSNorm-AR kernel",
 * Code walkthrough: the norm steps.)
 *
 * Kernels on `stream`: the tcgen05 GEMM whose epilogue writes h and, per row
 * and column block (128 columns in the persistent kernels, one tile of 256
 * or 512 otherwise), the partial sum of squares of h into `workspace`.  With
 * K >= 3072, or K >= 2048 and T >= 4096 (in the persistent kernels, K >=
 * 512; RARN_TUNE_GEMM_NORM_IN_EPILOGUE overrides) the same epilogue then waits for the
 * other column tiles of its 128-row block (a counter per block in the
 * workspace, zeroed by a one-CTA kernel launched just before), sums each
 * row's partials in column order and writes y; otherwise a norm kernel does
 * that last step.  Both orders give identical bits.  With K >= 1024 and so
 * few 128 x 256 tiles (ceil(T / 128) row blocks of H / 256) that they leave
 * at least half of the SMs idle, the product is split over K instead: S =
 * min(9, floor(min(SMs, 152) / tiles), floor(ceil(K / 64) / 8)) CTAs per tile
 * write binary32 partial products into the workspace and a CTA per row adds
 * them in split order, adds the residual (one rounding) and normalises (a
 * different binary32 summation order, within the same accuracy bound); this
 * needs the full rarn_gemm_workspace_bytes(T, H) and a 32-byte aligned
 * workspace, else the call runs without split K.  `workspace` is
 * caller-owned device memory of at least the bytes the non-split kernels use
 * (rarn_gemm_workspace_bytes where split K cannot apply; 16-byte aligned);
 * its contents are scratch and need no initialisation.
 *
 * Matrices are rarn_rows (row-major, row_stride in elements), all of one
 * 16-bit type (RARN_BF16 or RARN_F16; RARN_F32 returns UNSUPPORTED); gamma is
 * [H] of that type.  Bases 16-byte aligned and row strides multiples of 8
 * elements, else RARN_ERR_UNSUPPORTED.  H must be a multiple of 512 up to
 * 16384, or of 256 up to 8192 (else UNSUPPORTED); T and K are free (partial
 * tiles read zeros).  A
 * missing or short workspace returns RARN_ERR_INVALID_ARG; outputs (y, the
 * residual, the workspace) overlapping anything else return RARN_ERR_ALIAS.
 * Accuracy: P is a binary32 accumulation, so h may differ from the exact
 * rounding of P + residual by one unit in the last place where that exact
 * value lies within the accumulation error of a rounding boundary.
 */
rarn_status rarn_gemm_add_rms_norm(rarn_rows y, rarn_rows a, rarn_rows w, rarn_rows residual,
                                   const void *gamma, int64_t T, int64_t H, int64_t K, float eps,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * rarn_gemm_add_rms_norm for callers that cannot allocate device memory: it
 * takes no workspace argument and calls no cudaMalloc, cudaFree or other
 * allocating routine.  Such callers include plug-ins inside a host program
 * that owns every byte of device memory and hands out no allocator, runtimes
 * that plan all memory before they start serving and forbid allocation
 * afterwards, and latency-critical code that cannot afford the implicit
 * device synchronisation of cudaMalloc / cudaFree.  None of the source
 * pages ("RMSNorm kernel", "Tokenweave fused-RMSNorm-AR kernel", "sm80 GEMM
 * + ReduceScatter") has a counterpart.
 *
 * Scratch: the per-row partial sums of squares and the row-block counters
 * live in a file-scope device array of 2^20 binary32 values (4 MiB, 256-byte
 * aligned) that the library reserves on every GPU it is loaded on and keeps
 * until the process exits.  One launch sequence holds T (H / 128 + 1) of
 * those values, so a call with more rows than the array holds
 * (rarn_gemm_noalloc_rows(H): 16128 rows at H = 8192, 8064 at H = 16384)
 * runs as several launch sequences on `stream`, one after another.  Every
 * partial sum is written before it is read and the counters are zeroed by
 * the call itself, so nothing needs clearing between calls.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and keeps it; make
 * that first call before any stream capture begins.  A failed look-up
 * returns RARN_ERR_CUDA.
 *
 * Ordering: every call on a device shares the one array, which keeps the
 * last call's contents.  Calls that overlap on the GPU (different streams
 * with no ordering between them) race on it and give wrong results; issue
 * them on one stream or synchronise the streams.
 *
 * Arguments and errors as for rarn_gemm_add_rms_norm, checked once over all
 * T rows before anything is enqueued: overlaps between rows that different
 * launch sequences would cover return RARN_ERR_ALIAS like any other, and an
 * argument error leaves every buffer untouched.  (A launch failure, reported
 * as RARN_ERR_CUDA, can still come after earlier sequences were enqueued.)
 * Results are bit-identical to the workspace form's, with one exception:
 * where the workspace form splits K over S <= 9 CTAs per tile (S = the
 * split count rarn_plan_gemm reports), this entry point does
 * the same only where the split's partial products fit in the array next to
 * the partial sums, i.e. where
 *   64 * ceil((4 * ceil(T * H / 512) + ceil(T / 128)) / 64) + S * T * H <= 2^20
 * binary32 values (T = 8, H = 4096, S = 8 fits; T = 128, H = 4096 does not).
 * Otherwise it runs without split K: a different binary32 summation order,
 * within the same accuracy bound.
 */
rarn_status rarn_gemm_add_rms_norm_noalloc(rarn_rows y, rarn_rows a, rarn_rows w,
                                           rarn_rows residual, const void *gamma, int64_t T,
                                           int64_t H, int64_t K, float eps, void *stream);

/* Workspace bytes rarn_gemm_add_rms_norm needs for T rows of H: one binary32
 * per row and 128 columns, rounded up to 16 bytes, then one 32-bit counter
 * per 128-row block; where split K can apply (H <= 8192 and ceil(T / 128) *
 * H / 256 tiles leave at least half of 152 SMs idle) also, from the next
 * 256-byte boundary, S T H binary32 values for split K, S = min(9,
 * floor(152 / tiles)).  -1 if H is not supported. */
int64_t rarn_gemm_workspace_bytes(int64_t T, int64_t H);

/* Describe the kernel rarn_reduce_add_rms_norm_fp8in takes for a problem
 * (pure host logic, no GPU needed): T rows of H, R partials, storage type dt,
 * whether the codes are 16-byte aligned, and the device's SM count and opt-in
 * shared memory per CTA in bytes.  Writes a NUL-terminated description
 * ("q8in.ring ..." with the shared-memory ring's shape, or "q8in.rows ...")
 * into out[cap].  Errors: NULL out, cap 0, bad arguments:
 * RARN_ERR_INVALID_ARG; a shape the call rejects as unsupported:
 * RARN_ERR_UNSUPPORTED (out says so). */
rarn_status rarn_plan_fp8in(int64_t T, int64_t H, int32_t R, rarn_dtype dt, int codes_aligned16,
                            int32_t num_sms, int32_t max_smem, char *out, size_t cap);

/*
 * Tensor-parallel form: reduce-scatter, residual add + RMSNorm, all-gather
 * over N ranks (one GPU each), as the tokenweave fused-RMSNorm-AR kernel does
 * ("Tokenweave fused-RMSNorm-AR kernel", Code walkthrough).  Every rank q
 * holds a buffer of T x H elements (dense, row-major, type dt) that every
 * rank can address (a peer mapping, e.g. through rarn_ipc_import): on entry
 * it holds rank q's partial (the output of its row-parallel layer); on exit
 * it holds y for all T rows.  Rank r owns rows floor(r T / N) .. floor((r + 1)
 * T / N) - 1 (rarn_tp_rows) and keeps the residual of those rows only.  For
 * each of its rows rank r computes
 *   h = RN(((p_0 + p_1) + ... + p_{N-1}) + residual)   (binary32 adds in rank
 *       order, one rounding; residual <- h)
 *   y = RN((h * rsqrt(mean(h^2) + eps)) * gamma)
 * and writes y into row t of every rank's buffer, so that the reduce form over
 * the N ranks' partials (R = N) is what every rank ends up with, bit for bit.
 * The reads and writes of other ranks' buffers are plain 16-byte loads and
 * stores (no multimem, no TMA copies); buffers in memory of the current
 * device may also be prefetched into L2 (rarn_plan_tp).
 *
 * Ordering between ranks.  With signal pads (signals[q] non-NULL for every q:
 * RARN_TP_SIGNAL_BYTES of device memory per rank, zeroed once before first
 * use, addressable by every rank like the buffers), CTA b of every rank meets
 * CTA b of every other rank at entry -- so every rank's partial is complete
 * before any rank reads it -- and at exit -- so all rows of y are in this
 * rank's buffer before anything after the call on `stream` runs.  Every wait
 * is bounded (10 s); one that runs out sets watchdog bit 3 (rarn_watchdog),
 * that CTA's rows are not computed, and the pads must be zeroed again on
 * every rank before the next call.  With signals[0] == NULL there is no
 * device wait at all: the caller must order the call after every rank's
 * partial is complete and order any use of the buffer after every rank's
 * call has completed (e.g. host barriers around the call).  Every rank must
 * make the call with the same T, H, dt and signal setting on the same GPU
 * model (CTA b pairs with CTA b).  With signal pads the ranks must run on
 * different GPUs: a per-rank call whose other ranks' buffers are memory of
 * the current device returns RARN_ERR_UNSUPPORTED (on one GPU, use the world
 * launch, whose ranks share one cooperative grid).
 *
 * Errors: a NULL group, world_size outside 1 .. RARN_TP_MAX_RANKS, rank
 * outside 0 .. N-1, a NULL buffer or gamma with T > 0, a NULL residual for a
 * rank that owns rows (a rank without rows, T < N, may pass NULL), signal pads
 * given for some ranks only, T < 0, H <= 0, a NaN / negative / infinite eps,
 * an unknown dt: RARN_ERR_INVALID_ARG; H * sizeof(dt) not a multiple of 16,
 * more than 2048 16-byte packs per row, pointers not 16-byte aligned (pads: 4
 * bytes): RARN_ERR_UNSUPPORTED; buffers overlapping each other, the residual
 * or gamma: RARN_ERR_ALIAS.  T = 0 returns RARN_OK.  Asynchronous on `stream`.
 */
#define RARN_TP_MAX_RANKS 8
#define RARN_TP_SIGNAL_BYTES (1024 * RARN_TP_MAX_RANKS * 4)

typedef struct rarn_tp_group {
    int32_t world_size;                       /* N */
    int32_t rank;                             /* this rank, 0 .. N-1 */
    void *buffers[RARN_TP_MAX_RANKS];         /* rank q's [T, H] buffer, as this process
                                                 addresses it */
    uint32_t *signals[RARN_TP_MAX_RANKS];     /* rank q's signal pad, or all NULL */
} rarn_tp_group;

/* Rows [*r0, *r1) that rank r of N owns: floor(r T / N), floor((r + 1) T / N).
 * RARN_ERR_INVALID_ARG for T < 0, N < 1, r outside 0 .. N-1 or NULL outputs. */
rarn_status rarn_tp_rows(int64_t T, int32_t world_size, int32_t rank, int64_t *r0, int64_t *r1);

/* The launch a tensor-parallel call of T rows of H elements over N ranks
 * makes (world != 0: every rank's part in one launch, as
 * rarn_tp_reduce_add_rms_norm_world; 0: one rank's, as
 * rarn_tp_reduce_add_rms_norm) on a device with num_sms SMs (<= 0: the
 * current device's) that holds blocks_per_sm CTAs of the kernel per SM (<= 0:
 * the current device's occupancy for H and dt).  Writes a NUL-terminated
 * description into out[cap]: "tp.world ranks=N ctas=C block=B vpt=V
 * blocks_per_sm=P prefetch=F" ("tp.rank ..." for one rank), C CTAs per rank
 * of B threads, V 16-byte packs per thread, F = 1 when each CTA prefetches
 * its next row's streams into L2 while it works on the current one: where
 * the loads an SM holds in flight, P (N + 1) rows of H elements, come to at
 * most 64 KB, or 80 KB with one CTA per SM (RARN_TUNE_TP_PREFETCH
 * overrides).  The prefetch is only issued for streams in memory of the
 * launching device.  Pure host logic when num_sms and blocks_per_sm are
 * given.  Errors: NULL out, cap 0, T <= 0, H <= 0, N outside 1 ..
 * RARN_TP_MAX_RANKS, an unknown dt: RARN_ERR_INVALID_ARG; rows that the call
 * rejects as unsupported: RARN_ERR_UNSUPPORTED (out says so); a failed
 * device query: RARN_ERR_CUDA. */
rarn_status rarn_plan_tp(int64_t T, int64_t H, int32_t world_size, rarn_dtype dt, int world,
                         int32_t num_sms, int32_t blocks_per_sm, char *out, size_t cap);

/* This rank's part: `residual` holds this rank's rows of the residual
 * ([r1 - r0, H], dense, updated in place); gamma [H]. */
rarn_status rarn_tp_reduce_add_rms_norm(const rarn_tp_group *group, void *residual,
                                        const void *gamma, int64_t T, int64_t H, float eps,
                                        rarn_dtype dt, void *stream);

/* Every rank's part in one launch on the current device: every buffer (and
 * pad) is memory this device addresses, residuals[q] holds rank q's rows of
 * the residual, group->rank is ignored.  With signal pads the launch is
 * cooperative (every CTA resident at once, so the ranks' CTAs can meet in
 * their barriers); RARN_ERR_CUDA if the ranks' CTAs do not fit on the device
 * at once.  For a process that holds every rank's buffers on one GPU, and to
 * check the barrier on one GPU. */
rarn_status rarn_tp_reduce_add_rms_norm_world(const rarn_tp_group *group, void *const *residuals,
                                              const void *gamma, int64_t T, int64_t H, float eps,
                                              rarn_dtype dt, void *stream);

/*
 * Sharing device memory between the ranks' processes (CUDA IPC): a handle of
 * RARN_IPC_HANDLE_BYTES bytes names the allocation that contains `ptr` and
 * the offset of `ptr` in it, so that any pointer returned by an allocator
 * (a caching allocator's block inside a larger allocation included) can be
 * shared.  rarn_ipc_export writes the handle of `ptr` (device memory of the
 * current device); rarn_ipc_import opens a handle made by ANOTHER process
 * (CUDA cannot open a process's own handles) and returns the pointer through
 * which this process addresses that memory (peer access enabled lazily);
 * rarn_ipc_close releases what rarn_ipc_import opened.  The exporting
 * process must keep the memory allocated while any importer uses it.
 * Errors: NULL arguments: RARN_ERR_INVALID_ARG; a handle this library did not
 * write: RARN_ERR_INVALID_ARG; a failed CUDA call: RARN_ERR_CUDA.
 */
#define RARN_IPC_HANDLE_BYTES 96
rarn_status rarn_ipc_export(const void *ptr, void *handle);
rarn_status rarn_ipc_import(const void *handle, void **ptr);
rarn_status rarn_ipc_close(void *ptr);

/* Rows that one launch sequence of rarn_gemm_add_rms_norm_noalloc covers for
 * a row length H: floor(floor((2^20 - 16) / (H / 128 + 1)) / 128) * 128
 * (16128 at H = 8192, 8064 at H = 16384); -1 if H is not supported. */
int64_t rarn_gemm_noalloc_rows(int64_t H);

/* Describe the GEMM kernels' tiling for a problem on a device with `num_sms`
 * SMs (if <= 0 the current device is queried; pure host logic when > 0),
 * under the current tuning knobs.  Writes a NUL-terminated description into
 * out[cap]; RARN_ERR_UNSUPPORTED (out says so) for a shape or type the GEMM
 * form rejects. */
rarn_status rarn_plan_gemm(int64_t T, int64_t H, int64_t K, rarn_dtype dt, int32_t num_sms,
                           char *out, size_t cap);

/* Static text for a status code. */
const char *rarn_status_string(rarn_status s);

/* CUDA error code (cudaError_t as int) of the last RARN_ERR_CUDA returned on
 * the calling thread; 0 if none. */
int rarn_last_cuda_error(void);

/* Select the kernel family for later calls from any thread (process-wide).
 * Returns RARN_ERR_INVALID_ARG for an unknown value. */
rarn_status rarn_set_path(rarn_path p);
rarn_path rarn_get_path(void);

/*
 * Programmatic dependent launch (process-wide, on by default).  When on,
 * every launch carries the programmatic-serialization attribute: the kernel
 * may be scheduled while the previous kernel on the stream is still running
 * and waits (griddepcontrol.wait) for it to finish before it touches global
 * memory, and it lets the next such kernel launch once each of its CTAs has
 * started its last row.  Results are the same either way; only launch gaps
 * differ.
 */
rarn_status rarn_set_pdl(int enable);
int rarn_get_pdl(void);

/*
 * Planner overrides for measurements and tests (process-wide, read by every
 * later call from any thread).  Each knob holds -1 ("the planner's own
 * choice", the default) or one of the values listed beside it; the planner
 * still applies its own limits after an override (a register budget, the
 * shared memory that fits, the shapes a kernel can take), so an override can
 * only steer the choice among kernels that can run the call.  Results are
 * the same under every setting, up to the documented summation-order
 * differences between kernel families.  Nothing here is read from the
 * environment.
 */
typedef enum rarn_tuning {
    RARN_TUNE_ROWS_PER_THREAD = 0,  /* 1, 2, 4, 8 (16: scalar rows): 16-byte packs per
                                       thread of the CTA-per-row kernels (grown again
                                       until the row fits the register budget) */
    RARN_TUNE_ROWS_GRID = 1,        /* 1 .. 2^31-1: CTAs of the CTA-per-row kernels
                                       (at most T) */
    RARN_TUNE_ROWS_PIPELINE = 2,    /* 0: no software pipelining across rows */
    RARN_TUNE_L2_ROWS = 3,          /* 0 .. 8: rows each CTA prefetches into L2 before
                                       its dependency wait (device buffers) */
    RARN_TUNE_STREAM_PACKS = 4,     /* 1, 2, 4: 16-byte packs per consumer thread and
                                       pipeline chunk of the stream kernel */
    RARN_TUNE_STREAM_GROUPS = 5,    /* 1, 2: consumer groups of the stream kernel when
                                       RARN_PATH_STREAM is forced */
    RARN_TUNE_GEMM_COLS = 6,        /* 256, 512: columns per CTA tile of the GEMM form */
    RARN_TUNE_GEMM_SLAB = 7,        /* 32, 64: K slab of the GEMM form, in elements */
    RARN_TUNE_GEMM_CTAS_PER_SM = 8, /* 1, 2: the non-persistent GEMM kernel */
    RARN_TUNE_GEMM_PERSISTENT = 9,  /* 0, 1: the persistent warp-specialised kernels */
    RARN_TUNE_GEMM_PAIR = 10,       /* 0, 1: SM pairs (cta_group::2) */
    RARN_TUNE_GEMM_NORM_IN_EPILOGUE = 11, /* 0: y from a separate norm kernel; 1: y in the
                                             persistent kernels' epilogue wherever it can run
                                             there (default: where K >= 3072, or K >= 2048
                                             with T >= 4096) */
    RARN_TUNE_GEMM_TAIL_SPLIT = 12, /* 0: no 128-column halves in the last round */
    RARN_TUNE_GEMM_SPLIT_K = 13,    /* 0: no split K for few rows */
    RARN_TUNE_FP8IN_RING = 14,      /* 0: register kernels only; 1: the TMA-fed ring
                                       kernel wherever the shape allows it */
    RARN_TUNE_FP8IN_PACK16 = 15,    /* 0: 8-element packs in the register kernels */
    RARN_TUNE_TP_PREFETCH = 16,     /* 0, 1: whether each CTA of the tensor-parallel form
                                       prefetches its next row into L2 (only streams in
                                       memory of the current device) */
    RARN_TUNE_COUNT = 17
} rarn_tuning;

/* Set one knob (-1 restores the planner's choice).  An unknown knob or a
 * value outside its list returns RARN_ERR_INVALID_ARG and changes nothing. */
rarn_status rarn_set_tuning(rarn_tuning knob, int64_t value);
/* Current value of a knob into *value (-1: the planner's choice). */
rarn_status rarn_get_tuning(rarn_tuning knob, int64_t *value);
/* Every knob back to -1. */
rarn_status rarn_reset_tuning(void);

/*
 * Test hook for the watchdog: in the next launch (on any thread) of a stream
 * kernel (16-bit partials, or the TMA-fed kernel of
 * rarn_reduce_add_rms_norm_fp8in) or of the GEMM form, CTA 0 expects 16 bytes
 * more for pipeline fill number `fill` (0-based, in issue order) than its
 * copies bring, so that fill never completes; every shared-memory barrier wait of that launch is
 * bounded by `wait_limit_ns` (1 ns .. 2 s).  The waits on that fill run out:
 * the kernel sets the watchdog word (bit 0 / 1: stream consumer / producer;
 * bit 2: GEMM kernel) and returns with its outputs invalid, and the context
 * stays usable.  In the next tensor-parallel launch with signal pads instead,
 * CTA 0 of rank `fill` (modulo N) never signals at entry, so the other ranks'
 * CTA 0 (and its own) wait out the limit (bit 3); the pads must then be
 * zeroed before the next call.  Returns RARN_ERR_INVALID_ARG for a negative fill or a limit
 * out of range.  Not for production use.
 */
rarn_status rarn_test_stall(long long fill, unsigned long long wait_limit_ns);

/*
 * Describe the kernel the current path setting would launch for a problem,
 * as text such as "stream smem=...", without launching anything.
 * `vec_ok` says whether every pointer is 16-byte aligned; `num_sms` is the
 * device's SM count (if <= 0 the current device is queried).  Writes a
 * NUL-terminated string of at most `cap` bytes to `out`.  Pure host logic when
 * num_sms > 0.
 */
rarn_status rarn_plan(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt, int vec_ok,
                      int num_sms, char *out, size_t cap);

/* rarn_plan for a residual of storage type `rdt` (see the general forms). */
rarn_status rarn_plan_ex(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt,
                         rarn_dtype rdt, int vec_ok, int num_sms, char *out, size_t cap);

/* rarn_plan for the 8-bit output forms (residual of the inputs' type). */
rarn_status rarn_plan_fp8(rarn_op op, int64_t T, int64_t H, int32_t R, rarn_dtype dt, int vec_ok,
                          int num_sms, char *out, size_t cap);

/*
 * Watchdog word of the current device.  Kernels that wait on shared-memory
 * barriers or on other ranks give up after a bounded time, set a bit here and
 * return without hanging; their outputs are then not valid.  Bit 0: a
 * stream-kernel consumer wait timed out; bit 1: a stream-kernel producer
 * wait; bit 2: a wait in a GEMM-form kernel; bit 3: a wait of the
 * tensor-parallel form's barrier between ranks.  Synchronises the device.  If
 * `clear` is nonzero the word is reset to 0 after reading.
 */
rarn_status rarn_watchdog(uint32_t *flags, int clear);

/* Which host memory the *_host entry points can use on the current device:
 * 2 = any host memory, pageable included (the device reaches it through the
 * host's page tables, e.g. Grace with NVLink-C2C); 1 = pinned, mapped host
 * memory only; 0 = none; -1 = the query failed (no device). */
int rarn_host_access(void);

/*
 * Measurement aid: the launch floor of the row kernels.  Launches `grid` CTAs
 * of `block` threads of a kernel that does only what every row kernel does
 * besides its row work: one thread per CTA prefetches `row_bytes` bytes at
 * rows + blockIdx * row_bytes into L2 (skipped when rows is NULL), the CTA
 * waits for the previous kernel on the stream (griddepcontrol.wait) and lets
 * the next one launch, under the same programmatic-dependent-launch setting
 * (rarn_set_pdl) as the compute calls.  Timed in the same harness as a
 * compute call, it gives the time no schedule of that call can go below.
 * `rows` (device memory, 16-byte aligned) must span grid * row_bytes bytes;
 * row_bytes is a multiple of 16 up to 2^20.  Nothing is written.  Errors:
 * grid < 1, block outside 1..1024 or a bad row argument: RARN_ERR_INVALID_ARG;
 * a failed launch: RARN_ERR_CUDA.  The pages have no counterpart.
 */
rarn_status rarn_launch_floor(const void *rows, int64_t row_bytes, int32_t grid, int32_t block,
                              void *stream);

/* ABI version: (major << 16) | minor. */
int rarn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RARN_H */
