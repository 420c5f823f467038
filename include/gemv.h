/*
 * gemv.h -- C ABI of the GB300 (sm_103a) GEMV library.
 *
 * Computes the row-major matrix-vector product
 *
 *     y[i] = sum_{j=0}^{N-1} A[i,j] * x[j],   0 <= i < M,   A[i,j] = A[i*N + j]
 *
 * ("Making GEMV Fast", sections "Row-major indexing refresher" and
 * "Algorithm"; "llama.cpp GEMV CUDA", the kernel-equation paragraph).
 * Weights may be FP32, FP16, or weight-only quantised INT8 / INT4 with one
 * FP16 scale per row per 128 contiguous columns ("membound", section "The
 * kernel decode actually runs: dequant GEMV").  Accumulation and y are FP32.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named A, x, y, scales, W, buf and sink are DEVICE pointers on the
 *   current CUDA device.  The caller allocates and owns them.  The library
 *   never allocates device or host memory; its only device state is one
 *   status word per device, a static variable inside the library.
 * - FP16 data is passed as IEEE 754 binary16 bit patterns (uint16_t).
 * - `stream` is a cudaStream_t (CUstream) passed as void*; NULL selects the
 *   legacy default stream.  Every call only enqueues work and returns: a
 *   status of GEMV_OK means "validated and launched", not "finished".
 * - Sizes are element counts (int64_t).  M == 0 is a no-op.  N == 0 writes
 *   y[0..M) = 0 (A and x may then be NULL).  Negative sizes are rejected.
 * - Alignment: each pointer must be aligned to its element size, else
 *   GEMV_ERR_MISALIGNED.  16-byte aligned A and x with a row pitch that is a
 *   multiple of 16 bytes take the vectorised kernels; any other legal layout
 *   takes an element-wise kernel that gives the same results more slowly.
 * - y must not overlap A, x or scales (not checked).
 * - Errors are returned, never raised: the library does not exit, abort or
 *   trap.  Launch failures return GEMV_ERR_LAUNCH (gemv_last_cuda_error()
 *   gives the CUDA code).  A device-side wait that gives up sets the device
 *   status word, which gemv_get_device_error() reports as GEMV_ERR_TIMEOUT.
 * - Calls on different streams may run concurrently; the entry points keep
 *   no per-call host state and are safe to call from several threads.
 */
#ifndef MEMORY_BOUND_GEMV_GB300_GEMV_H
#define MEMORY_BOUND_GEMV_GB300_GEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMV_OK = 0,
    GEMV_ERR_INVALID_VALUE = 1, /* NULL pointer, negative size, bad variant id */
    GEMV_ERR_MISALIGNED = 2,    /* a pointer not aligned to its element size */
    GEMV_ERR_UNSUPPORTED = 3,   /* e.g. INT4 with odd N, size beyond the index range */
    GEMV_ERR_LAUNCH = 4,        /* the CUDA launch failed */
    GEMV_ERR_TIMEOUT = 5,       /* a device-side wait gave up (see gemv_get_device_error) */
    GEMV_ERR_CUDA = 6,          /* another CUDA runtime call failed */
    GEMV_ERR_TIMEOUT_UNDRAINED = 7 /* as GEMV_ERR_TIMEOUT, and the bounded wait for the block's own
                                      copies still in flight gave up too (see
                                      gemv_get_device_error) */
} gemv_status_t;

/* Storage types, used by the variant-introspection calls. */
typedef enum {
    GEMV_F32 = 0,
    GEMV_F16 = 1,
    GEMV_Q8 = 2,
    GEMV_Q4 = 3,
    GEMV_F16_X32 = 4 /* binary16 weights, FP32 x (gemv_f16_xf32) */
} gemv_dtype_t;

/*
 * FP32 GEMV.  A: float [M][N] row-major, x: float [N], y: float [M].
 * "cuda-gemv-optimization", kernel 4 "Warp-level reduction"; "Making GEMV
 * Fast", section "Turning that access pattern into code".
 */
gemv_status_t gemv_f32(const float *A, const float *x, float *y, int64_t M, int64_t N,
                       void *stream);

/*
 * FP16 weights and x, FP32 accumulate and output.  A: binary16 [M][N],
 * x: binary16 [N], y: float [M].
 * "membound", section "The stages": kernel "vec" (128-bit loads, FP32
 * accumulation of converted halves); "llama.cpp GEMV CUDA" (FP16 weights and
 * hidden state, FP32 accumulate and output).
 */
gemv_status_t gemv_f16(const uint16_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                       void *stream);

/*
 * INT8 weight-only GEMV: y[i] = sum_j s[i, j/128] * q[i,j] * x[j].
 * A: int8 [M][N] (q in [-128, 127]); scales: binary16 [M][ceil(N/128)]
 * row-major; x: binary16 [N]; y: float [M].  The dequantised weight
 * FP32(s) * q is exact in FP32.
 * "membound", section "The kernel decode actually runs: dequant GEMV" (the
 * page uses one scale per row; a row whose group scales are all equal is that
 * case).
 */
gemv_status_t gemv_q8(const int8_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                      const uint16_t *scales, void *stream);

/*
 * INT4 weight-only GEMV, same formula as gemv_q8.  A: uint8 [M][N/2]; column
 * j of a row is byte j/2, low nibble for even j and high nibble for odd j,
 * read as 4-bit two's complement in [-8, 7].  N must be even, else
 * GEMV_ERR_UNSUPPORTED.  scales, x, y as for gemv_q8.
 * "membound", section "The kernel decode actually runs: dequant GEMV"
 * (two weights per byte, symmetric per-group-of-128 FP16 scales).
 */
gemv_status_t gemv_q4(const uint8_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                      const uint16_t *scales, void *stream);

/*
 * FP16 weights with an FP32 x: A: binary16 [M][N], x: float [N], y: float
 * [M].  Each weight is widened to FP32 and multiplied by x[j] in FP32.  x must
 * be 4-byte aligned; the vectorised kernels need A and x 16-byte aligned and
 * N a multiple of 8.
 * "llama.cpp GEMV CUDA", implementation note (the hidden state may be kept in
 * FP32 while the weights are FP16).
 */
gemv_status_t gemv_f16_xf32(const uint16_t *A, const float *x, float *y, int64_t M, int64_t N,
                            void *stream);

/*
 * INT8 weight-only GEMV with ONE scale per row: y[i] = s[i] * sum_j q[i,j] *
 * x[j], computed as sum_j (FP32(s[i]) * q[i,j]) * x[j].  A: int8 [M][N];
 * row_scales: binary16 [M]; x: binary16 [N]; y: float [M].  Same results as
 * gemv_q8 with every group scale of row i equal to s[i].  The bulk-copy
 * pipeline is not used for this layout (a row's scales are not a 16-byte
 * block); the row-tile and warp-per-row kernels are.
 * "membound", section "The kernel decode actually runs: dequant GEMV" (the
 * per-row scale of the page's kernel).
 */
gemv_status_t gemv_q8_rowscale(const int8_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                               const uint16_t *row_scales, void *stream);
/* gemv_q8_rowscale with the launch flags of gemv_ex (below). */
gemv_status_t gemv_q8_rowscale_ex(const int8_t *A, const uint16_t *x, float *y, int64_t M,
                                  int64_t N, const uint16_t *row_scales, unsigned flags,
                                  void *stream);

/*
 * Any of the GEMVs above with 128-column scale groups (dtype: gemv_dtype_t)
 * with launch flags.  scales is ignored for the unquantised types.
 *
 * GEMV_FLAG_OVERLAP_PRECEDING: the caller guarantees that A and scales are
 * not written by the kernel that precedes this call on `stream` (model
 * weights in a decode loop are the intended case).  The GEMV is then launched
 * with programmatic dependent launch: its blocks may start while the
 * preceding kernel is still running and begin streaming A and scales at once;
 * they read x and write y only after the preceding kernel has completed and
 * its memory is visible (griddepcontrol.wait).  Every GEMV kernel of this
 * library signals early that its successor may start, so a chain of GEMVs on
 * one stream overlaps each launch's start-up with the previous one's tail.
 * Kernel families without this support are launched normally.  Any other flag
 * bit returns GEMV_ERR_INVALID_VALUE.
 * Launch overlap as described for NVIDIA's programmatic dependent launch;
 * the pages have no counterpart (their kernels are timed one launch at a time,
 * "membound", "Results").
 */
#define GEMV_FLAG_OVERLAP_PRECEDING 1u
gemv_status_t gemv_ex(int dtype, const void *A, const void *x, float *y, int64_t M, int64_t N,
                      const uint16_t *scales, unsigned flags, void *stream);

/*
 * gemv_ex with x and y in HOST memory: one call per decode step that takes
 * the input vector from, and returns the output to, page-locked host buffers.
 * x_host: page-locked host memory (cudaHostAlloc / cudaHostRegister / a
 * pinned torch tensor), N elements of x's type; else GEMV_ERR_INVALID_VALUE.
 * x_dev: device buffer of the same size that receives x (the caller owns it;
 * 16-byte aligned for the vectorised kernels).  y_host: page-locked host
 * memory (device memory is accepted too) of M floats, written by the GEMV
 * kernel directly; read it after synchronising `stream`.  A, scales and dtype
 * as for gemv_ex.
 * The copy of x is a small kernel that reads the host buffer over the
 * CPU-GPU link; it is launched with programmatic dependent launch (its blocks
 * are scheduled while the preceding kernel drains) and reads x only after
 * that kernel has completed.  The GEMV is launched the same way after it and
 * waits for the copy to complete before it reads A, scales or x, so the call
 * keeps the ordering of plain launches.
 * GEMV_FLAG_OVERLAP_PRECEDING: the kernel that precedes the call on `stream`
 * writes neither A, scales nor x_host (a previous call of this function
 * qualifies); the copy then reads x_host before that kernel has finished and
 * writes x_dev only after it, and the GEMV streams its weights while x is
 * still being fetched.  x_host must not change until the call has run on the
 * stream.
 * Same results as gemv_ex on device copies of x (bit for bit).
 * The pages time device-resident operands only; this call has no
 * counterpart there.
 */
gemv_status_t gemv_ex_host(int dtype, const void *A, const void *x_host, void *x_dev, float *y_host,
                           int64_t M, int64_t N, const uint16_t *scales, unsigned flags,
                           void *stream);

/*
 * gemv_ex_host for callers that cannot allocate device memory: the same
 * computation and results, with the device copy of x kept in a fixed array
 * inside the library instead of a caller-provided x_dev.  Meant for code
 * that may not allocate once it is running (real-time or certified loops
 * that allocate only at start-up), plug-ins whose host program owns the
 * device allocator, and callers that have only this C ABI.  The other
 * arguments are those of gemv_ex_host.
 * Limit: x may take at most GEMV_NOALLOC_X_MAX_BYTES bytes (N <= 131072
 * binary16 values or 65536 FP32 values); a longer x returns
 * GEMV_ERR_UNSUPPORTED before anything is launched.  Every GPU that loads the
 * library holds this array (256 KiB) until the process exits; nothing is
 * allocated by the call.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * All calls on a device share the one array and leave the last x in it; it
 * is fully rewritten before each use, so nothing needs clearing.  Calls that
 * can run at the same time on the GPU (different streams, or other threads
 * without ordering) race on it: issue them on one stream.
 * The pages have no counterpart to this entry point.
 */
#define GEMV_NOALLOC_X_MAX_BYTES 262144
gemv_status_t gemv_ex_host_noalloc(int dtype, const void *A, const void *x_host, float *y_host,
                                   int64_t M, int64_t N, const uint16_t *scales, unsigned flags,
                                   void *stream);

/*
 * Pure-read bandwidth probe: streams buf[0..bytes) once, either with the
 * same 16-byte read-only loads the GEMV kernels use or (the "bulk_" patterns)
 * with bulk asynchronous copies into shared-memory rings, and folds every
 * word into the low 32 bits of *sink with XOR (so no read is dead code).
 * bytes must be a multiple of 16 and buf 16-byte aligned.  `variant` selects
 * the read pattern (0 .. gemv_probe_variant_count()-1).  A bulk pattern whose
 * bounded wait gives up sets bit 63 of *sink (and bit 62 when its wait for
 * the copies still in flight gave up too).  Achieved bytes / time is the
 * measured read ceiling that memory-bandwidth utilisation is quoted against.
 * "membound", section "Why GEMV, and why MBU" (pure-read probe as the
 * denominator for a read-dominated kernel).
 */
gemv_status_t gemv_probe_read(const void *buf, size_t bytes, unsigned long long *sink,
                              int variant, void *stream);
int gemv_probe_variant_count(void);
const char *gemv_probe_variant_name(int variant);

/*
 * Copy probe: reads src[0..bytes) and writes it to dst with the same 16-byte
 * streaming loads (and streaming stores) -- the read + write ceiling that a
 * balanced kernel such as the row softmax is quoted against ("membound",
 * section "Bonus kernel: online softmax": the copy ceiling, not pure read, is
 * the denominator of a kernel that reads and writes every element once).
 * bytes a multiple of 16, both pointers 16-byte aligned, no overlap.
 */
gemv_status_t gemv_probe_copy(const void *src, void *dst, size_t bytes, int variant, void *stream);
int gemv_probe_copy_variant_count(void);
const char *gemv_probe_copy_variant_name(int variant);

/*
 * Row softmax of binary16 data: y[i, j] = exp(x[i,j] - m_i) / sum_k exp(x[i,k] - m_i)
 * with m_i the maximum of row i, FP32 arithmetic, binary16 output (round to
 * nearest even).  x and y: binary16 [M][N] row-major; y may be x (in place).
 * "membound", section "Bonus kernel: online softmax" (the online update of
 * the running maximum and sum, Milakov & Gimelshein).  Rows of up to 131072
 * columns with N % 8 == 0 and 16-byte aligned pointers are read once and
 * written once (one block, or a cluster of up to eight blocks combining
 * their partial maxima and sums through distributed shared memory); any other
 * shape uses two passes over the row.  Rows whose elements are all -inf are
 * not supported (their result is unspecified).
 */
gemv_status_t gemv_softmax_f16(const uint16_t *x, uint16_t *y, int64_t M, int64_t N, void *stream);
int gemv_softmax_variant_count(void);
const char *gemv_softmax_variant_name(int variant);
gemv_status_t gemv_softmax_run_variant(int variant, const uint16_t *x, uint16_t *y, int64_t M,
                                       int64_t N, void *stream);

/*
 * Symmetric weight quantisation: produces the A and scales operands of
 * gemv_q8 (per_row = 0: one scale per 128 columns, scales [M][ceil(N/128)]),
 * gemv_q8_rowscale (per_row = 1: scales [M]) and gemv_q4 (one scale per 128
 * columns, A packed as gemv_q4 reads it; N must be even, else
 * GEMV_ERR_UNSUPPORTED).
 * W: [M][N] row-major, FP32 (w_dtype = GEMV_F32) or binary16 (GEMV_F16).
 * Per group, in FP32: a = max|w|; s = a / qmax (qmax 127 for INT8, 7 for
 * INT4; IEEE division); the stored scale is binary16(s) rounded to nearest
 * even (an overflow to infinity stores 65504 instead); each code is
 * q = clamp(rint(w / scale), -qmax, qmax), with q = 0 where the scale is 0 or w
 * is NaN.  sq_err: NULL, or a device double to which the call ADDS
 * sum (w - scale*q)^2 over all weights (the caller zeroes it; the order of the
 * additions varies, so the last bits may differ between runs).  Codes and
 * scales are deterministic.  W, A and scales must not overlap.
 * "membound", section "The kernel decode actually runs: dequant GEMV" (INT8
 * with a symmetric per-row scale, INT4 with symmetric per-128-column scales,
 * and the quantisation RMSE of U[-1,1] weights: 2.3e-3 and 4.1e-2).
 */
gemv_status_t gemv_quantize_q8(const void *W, int w_dtype, int8_t *A, uint16_t *scales, int64_t M,
                               int64_t N, int per_row, double *sq_err, void *stream);
gemv_status_t gemv_quantize_q4(const void *W, int w_dtype, uint8_t *A, uint16_t *scales, int64_t M,
                               int64_t N, double *sq_err, void *stream);

/*
 * Dequantise to FP32: W[i*N + j] = FP32(s[i, j/128]) * q[i,j], using the
 * same unpacking code as the GEMV kernels.  The product is exact, so W must
 * equal the oracle's dequantised weights bit for bit.  Test helper:
 * "membound", section "dequant GEMV" (reference computed on q*s exactly).
 */
gemv_status_t gemv_dequant_q8(const int8_t *A, const uint16_t *scales, float *W, int64_t M,
                              int64_t N, void *stream);
gemv_status_t gemv_dequant_q4(const uint8_t *A, const uint16_t *scales, float *W, int64_t M,
                              int64_t N, void *stream);

/*
 * Kernel variants.  Every dtype has a table of compiled variants (kernel
 * family, threads per row, loads in flight, warps per block, how x is
 * staged).  The plain entry points pick one by shape; these calls run a
 * chosen one so that each can be checked and timed.  A variant that cannot
 * serve the given shape or alignment returns GEMV_ERR_UNSUPPORTED.
 *
 * Families: 0 = rows of a warp (or of a fraction of one) streamed with a
 * rolling buffer of loads; 1 = row tiles: a group of threads requests a whole
 * row at once and a persistent grid walks consecutive rows in order;
 * 2 = element-wise kernel for layouts without 16-byte alignment;
 * 3 = bulk-copy pipeline: tiles of consecutive rows streamed into a ring of
 * shared-memory stages by bulk async copies (rows_per_group = rows per stage,
 * threads_per_row = consumer threads of the block, plus one producer warp);
 * 4 = row bands: for rows of exactly threads_per_row * unroll 16-byte chunks,
 * each thread keeps the x of its chunks in registers and a window of
 * rows_per_group rows in flight in registers; tiles of consecutive rows are
 * dealt to the blocks of a persistent grid in grid-stride order;
 * 5 = staged row bands: the same work split, with the tiles streamed into a
 * ring of shared-memory stages by bulk async copies (rows_per_group = rows
 * per window of tiles);
 * 6 = MMA row bands (INT8 / INT4): tiles of two consecutive rows, each warp
 * takes `unroll` steps of 512 bytes of each row (rows of exactly warps *
 * unroll * 512 bytes); the exact binary16 codes are multiplied by x and
 * summed in FP32 by the warp-level MMA instruction (mma.sync m16n8k16), x
 * held in registers; rows_per_group = rows per window of tiles;
 * 7 = staged MMA row bands: the same arithmetic, with tiles of one or more
 * row pairs streamed into a ring of shared-memory stages by bulk async
 * copies (rows_per_group = rows per window of tiles).
 */
typedef struct {
    int dtype;           /* gemv_dtype_t */
    int kind;            /* kernel family, see above */
    int threads_per_row; /* threads that share one row: 1..32 (family 0), 1..512 (family 1),
                            the consumer threads of the block (family 3), the block (families 4-7) */
    int rows_per_group;  /* rows one lane group streams together (family 0, x reuse); rows per
                            stage (family 3); rows in flight per thread (families 4, 6), rows
                            per window (families 5, 7) */
    int unroll;          /* family 0: loads in flight per lane; family 1: chunks per thread;
                            family 3: chunks per consumer thread and row when the variant is
                            specialised for rows of exactly unroll * threads_per_row chunks
                            (0: any row length); families 4, 5: chunks per thread and row;
                            families 6, 7: 512-byte steps per warp and row */
    int warps;           /* warps per block */
    int math;            /* 0: operands converted to FP32; 1: binary16 operands into
                            mixed-precision FMAs with FP32 accumulation */
    int xmode;          /* 0: x copied to shared memory by a bulk async copy,
                           1: x copied to shared memory by vector loads,
                           2: x read through the L1 cache, 3: element-wise kernel,
                           4: x held in registers (families 4, 5) */
    char name[48];
} gemv_variant_info_t;

int gemv_variant_count(int dtype);
gemv_status_t gemv_variant_info(int dtype, int variant, gemv_variant_info_t *info);
/* Variant the plain entry point would use for these arguments (-1 on bad args). */
int gemv_select_variant(int dtype, const void *A, const void *x, int64_t M, int64_t N);
gemv_status_t gemv_run_variant(int dtype, int variant, const void *A, const void *x, float *y,
                               int64_t M, int64_t N, const uint16_t *scales, void *stream);
/* gemv_run_variant with the launch flags of gemv_ex. */
gemv_status_t gemv_run_variant_ex(int dtype, int variant, const void *A, const void *x, float *y,
                                  int64_t M, int64_t N, const uint16_t *scales, unsigned flags,
                                  void *stream);
/* The same two calls for gemv_q8_rowscale (variant ids index the INT8 table;
 * the bulk-copy variants return GEMV_ERR_UNSUPPORTED there). */
int gemv_q8_rowscale_select_variant(const int8_t *A, const uint16_t *x, int64_t M, int64_t N);
gemv_status_t gemv_q8_rowscale_run_variant(int variant, const int8_t *A, const uint16_t *x, float *y,
                                           int64_t M, int64_t N, const uint16_t *row_scales,
                                           void *stream);

/*
 * Synchronises `stream`, reads and clears this device's status word.
 * Returns GEMV_ERR_TIMEOUT if any kernel gave up a bounded wait since the
 * last call, GEMV_OK otherwise (GEMV_ERR_CUDA if the CUDA calls fail).
 * GEMV_ERR_TIMEOUT_UNDRAINED: a block that gave up then also gave up waiting
 * for a bulk copy it had issued, so that copy may have landed in shared
 * memory after the block exited; treat every result computed on this device
 * since the previous call as suspect.
 */
gemv_status_t gemv_get_device_error(void *stream);

/* Test hooks.  Limit of every device-side wait in nanoseconds (default one
 * second; values below 100 us are raised to 100 us, 0 restores the default),
 * and switches that make the next launches arm a barrier for a bulk copy
 * without issuing the copy, so that the bounded wait on it runs out (nothing
 * is copied, nothing faults):
 *   GEMV_DEBUG_SKIP_X        the bulk copy of x (GEMV kernels staging x that way);
 *   GEMV_DEBUG_SKIP_STAGE    the first weight stage of every bulk-pipeline block;
 *   GEMV_DEBUG_SKIP_SEGMENT  the first row segment of every softmax block that
 *                            stages rows by bulk copies;
 *   GEMV_DEBUG_SKIP_PROBE    the first chunk of every bulk-copy probe block.
 * gemv_debug_skip_x_copy(on) sets or clears GEMV_DEBUG_SKIP_X alone. */
#define GEMV_DEBUG_SKIP_X 1u
#define GEMV_DEBUG_SKIP_STAGE 2u
#define GEMV_DEBUG_SKIP_SEGMENT 4u
#define GEMV_DEBUG_SKIP_PROBE 8u
void gemv_debug_set_wait_limit_ns(uint64_t ns);
void gemv_debug_skip_x_copy(int on);
void gemv_debug_skip_copies(unsigned int mask);

/* Test hook: a kernel that lets the next kernel on `stream` start at once
 * (programmatic dependent launch) and only after delay_ns fills
 * dst[0..bytes) with the 32-bit pattern `word` -- a preceding kernel that
 * writes a GEMV's operands late, for checking the ordering of gemv_ex_host.
 * dst: device memory, 4-byte aligned; bytes a multiple of 4; delay_ns at most
 * one second (longer is clamped). */
gemv_status_t gemv_debug_late_fill(void *dst, size_t bytes, uint32_t word, uint64_t delay_ns,
                                   void *stream);

const char *gemv_status_string(gemv_status_t status);
int gemv_last_cuda_error(void); /* last cudaError_t seen by this thread, 0 if none */
const char *gemv_build_info(void);

#ifdef __cplusplus
}
#endif

#endif
