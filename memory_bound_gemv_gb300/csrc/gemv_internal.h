// Internal declarations shared by the kernel translation units and the C-ABI
// shim.  Not part of the public interface (include/gemv.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mbg {

// Storage types.  DT_F16X32: binary16 weights with an FP32 x.
enum { DT_F32 = 0, DT_F16 = 1, DT_Q8 = 2, DT_Q4 = 3, DT_F16X32 = 4, DT_COUNT = 5 };

// x staging: bulk copy into shared memory, vector loads into shared memory,
// read through L1, element-wise kernel, held in registers (row-band kernel).
enum { XMODE_BULK = 0, XMODE_VEC = 1, XMODE_L1 = 2, XMODE_ELEM = 3, XMODE_REG = 4 };

// Kernel families: warp/sub-warp rows streamed with a rolling buffer, row
// tiles walked by a persistent grid, element-wise fallback, bulk-copy
// pipeline, row bands with x in registers (rows in flight in registers, or
// staged in shared memory by bulk copies), row bands whose quantised
// products run on the MMA unit (rows in flight in registers, or staged).
enum { KIND_VEC = 0, KIND_TILE = 1, KIND_ELEM = 2, KIND_BULK = 3, KIND_BAND = 4, KIND_SBAND = 5,
       KIND_MMA = 6, KIND_SMMA = 7 };

// Dot-product arithmetic: operands converted to FP32, or binary16 operands
// fed to mixed-precision FMAs with FP32 accumulation.
enum { MATH_F32 = 0, MATH_MIXED = 1 };

// Device status bits (the device status word).  DEVERR_UNDRAINED: after a
// wait gave up, the bounded wait for the block's own copies still in flight
// gave up too, so a copy may have landed in shared memory the block no
// longer owned.
enum : unsigned int { DEVERR_TIMEOUT = 1u, DEVERR_UNDRAINED = 2u };

// Test hooks: copies that a launch arms its barrier for but does not issue,
// so that the bounded wait on it runs out (nothing is copied, nothing
// faults).  SKIP_X: the bulk copy of x; SKIP_STAGE: the first weight stage
// of every bulk-pipeline block; SKIP_SEGMENT: the first row segment of every
// softmax block that stages rows by bulk copies; SKIP_PROBE: the first chunk
// of every bulk-copy probe block.
enum : unsigned int { SKIP_X = 1u, SKIP_STAGE = 2u, SKIP_SEGMENT = 4u, SKIP_PROBE = 8u };

// Columns per FP16 scale in the quantised formats.
constexpr int kGroup = 128;

// Row tiles whose warp partials are combined behind one block barrier.  One:
// the barrier after every tile keeps a block's warps in step, so each block
// requests its next tile as one dense unit; batching 8 tiles per barrier let
// the warps drift apart and measured 5-25 % slower on GB300.
constexpr int kTileBatch = 1;

struct GemvArgs {
    const void *A;            // weights, row-major, row pitch `row_bytes`
    const void *x;            // input vector
    float *y;                 // output
    const uint16_t *scales;   // [M][groups] binary16, quantised types only
    int64_t M;
    int64_t N;
    int64_t row_bytes;        // bytes per row of A
    int64_t groups;           // ceil(N / 128)
    int nchunks;              // row_bytes / 16 (vector kernels)
    unsigned int *err;        // device status word
    uint64_t wait_limit_ns;   // bound of every device-side wait
    unsigned int skip_copies; // test hook (SKIP_*): arm the barrier but issue no copy
    int scale_shift;          // scale group of 16-byte chunk c: c >> scale_shift
    int scale_elem_shift;     // scale group of column j: j >> scale_elem_shift
    int pdl;                  // stream the weights before waiting for the preceding
                              // kernel (kernels with PDL support are always launched
                              // with programmatic serialisation; without this flag they
                              // wait before touching memory)
};

struct Variant {
    int dtype;
    int lanes_per_row;   // threads sharing one row (tile kernels: up to 512)
    int rows_per_group;  // RPW (vector kernels)
    int unroll;          // U (vector kernels) or chunks per thread per row (tile kernels)
    int warps;           // warps per block
    int xmode;
    const char *name;
    // Launches the kernel on `grid` blocks with `smem` bytes of dynamic shared memory.
    void (*launch)(const GemvArgs &, unsigned grid, size_t smem, cudaStream_t, bool pdl);
    // Raises the kernel's dynamic shared memory limit.
    cudaError_t (*set_smem_limit)(int bytes);
    int kind;
    int x_offset;        // bytes of shared memory in front of the staged x
    // Resident blocks per SM for a given dynamic shared memory size (tile kernels).
    cudaError_t (*occupancy)(int *blocks, size_t smem);
    int math;            // MATH_F32 or MATH_MIXED
    int stages;          // bulk-pipeline depth (KIND_BULK)
    bool x_regs = false; // bulk pipeline keeps x in registers, not in shared memory
    int tile_rows = 1;   // row bands: consecutive rows per tile
    int max_blocks_per_sm = 0;  // cap on the persistent grid (0: as many as fit), leaving room
                                // for the next launch's blocks to start alongside
    int scale_align = 2;        // MMA row bands: alignment (bytes) the kernel needs of the scales
    bool supports_pdl() const
    {
        return kind == KIND_TILE || kind == KIND_BULK || kind == KIND_BAND || kind == KIND_SBAND ||
               kind == KIND_MMA || kind == KIND_SMMA;
    }
    int rows_per_block() const
    {
        if (kind == KIND_TILE) return warps * 32 / lanes_per_row;
        if (kind == KIND_BULK) return rows_per_group;
        if (kind == KIND_BAND || kind == KIND_SBAND || kind == KIND_MMA || kind == KIND_SMMA)
            return tile_rows;  // one block per tile at most
        return warps * (32 / lanes_per_row) * rows_per_group;
    }
};

// Shared-memory layout of the bulk-pipeline kernel (host and device agree on
// it): S "full" and S "reduced" barriers, the x barrier and the abort flag,
// one set of warp partials per stage, x, S stages of RS rows of A, and
// (quantised) S stages of RS rows of scales.  T counts consumer threads.
struct BulkLayout {
    int part, x, stage, scale, total;   // byte offsets and total size
    int stage_bytes, scale_bytes;       // capacity of one stage
};

__host__ __device__ inline int round16(int64_t v) { return static_cast<int>((v + 15) / 16 * 16); }

// Shared-memory layout of the staged row-band kernel (host and device agree
// on it): S mbarriers, the warp partials [2][U][NW], then S stages of G rows
// of A followed by their G rows of scales.
struct StageBandLayout {
    int part, stage, stage_bytes, scale_off, total;
};

__host__ __device__ inline StageBandLayout stageband_layout(int S, int U, int NW, int G, int64_t row_bytes,
                                                           int64_t groups, bool quant)
{
    StageBandLayout L;
    L.part = round16(8 * S);
    L.stage = (L.part + 2 * U * NW * 4 + 127) / 128 * 128;
    L.scale_off = static_cast<int>(G * row_bytes);
    L.stage_bytes = L.scale_off + (quant ? round16(G * 2 * groups) : 0);
    L.total = L.stage + S * L.stage_bytes;
    return L;
}

__host__ __device__ inline BulkLayout bulk_layout(int S, int RS, int T, int64_t row_bytes,
                                                  int64_t x_bytes, int64_t groups, bool quant)
{
    BulkLayout L;
    L.part = round16(8 * (2 * S + 1) + 4);
    L.x = L.part + round16(static_cast<int64_t>(S) * T * RS * 4);  // one partial per thread and row
    L.stage = L.x + round16(x_bytes);
    L.stage_bytes = static_cast<int>(RS * row_bytes);
    L.scale = L.stage + S * L.stage_bytes;
    // one scale per row (groups == 1) is read from global memory, not staged
    L.scale_bytes = (quant && groups > 1) ? round16(RS * 2 * groups) : 0;
    L.total = L.scale + S * L.scale_bytes;
    return L;
}

// Variant tables, one per storage type (defined in gemv_<dtype>.cu).
const Variant *variants_f32(int *count);
const Variant *variants_f16(int *count);
const Variant *variants_q8(int *count);
const Variant *variants_q4(int *count);
const Variant *variants_f16x32(int *count);

// Probe kernels (gemv_probe.cu).
struct ProbeVariant {
    const char *name;
    int threads;
    int unroll;
    int blocks_per_sm;
    int segment;  // 0: grid-stride tiles, 1: one contiguous segment per warp, 2: prefetching tiles
    // limit_ns bounds the bulk patterns' waits; skip_first: SKIP_PROBE hook
    void (*launch)(const void *buf, size_t n16, unsigned long long *sink, unsigned grid,
                   uint64_t limit_ns, bool skip_first, cudaStream_t s);
};
const ProbeVariant *probe_variants(int *count);

// Dequantisation kernels (gemv_dequant.cu).
void launch_dequant(int dtype, const void *A, const uint16_t *scales, float *W, int64_t M,
                    int64_t N, bool vec, cudaStream_t s);

// N == 0: y = 0.
void launch_fill_zero(float *y, int64_t M, cudaStream_t s);

// Copy of x from page-locked host memory by a kernel (gemv_host.cu), launched
// with programmatic stream serialisation; early: x is read before the wait
// for the preceding kernel.
void launch_copy_in(const void *src, void *dst, int64_t bytes, bool early, cudaStream_t s);

// Test helper (gemv_host.cu): a kernel that lets its successor start at once
// and fills dst with `word` only after delay_ns.
void launch_late_fill(void *dst, size_t bytes, uint32_t word, uint64_t delay_ns, cudaStream_t s);

// Symmetric quantisation (gemv_quantize.cu): bits 8 or 4; one scale per row
// or per 128 columns; FP32 or binary16 weights.
void launch_quantize(int bits, bool per_row, bool f16in, const void *W, void *A, uint16_t *scales,
                     double *sq_err, int64_t M, int64_t N, int sm_count, cudaStream_t s);

// Row softmax (gemv_softmax.cu).  variant < 0 chooses; cudaErrorNotSupported
// when the variant cannot serve the shape or alignment.
cudaError_t launch_softmax(const uint16_t *x, uint16_t *y, int64_t M, int64_t N, int variant,
                           unsigned int *err, uint64_t wait_limit_ns, unsigned int skip,
                           cudaStream_t s);
int softmax_variant_count();
const char *softmax_variant_name(int v);

// Copy probe (gemv_softmax.cu).
cudaError_t launch_copy_probe(const void *src, void *dst, size_t bytes, int variant, int sm_count,
                              cudaStream_t s);
int copy_variant_count();
const char *copy_variant_name(int v);

}  // namespace mbg
