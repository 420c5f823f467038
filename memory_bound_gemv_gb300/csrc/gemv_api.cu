// C-ABI entry points (include/gemv.h): argument validation, variant choice,
// per-device set-up and error reporting.  All device work is in the kernels
// of the other translation units; this file launches them and never
// allocates memory.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>
#include <climits>
#include <functional>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/gemv.h"
#include "gemv_internal.h"

#define MBG_STR2(v) #v
#define MBG_STR(v) MBG_STR2(v)

namespace mbg {
namespace {

// The device status word (bit DEVERR_TIMEOUT: a bounded wait gave up).  A
// static device variable, so the library needs no allocation for it.
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;
// Largest x kept in shared memory by the automatic choice; longer x is read
// through L1 so that several blocks still fit on an SM.
constexpr int64_t kAutoSmemX = 64 * 1024;
// Matrices up to this size may take a row band with a capped grid.
constexpr int64_t kSmallMatrixBytes = 16ll << 20;
// Widest row group and chunks per thread of the compiled tile kernels.
constexpr int kTileMaxThreads = 512;
constexpr int kTileChunks = 8;

struct DeviceState {
    std::once_flag once;
    cudaError_t init_error = cudaSuccess;
    unsigned int *status = nullptr;  // device address of g_device_status
    int sm_count = 0;
    int max_smem = 0;                // opt-in dynamic shared memory per block
    // resident blocks per SM of a tile variant, keyed by (dtype, variant, smem bytes)
    std::mutex occ_mutex;
    std::map<std::tuple<int, int, size_t>, int> occ;
};
DeviceState g_devices[kMaxDevices];

std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};
std::atomic<unsigned int> g_skip_copies{0};
thread_local int t_last_cuda_error = 0;

gemv_status_t cuda_fail(cudaError_t e, gemv_status_t code)
{
    t_last_cuda_error = static_cast<int>(e);
    return code;
}

const Variant *table(int dtype, int *count)
{
    switch (dtype) {
    case DT_F32: return variants_f32(count);
    case DT_F16: return variants_f16(count);
    case DT_Q8: return variants_q8(count);
    case DT_Q4: return variants_q4(count);
    case DT_F16X32: return variants_f16x32(count);
    default: *count = 0; return nullptr;
    }
}

void init_device(DeviceState &d, int dev)
{
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    for (int dt = 0; e == cudaSuccess && dt < DT_COUNT; ++dt) {
        int n = 0;
        const Variant *v = table(dt, &n);
        for (int k = 0; e == cudaSuccess && k < n; ++k) e = v[k].set_smem_limit(d.max_smem);
    }
    d.init_error = e;
}

// Set-up of the current device on its first use (symbol address of the status
// word, SM count, shared-memory limits).  Returns nullptr on failure.
DeviceState *current_device()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState &d = g_devices[dev];
    std::call_once(d.once, init_device, std::ref(d), dev);
    if (d.init_error != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(d.init_error);
        return nullptr;
    }
    return &d;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t row_bytes_of(int dtype, int64_t N)
{
    switch (dtype) {
    case DT_F32: return 4 * N;
    case DT_F16:
    case DT_F16X32: return 2 * N;
    case DT_Q8: return N;
    default: return N / 2;
    }
}

int a_align(int dtype) { return dtype == DT_F32 ? 4 : (dtype == DT_F16 || dtype == DT_F16X32) ? 2 : 1; }
int x_align(int dtype) { return (dtype == DT_F32 || dtype == DT_F16X32) ? 4 : 2; }
int x_elem_bytes(int dtype) { return (dtype == DT_F32 || dtype == DT_F16X32) ? 4 : 2; }

bool is_quant(int dtype) { return dtype == DT_Q8 || dtype == DT_Q4; }

// Scale grouping: 128 columns per scale, or one scale per row.
enum { SCALES_GROUP128 = 0, SCALES_PER_ROW = 1 };
int64_t scale_groups(int64_t N, int mode) { return mode == SCALES_PER_ROW ? 1 : (N + kGroup - 1) / kGroup; }

// Common argument checks.  Returns GEMV_OK when the call may proceed.
gemv_status_t validate(int dtype, const void *A, const void *x, const float *y, int64_t M,
                       int64_t N, const uint16_t *scales)
{
    if (dtype < 0 || dtype >= DT_COUNT) return GEMV_ERR_INVALID_VALUE;
    if (M < 0 || N < 0) return GEMV_ERR_INVALID_VALUE;
    if (M == 0) return GEMV_OK;
    if (!y) return GEMV_ERR_INVALID_VALUE;
    if (!aligned(y, 4)) return GEMV_ERR_MISALIGNED;
    if (N == 0) return GEMV_OK;
    if (!A || !x) return GEMV_ERR_INVALID_VALUE;
    const bool quant = dtype == DT_Q8 || dtype == DT_Q4;
    if (quant && !scales) return GEMV_ERR_INVALID_VALUE;
    if (dtype == DT_Q4 && (N % 2)) return GEMV_ERR_UNSUPPORTED;
    if (!aligned(A, a_align(dtype)) || !aligned(x, x_align(dtype))) return GEMV_ERR_MISALIGNED;
    if (quant && !aligned(scales, 2)) return GEMV_ERR_MISALIGNED;
    // index range: byte offsets of A must fit in int64
    if (M > INT64_MAX / (row_bytes_of(dtype, N) > 0 ? row_bytes_of(dtype, N) : 1))
        return GEMV_ERR_UNSUPPORTED;
    return GEMV_OK;
}

// Dynamic shared memory of variant v for a row of N columns.
size_t smem_bytes(const Variant &v, int dtype, int64_t N, int64_t groups)
{
    if (v.kind == KIND_BULK) {
        const int64_t rb = row_bytes_of(dtype, N);
        const int64_t xb = v.x_regs ? 0 : N * x_elem_bytes(dtype);
        const BulkLayout L = bulk_layout(v.stages, v.rows_per_group, v.warps * 32, rb, xb, groups,
                                         is_quant(dtype));
        return static_cast<size_t>(L.total);
    }
    if (v.kind == KIND_BAND) return 0;  // x in registers, static shared memory only
    if (v.kind == KIND_MMA) return 0;  // x in registers, static shared memory only
    if (v.kind == KIND_SBAND || v.kind == KIND_SMMA) {
        const StageBandLayout L = stageband_layout(v.stages, v.rows_per_group, v.warps, v.tile_rows,
                                                   row_bytes_of(dtype, N), groups, is_quant(dtype));
        return static_cast<size_t>(L.total);
    }
    if (v.xmode == XMODE_BULK || v.xmode == XMODE_VEC)
        return static_cast<size_t>(v.x_offset) + static_cast<size_t>(N) * x_elem_bytes(dtype);
    if (v.kind == KIND_TILE) return static_cast<size_t>(v.x_offset);
    return 0;
}

// Can variant v serve this call?
bool variant_fits(const Variant &v, const DeviceState &d, int dtype, const void *A, const void *x,
                  int64_t M, int64_t N, const uint16_t *scales, int smode = SCALES_GROUP128)
{
    const int64_t groups = scale_groups(N, smode);
    if (v.xmode == XMODE_ELEM) {
        const int64_t blocks = (M + v.warps - 1) / v.warps;
        return blocks <= INT_MAX;
    }
    const int64_t rb = row_bytes_of(dtype, N);
    if (rb % 16 || !aligned(A, 16) || !aligned(x, 16)) return false;
    if (rb / 16 > INT_MAX / 64) return false;
    if (static_cast<int64_t>(smem_bytes(v, dtype, N, groups)) > d.max_smem) return false;
    if (v.kind == KIND_BULK) {
        // a fixed chunk count per consumer thread must match the row exactly
        if (v.unroll > 0 && rb / 16 != static_cast<int64_t>(v.unroll) * v.lanes_per_row) return false;
        // one stage (rows + their scales) is one transaction count of an mbarrier
        const int64_t g = groups;
        const bool quant = is_quant(dtype);
        // staged scales: one bulk copy per stage; one scale per row: read directly
        if (quant && g > 1 && ((2 * g) % 16 || !aligned(scales, 16))) return false;
        const int64_t tx = v.rows_per_group * (rb + (quant ? 2 * g : 0));
        if (tx >= (1 << 20)) return false;
        return true;  // persistent grid
    }
    if (v.kind == KIND_BAND) {
        // every thread takes exactly `unroll` chunks of each row
        return rb / 16 == static_cast<int64_t>(v.lanes_per_row) * v.unroll;  // persistent grid
    }
    if (v.kind == KIND_MMA) {
        // every warp takes exactly `unroll` steps of 512 bytes of each row; the
        // first INT4 layout reads the scales of two neighbouring groups as one
        // 4-byte word
        if (!aligned(scales, v.scale_align)) return false;
        return is_quant(dtype) && rb == static_cast<int64_t>(v.warps) * v.unroll * 512;  // persistent grid
    }
    if (v.kind == KIND_SMMA) {
        if (!is_quant(dtype) || rb != static_cast<int64_t>(v.warps) * v.unroll * 512) return false;
        // a tile's scales are one bulk copy: rows of scales a multiple of 16 bytes
        if ((2 * groups) % 16 || !aligned(scales, 16)) return false;
        const int64_t tx = v.tile_rows * (rb + 2 * groups);
        return tx < (1 << 20);  // persistent grid
    }
    if (v.kind == KIND_SBAND) {
        if (rb / 16 != static_cast<int64_t>(v.lanes_per_row) * v.unroll) return false;
        // a tile's scales are one bulk copy: 16-byte aligned rows of scales
        if (is_quant(dtype) && ((2 * groups) % 16 || !aligned(scales, 16))) return false;
        // one stage is one transaction count of an mbarrier
        const int64_t tx = v.tile_rows * (rb + (is_quant(dtype) ? 2 * groups : 0));
        return tx < (1 << 20);  // persistent grid
    }
    if (v.kind == KIND_TILE) {
        // every row must be covered by one request per thread
        if (rb / 16 > static_cast<int64_t>(v.lanes_per_row) * v.unroll) return false;
        return true;  // persistent grid: the block count never exceeds the SM slots
    }
    const int64_t blocks = (M + v.rows_per_block() - 1) / v.rows_per_block();
    return blocks <= INT_MAX;
}

// Blocks of a tile variant that fit on the GPU at once (0 on failure).
int resident_blocks(DeviceState &d, int dtype, int vid, const Variant &v, size_t smem)
{
    const auto key = std::make_tuple(dtype, vid, smem);
    {
        std::lock_guard<std::mutex> g(d.occ_mutex);
        auto it = d.occ.find(key);
        if (it != d.occ.end()) return it->second;
    }
    int per_sm = 0;
    const cudaError_t e = v.occupancy(&per_sm, smem);
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return 0;
    }
    if (v.max_blocks_per_sm > 0 && per_sm > v.max_blocks_per_sm) per_sm = v.max_blocks_per_sm;
    const int total = per_sm * d.sm_count;
    std::lock_guard<std::mutex> g(d.occ_mutex);
    d.occ[key] = total;
    return total;
}

int find_variant(int dtype, int lpr, int xmode, int kind = KIND_VEC, int warps = 0, int unroll = 0)
{
    int n = 0;
    const Variant *v = table(dtype, &n);
    for (int k = 0; k < n; ++k)
        if (v[k].lanes_per_row == lpr && v[k].xmode == xmode && v[k].kind == kind &&
            (warps == 0 || v[k].warps == warps) && (unroll == 0 || v[k].unroll == unroll))
            return k;
    return -1;
}

// The automatic choice (measured on GB300 over the workload families):
// - layouts the vector kernels cannot take: element-wise kernel;
// - FP32 and FP16 rows that a row-band variant covers exactly (x in
//   registers): the first such variant in table order (measured best first;
//   variants with a capped grid only for matrices up to 16 MB);
// - INT8, and INT4 rows of at least 4 KB: the bulk-copy pipeline, with
//   8-16 KB of rows per stage;
// - otherwise row tiles with the narrowest group that requests a whole row at
//   once: FP32/FP16 rows of 2-16 KB in 128-thread blocks with x through L1;
//   otherwise 256-thread blocks, x through L1 for groups of 128 threads or
//   more, in shared memory below that and for an FP32 x of FP16 weights;
// - rows too long for a tile, or x too long for shared memory: warp per row
//   with a rolling buffer.
int choose_variant(const DeviceState &d, int dtype, const void *A, const void *x, int64_t M,
                   int64_t N, const uint16_t *scales, int smode = SCALES_GROUP128)
{
    int n = 0;
    const Variant *v = table(dtype, &n);
    const int64_t rb = row_bytes_of(dtype, N);
    const bool vec_ok = rb % 16 == 0 && aligned(A, 16) && aligned(x, 16);
    if (!vec_ok) return find_variant(dtype, 32, XMODE_ELEM, KIND_ELEM);
    const int64_t chunks = rb / 16;
    const bool small_x = N * x_elem_bytes(dtype) <= kAutoSmemX;
    if (dtype == DT_F32 || dtype == DT_F16 || dtype == DT_F16X32) {
        for (int k = 0; k < n; ++k) {
            // a capped grid only for small matrices, where the next launch's
            // blocks starting beside it matter more than bytes in flight
            if (v[k].max_blocks_per_sm > 0 && M * rb > kSmallMatrixBytes) continue;
            if (v[k].kind == KIND_BAND && variant_fits(v[k], d, dtype, A, x, M, N, scales, smode)) return k;
        }
    }
    // the quantised types are bound by instruction issue: a row band or a
    // bulk-copy pipeline specialised for exactly this row length comes first,
    // in table order (measured best first); otherwise the general pipelines
    // for INT8 and for INT4 rows of 4 KB or more, and row tiles for shorter
    // INT4 rows
    if ((dtype == DT_Q8 || dtype == DT_Q4) && small_x) {
        for (int k = 0; k < n; ++k) {
            if ((v[k].kind == KIND_MMA || v[k].kind == KIND_SMMA || v[k].kind == KIND_BAND ||
                 (v[k].kind == KIND_BULK && v[k].unroll > 0)) &&
                variant_fits(v[k], d, dtype, A, x, M, N, scales, smode))
                return k;
        }
    }
    if ((dtype == DT_Q8 || (dtype == DT_Q4 && rb >= 4096)) && small_x) {
        int rs = 1;
        while (rs < 8 && 2 * rs * rb <= 16 * 1024) rs *= 2;
        // consumer warps: INT8 with four rows per stage takes four (more chunks
        // each); INT4 takes seven when 224 consumers split the row's chunks more
        // evenly than 256 (every consumer then takes the same number of chunks;
        // measured +9 % at 14336 columns, within noise for INT8)
        int warps = 8;
        if (dtype == DT_Q8 && rs == 4)
            warps = 4;
        else if (dtype == DT_Q4 && (chunks + 223) / 224 * 224 < (chunks + 255) / 256 * 256)
            warps = 7;
        for (int attempt = 0; attempt < 2; ++attempt, warps = 8) {
            for (int k = 0; k < n; ++k) {
                if (v[k].kind == KIND_BULK && v[k].rows_per_group == rs && v[k].warps == warps &&
                    v[k].unroll == 0 && variant_fits(v[k], d, dtype, A, x, M, N, scales, smode))
                    return k;
            }
        }
    }
    if (small_x && chunks <= static_cast<int64_t>(kTileMaxThreads) * kTileChunks) {
        int g = 1;
        while (static_cast<int64_t>(g) * kTileChunks < chunks) g *= 2;
        const int warps = g > 256 ? g / 32 : 8;
        const bool via_l1 = (dtype == DT_F32 || dtype == DT_F16) && g >= 128;
        if ((dtype == DT_F32 || dtype == DT_F16) && g >= 32 && g <= 128) {
            // rows of 2-16 KB: 128-thread blocks (finer tiles, more blocks per
            // SM) with x through L1 (measured +5-18 % on 1024-8192 columns);
            // rows of 4-8 KB as one row per block with four chunks per thread
            int k = g == 64 ? find_variant(dtype, 128, XMODE_L1, KIND_TILE, 4, 4) : -1;
            if (k < 0 || !variant_fits(v[k], d, dtype, A, x, M, N, scales, smode))
                k = find_variant(dtype, g, XMODE_L1, KIND_TILE, 4, kTileChunks);
            if (k >= 0 && variant_fits(v[k], d, dtype, A, x, M, N, scales, smode)) return k;
        }
        if (dtype == DT_Q4 && g == 16) {
            // INT4 rows of 1-2 KB: one row per 128-thread block, four chunks per
            // thread (measured +6 % at 4096 columns)
            const int k = find_variant(dtype, 32, XMODE_BULK, KIND_TILE, 4, 4);
            if (k >= 0 && variant_fits(v[k], d, dtype, A, x, M, N, scales, smode)) return k;
        }
        int k = find_variant(dtype, g, via_l1 ? XMODE_L1 : XMODE_BULK, KIND_TILE, warps);
        if (k >= 0 && variant_fits(v[k], d, dtype, A, x, M, N, scales, smode)) return k;
        k = find_variant(dtype, g, XMODE_BULK, KIND_TILE, warps);
        if (k >= 0 && variant_fits(v[k], d, dtype, A, x, M, N, scales, smode)) return k;
    }
    int k = small_x ? find_variant(dtype, 32, XMODE_BULK) : find_variant(dtype, 32, XMODE_L1);
    if (k < 0 || !variant_fits(v[k], d, dtype, A, x, M, N, scales, smode))
        k = find_variant(dtype, 32, XMODE_ELEM, KIND_ELEM);
    return k;
}

gemv_status_t run(int dtype, int vid, const void *A, const void *x, float *y, int64_t M, int64_t N,
                  const uint16_t *scales, void *stream, unsigned flags = 0, int smode = SCALES_GROUP128)
{
    gemv_status_t st = validate(dtype, A, x, y, M, N, scales);
    if (st != GEMV_OK) return st;
    int n = 0;
    const Variant *tab = table(dtype, &n);
    if (vid >= n) return GEMV_ERR_INVALID_VALUE;
    if (M == 0) return GEMV_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        launch_fill_zero(y, M, s);
        const cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
    }
    DeviceState *d = current_device();
    if (!d) return GEMV_ERR_CUDA;
    if (vid < 0) {
        vid = choose_variant(*d, dtype, A, x, M, N, scales, smode);
        if (vid < 0) return GEMV_ERR_UNSUPPORTED;
    }
    const Variant &v = tab[vid];
    if (!variant_fits(v, *d, dtype, A, x, M, N, scales, smode)) return GEMV_ERR_UNSUPPORTED;

    GemvArgs a{};
    a.A = A;
    a.x = x;
    a.y = y;
    a.scales = scales;
    a.M = M;
    a.N = N;
    a.row_bytes = row_bytes_of(dtype, N);
    a.groups = scale_groups(N, smode);
    {
        // chunk / column -> scale group: c >> scale_shift, j >> scale_elem_shift
        const int epc = dtype == DT_Q4 ? 32 : dtype == DT_Q8 ? 16 : 8;
        int lg = 0;
        while ((1 << lg) < kGroup / epc) ++lg;
        a.scale_shift = smode == SCALES_PER_ROW ? 30 : lg;
        a.scale_elem_shift = smode == SCALES_PER_ROW ? 62 : 7;
    }
    a.nchunks = static_cast<int>(a.row_bytes / 16);
    a.err = d->status;
    a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    a.skip_copies = g_skip_copies.load(std::memory_order_relaxed);
    a.pdl = ((flags & GEMV_FLAG_OVERLAP_PRECEDING) && v.supports_pdl()) ? 1 : 0;

    int64_t blocks;
    const size_t smem = smem_bytes(v, dtype, N, a.groups);
    if (v.xmode == XMODE_ELEM) {
        blocks = (M + v.warps - 1) / v.warps;
    } else {
        blocks = (M + v.rows_per_block() - 1) / v.rows_per_block();
        if (v.kind == KIND_TILE || v.kind == KIND_BULK || v.kind == KIND_BAND || v.kind == KIND_SBAND ||
            v.kind == KIND_MMA || v.kind == KIND_SMMA) {
            const int resident = resident_blocks(*d, dtype, vid, v, smem);
            if (resident <= 0) return GEMV_ERR_CUDA;
            if (blocks > resident) blocks = resident;
        }
    }
    // the kernel families that support it are always launched with
    // programmatic serialisation; without the flag they wait for the
    // preceding kernel before touching memory (same ordering as a plain launch)
    v.launch(a, static_cast<unsigned>(blocks), smem, s, v.supports_pdl());
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

}  // namespace
}  // namespace mbg

using namespace mbg;

extern "C" {

gemv_status_t gemv_f32(const float *A, const float *x, float *y, int64_t M, int64_t N, void *stream)
{
    return run(DT_F32, -1, A, x, y, M, N, nullptr, stream);
}

gemv_status_t gemv_f16(const uint16_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                       void *stream)
{
    return run(DT_F16, -1, A, x, y, M, N, nullptr, stream);
}

gemv_status_t gemv_q8(const int8_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                      const uint16_t *scales, void *stream)
{
    return run(DT_Q8, -1, A, x, y, M, N, scales, stream);
}

gemv_status_t gemv_q4(const uint8_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                      const uint16_t *scales, void *stream)
{
    return run(DT_Q4, -1, A, x, y, M, N, scales, stream);
}

gemv_status_t gemv_f16_xf32(const uint16_t *A, const float *x, float *y, int64_t M, int64_t N,
                           void *stream)
{
    return run(DT_F16X32, -1, A, x, y, M, N, nullptr, stream);
}

gemv_status_t gemv_q8_rowscale(const int8_t *A, const uint16_t *x, float *y, int64_t M, int64_t N,
                               const uint16_t *row_scales, void *stream)
{
    return run(DT_Q8, -1, A, x, y, M, N, row_scales, stream, 0, SCALES_PER_ROW);
}

gemv_status_t gemv_q8_rowscale_ex(const int8_t *A, const uint16_t *x, float *y, int64_t M,
                                  int64_t N, const uint16_t *row_scales, unsigned flags,
                                  void *stream)
{
    if (flags & ~static_cast<unsigned>(GEMV_FLAG_OVERLAP_PRECEDING)) return GEMV_ERR_INVALID_VALUE;
    return run(DT_Q8, -1, A, x, y, M, N, row_scales, stream, flags, SCALES_PER_ROW);
}

// Address through which kernels reach p: page-locked host memory (and, when
// allow_device, device or managed memory); nullptr for anything else.
static void *device_view(const void *p, bool allow_device)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (at.type == cudaMemoryTypeHost) return at.devicePointer;
    if (allow_device && (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged))
        return const_cast<void *>(p);
    return nullptr;
}

gemv_status_t gemv_ex_host(int dtype, const void *A, const void *x_host, void *x_dev, float *y_host,
                           int64_t M, int64_t N, const uint16_t *scales, unsigned flags,
                           void *stream)
{
    if (flags & ~static_cast<unsigned>(GEMV_FLAG_OVERLAP_PRECEDING)) return GEMV_ERR_INVALID_VALUE;
    gemv_status_t st = validate(dtype, A, x_dev, y_host, M, N, scales);
    if (st != GEMV_OK || M == 0) return st;
    float *y = static_cast<float *>(device_view(y_host, true));
    if (!y) return GEMV_ERR_INVALID_VALUE;
    if (N == 0) return run(dtype, -1, A, x_dev, y, M, N, scales, stream);
    if (!x_host) return GEMV_ERR_INVALID_VALUE;
    if (!aligned(x_host, x_align(dtype))) return GEMV_ERR_MISALIGNED;
    const void *xh = device_view(x_host, false);
    if (!xh) return GEMV_ERR_INVALID_VALUE;
    if (!current_device()) return GEMV_ERR_CUDA;
    launch_copy_in(xh, x_dev, N * x_elem_bytes(dtype), (flags & GEMV_FLAG_OVERLAP_PRECEDING) != 0,
                   static_cast<cudaStream_t>(stream));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, GEMV_ERR_LAUNCH);
    // the GEMV waits for the copy (griddepcontrol.wait) before it reads x;
    // it streams weights before that wait only under the caller's promise
    // that the kernel before this call leaves them alone (the copy itself
    // never writes them)
    return run(dtype, -1, A, x_dev, y, M, N, scales, stream, flags);
}

gemv_status_t gemv_ex(int dtype, const void *A, const void *x, float *y, int64_t M, int64_t N,
                      const uint16_t *scales, unsigned flags, void *stream)
{
    if (flags & ~static_cast<unsigned>(GEMV_FLAG_OVERLAP_PRECEDING)) return GEMV_ERR_INVALID_VALUE;
    return run(dtype, -1, A, x, y, M, N, scales, stream, flags);
}

int gemv_variant_count(int dtype)
{
    int n = 0;
    table(dtype, &n);
    return n;
}

gemv_status_t gemv_variant_info(int dtype, int variant, gemv_variant_info_t *info)
{
    int n = 0;
    const Variant *v = table(dtype, &n);
    if (!info || variant < 0 || variant >= n) return GEMV_ERR_INVALID_VALUE;
    const Variant &w = v[variant];
    info->dtype = w.dtype;
    info->kind = w.kind;
    info->threads_per_row = w.lanes_per_row;
    info->rows_per_group = w.rows_per_group;
    info->unroll = w.unroll;
    info->warps = w.warps;
    info->math = w.math;
    info->xmode = w.xmode;
    snprintf(info->name, sizeof(info->name), "%s", w.name);
    return GEMV_OK;
}

static int select_variant(int dtype, const void *A, const void *x, int64_t M, int64_t N, int smode)
{
    if (dtype < 0 || dtype >= DT_COUNT || M <= 0 || N <= 0 || !A || !x) return -1;
    if (dtype == DT_Q4 && (N % 2)) return -1;
    if (!aligned(A, a_align(dtype)) || !aligned(x, x_align(dtype))) return -1;
    DeviceState *d = current_device();
    if (!d) return -1;
    return choose_variant(*d, dtype, A, x, M, N, nullptr, smode);
}

int gemv_select_variant(int dtype, const void *A, const void *x, int64_t M, int64_t N)
{
    return select_variant(dtype, A, x, M, N, SCALES_GROUP128);
}

int gemv_q8_rowscale_select_variant(const int8_t *A, const uint16_t *x, int64_t M, int64_t N)
{
    return select_variant(DT_Q8, A, x, M, N, SCALES_PER_ROW);
}

gemv_status_t gemv_q8_rowscale_run_variant(int variant, const int8_t *A, const uint16_t *x, float *y,
                                           int64_t M, int64_t N, const uint16_t *row_scales,
                                           void *stream)
{
    if (variant < 0) return GEMV_ERR_INVALID_VALUE;
    return run(DT_Q8, variant, A, x, y, M, N, row_scales, stream, 0, SCALES_PER_ROW);
}

gemv_status_t gemv_run_variant(int dtype, int variant, const void *A, const void *x, float *y,
                               int64_t M, int64_t N, const uint16_t *scales, void *stream)
{
    if (variant < 0) return GEMV_ERR_INVALID_VALUE;
    return run(dtype, variant, A, x, y, M, N, scales, stream);
}

gemv_status_t gemv_run_variant_ex(int dtype, int variant, const void *A, const void *x, float *y,
                                  int64_t M, int64_t N, const uint16_t *scales, unsigned flags,
                                  void *stream)
{
    if (variant < 0) return GEMV_ERR_INVALID_VALUE;
    if (flags & ~static_cast<unsigned>(GEMV_FLAG_OVERLAP_PRECEDING)) return GEMV_ERR_INVALID_VALUE;
    return run(dtype, variant, A, x, y, M, N, scales, stream, flags);
}

gemv_status_t gemv_probe_read(const void *buf, size_t bytes, unsigned long long *sink, int variant,
                              void *stream)
{
    int n = 0;
    const ProbeVariant *pv = probe_variants(&n);
    if (variant < 0 || variant >= n || !sink) return GEMV_ERR_INVALID_VALUE;
    if (bytes == 0) return GEMV_OK;
    if (!buf) return GEMV_ERR_INVALID_VALUE;
    if (bytes % 16 || !aligned(buf, 16) || !aligned(sink, 8)) return GEMV_ERR_MISALIGNED;
    DeviceState *d = current_device();
    if (!d) return GEMV_ERR_CUDA;
    const ProbeVariant &p = pv[variant];
    const unsigned grid = static_cast<unsigned>(d->sm_count * p.blocks_per_sm);
    p.launch(buf, bytes / 16, sink, grid, g_wait_limit_ns.load(std::memory_order_relaxed),
             (g_skip_copies.load(std::memory_order_relaxed) & SKIP_PROBE) != 0,
             static_cast<cudaStream_t>(stream));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

int gemv_probe_variant_count(void)
{
    int n = 0;
    probe_variants(&n);
    return n;
}

const char *gemv_probe_variant_name(int variant)
{
    int n = 0;
    const ProbeVariant *pv = probe_variants(&n);
    return (variant >= 0 && variant < n) ? pv[variant].name : nullptr;
}

static gemv_status_t dequant(int dtype, const void *A, const uint16_t *scales, float *W, int64_t M,
                             int64_t N, void *stream)
{
    if (M < 0 || N < 0) return GEMV_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMV_OK;
    if (!A || !scales || !W) return GEMV_ERR_INVALID_VALUE;
    if (dtype == DT_Q4 && (N % 2)) return GEMV_ERR_UNSUPPORTED;
    if (!aligned(scales, 2) || !aligned(W, 4)) return GEMV_ERR_MISALIGNED;
    if (M > INT64_MAX / N) return GEMV_ERR_UNSUPPORTED;
    const int64_t rb = row_bytes_of(dtype, N);
    const bool vec = rb % 16 == 0 && aligned(A, 16);
    launch_dequant(dtype, A, scales, W, M, N, vec, static_cast<cudaStream_t>(stream));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

static gemv_status_t quantize(int bits, bool per_row, const void *W, int w_dtype, void *A,
                              uint16_t *scales, int64_t M, int64_t N, double *sq_err, void *stream)
{
    if (M < 0 || N < 0) return GEMV_ERR_INVALID_VALUE;
    if (w_dtype != DT_F32 && w_dtype != DT_F16) return GEMV_ERR_INVALID_VALUE;
    if (bits == 4 && (N % 2)) return GEMV_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return GEMV_OK;
    if (!W || !A || !scales) return GEMV_ERR_INVALID_VALUE;
    if (!aligned(W, w_dtype == DT_F32 ? 4 : 2) || !aligned(scales, 2) ||
        (sq_err && !aligned(sq_err, 8)))
        return GEMV_ERR_MISALIGNED;
    if (M > INT64_MAX / (4 * N)) return GEMV_ERR_UNSUPPORTED;
    DeviceState *d = current_device();
    if (!d) return GEMV_ERR_CUDA;
    launch_quantize(bits, per_row, w_dtype == DT_F16, W, A, scales, sq_err, M, N, d->sm_count,
                    static_cast<cudaStream_t>(stream));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

gemv_status_t gemv_quantize_q8(const void *W, int w_dtype, int8_t *A, uint16_t *scales, int64_t M,
                               int64_t N, int per_row, double *sq_err, void *stream)
{
    return quantize(8, per_row != 0, W, w_dtype, A, scales, M, N, sq_err, stream);
}

gemv_status_t gemv_quantize_q4(const void *W, int w_dtype, uint8_t *A, uint16_t *scales, int64_t M,
                               int64_t N, double *sq_err, void *stream)
{
    return quantize(4, false, W, w_dtype, A, scales, M, N, sq_err, stream);
}

gemv_status_t gemv_dequant_q8(const int8_t *A, const uint16_t *scales, float *W, int64_t M,
                              int64_t N, void *stream)
{
    return dequant(DT_Q8, A, scales, W, M, N, stream);
}

gemv_status_t gemv_dequant_q4(const uint8_t *A, const uint16_t *scales, float *W, int64_t M,
                              int64_t N, void *stream)
{
    return dequant(DT_Q4, A, scales, W, M, N, stream);
}

static gemv_status_t softmax_run(const uint16_t *x, uint16_t *y, int64_t M, int64_t N, int variant,
                                 void *stream)
{
    if (M < 0 || N < 0) return GEMV_ERR_INVALID_VALUE;
    if (variant >= softmax_variant_count()) return GEMV_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMV_OK;
    if (!x || !y) return GEMV_ERR_INVALID_VALUE;
    if (!aligned(x, 2) || !aligned(y, 2)) return GEMV_ERR_MISALIGNED;
    if (M > INT64_MAX / N) return GEMV_ERR_UNSUPPORTED;
    DeviceState *d = current_device();
    if (!d) return GEMV_ERR_CUDA;
    const cudaError_t e = launch_softmax(x, y, M, N, variant, d->status,
                                         g_wait_limit_ns.load(std::memory_order_relaxed),
                                         g_skip_copies.load(std::memory_order_relaxed),
                                         static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return GEMV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

gemv_status_t gemv_softmax_f16(const uint16_t *x, uint16_t *y, int64_t M, int64_t N, void *stream)
{
    return softmax_run(x, y, M, N, -1, stream);
}

gemv_status_t gemv_softmax_run_variant(int variant, const uint16_t *x, uint16_t *y, int64_t M,
                                       int64_t N, void *stream)
{
    if (variant < 0) return GEMV_ERR_INVALID_VALUE;
    return softmax_run(x, y, M, N, variant, stream);
}

int gemv_softmax_variant_count(void) { return softmax_variant_count(); }
const char *gemv_softmax_variant_name(int variant) { return softmax_variant_name(variant); }

gemv_status_t gemv_probe_copy(const void *src, void *dst, size_t bytes, int variant, void *stream)
{
    if (variant < 0 || variant >= copy_variant_count()) return GEMV_ERR_INVALID_VALUE;
    if (bytes == 0) return GEMV_OK;
    if (!src || !dst) return GEMV_ERR_INVALID_VALUE;
    if (bytes % 16 || !aligned(src, 16) || !aligned(dst, 16)) return GEMV_ERR_MISALIGNED;
    DeviceState *d = current_device();
    if (!d) return GEMV_ERR_CUDA;
    const cudaError_t e = launch_copy_probe(src, dst, bytes, variant, d->sm_count,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

int gemv_probe_copy_variant_count(void) { return copy_variant_count(); }
const char *gemv_probe_copy_variant_name(int variant) { return copy_variant_name(variant); }

gemv_status_t gemv_get_device_error(void *stream)
{
    DeviceState *d = current_device();
    if (!d) return GEMV_ERR_CUDA;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, GEMV_ERR_CUDA);
    unsigned int word = 0;
    e = cudaMemcpy(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, GEMV_ERR_CUDA);
    if (word) {
        const unsigned int zero = 0;
        e = cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, GEMV_ERR_CUDA);
    }
    if (word & DEVERR_UNDRAINED) return GEMV_ERR_TIMEOUT_UNDRAINED;
    return (word & DEVERR_TIMEOUT) ? GEMV_ERR_TIMEOUT : GEMV_OK;
}

void gemv_debug_set_wait_limit_ns(uint64_t ns)
{
    // 0 restores the default; anything shorter than 100 us is raised to it so
    // that a copy that was issued always has time to land before its block
    // exits.
    if (ns == 0) ns = 1000000000ull;
    if (ns < 100000ull) ns = 100000ull;
    g_wait_limit_ns.store(ns, std::memory_order_relaxed);
}

void gemv_debug_skip_x_copy(int on)
{
    if (on) g_skip_copies.fetch_or(SKIP_X, std::memory_order_relaxed);
    else g_skip_copies.fetch_and(~static_cast<unsigned int>(SKIP_X), std::memory_order_relaxed);
}

gemv_status_t gemv_debug_late_fill(void *dst, size_t bytes, uint32_t word, uint64_t delay_ns, void *stream)
{
    if (bytes == 0) return GEMV_OK;
    if (!dst) return GEMV_ERR_INVALID_VALUE;
    if (bytes % 4 || !aligned(dst, 4)) return GEMV_ERR_MISALIGNED;
    if (delay_ns > 1000000000ull) delay_ns = 1000000000ull;
    if (!current_device()) return GEMV_ERR_CUDA;
    launch_late_fill(dst, bytes, word, delay_ns, static_cast<cudaStream_t>(stream));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GEMV_OK : cuda_fail(e, GEMV_ERR_LAUNCH);
}

void gemv_debug_skip_copies(unsigned int mask)
{
    g_skip_copies.store(mask & (SKIP_X | SKIP_STAGE | SKIP_SEGMENT | SKIP_PROBE), std::memory_order_relaxed);
}

const char *gemv_status_string(gemv_status_t status)
{
    switch (status) {
    case GEMV_OK: return "GEMV_OK";
    case GEMV_ERR_INVALID_VALUE: return "GEMV_ERR_INVALID_VALUE";
    case GEMV_ERR_MISALIGNED: return "GEMV_ERR_MISALIGNED";
    case GEMV_ERR_UNSUPPORTED: return "GEMV_ERR_UNSUPPORTED";
    case GEMV_ERR_LAUNCH: return "GEMV_ERR_LAUNCH";
    case GEMV_ERR_TIMEOUT: return "GEMV_ERR_TIMEOUT";
    case GEMV_ERR_CUDA: return "GEMV_ERR_CUDA";
    case GEMV_ERR_TIMEOUT_UNDRAINED: return "GEMV_ERR_TIMEOUT_UNDRAINED";
    default: return "GEMV_ERR_UNKNOWN";
    }
}

int gemv_last_cuda_error(void) { return t_last_cuda_error; }

const char *gemv_build_info(void)
{
    return "memory_bound_gemv_gb300: sm_103a, CUDA " MBG_STR(CUDART_VERSION);
}

}  // extern "C"
