// GEMV kernel templates (sm_103a).
//
// mbg_warprow_kernel: the vectorised path.  A lane group of LPR lanes owns RPW
// consecutive rows; lane t of the group streams the 16-byte chunks
// t, t+LPR, t+2*LPR, ... of each of those rows, so with LPR = 32 a warp reads
// 512 contiguous bytes of a row per step ("cuda-gemv-optimization", kernel 4;
// "Making GEMV Fast", section "Turning that access pattern into code";
// "membound", kernel "vec").  Short rows use LPR < 32 so that one warp serves
// several rows at once.  U chunks per row and lane are kept in flight in a
// rolling register buffer: the load of chunk c + U*LPR is issued before
// chunk c is consumed.  x is staged once per block in shared memory (one bulk
// async copy tracked by an mbarrier, or cooperative vector loads), or read
// through L1; the first U chunks of A are requested before x is waited for,
// so the copy of x overlaps the first DRAM round trip.  Lane partials are
// combined with an XOR butterfly inside the group and one lane stores y.
//
// mbg_elem_kernel: element-wise path for layouts the vector path cannot take
// (unaligned pointers or a row pitch that is not a multiple of 16 bytes).
#pragma once

#include "gemv_device.cuh"
#include <type_traits>

namespace mbg {

template <int DT, int LPR, int RPW, int U, int WARPS, int XMODE>
__global__ void __launch_bounds__(WARPS * 32) mbg_warprow_kernel(const GemvArgs p)
{
    using F = Fmt<DT>;
    constexpr int EPC = F::EPC;
    constexpr int XCB = x_chunk_bytes<DT>();
    constexpr int XV = x_chunk_vecs<DT>();
    constexpr int GPW = 32 / LPR;
    constexpr int ROWS_PER_WARP = GPW * RPW;
    constexpr int ROWS_PER_BLOCK = WARPS * ROWS_PER_WARP;
    static_assert(32 % LPR == 0, "lanes per row must divide the warp");
    static_assert(XMODE == XMODE_BULK || XMODE == XMODE_VEC || XMODE == XMODE_L1, "xmode");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    unsigned char *xs = smem + 16;

    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = lane % LPR;
    const int64_t row_base = static_cast<int64_t>(blockIdx.x) * ROWS_PER_BLOCK +
                             static_cast<int64_t>(warp) * ROWS_PER_WARP + (lane / LPR) * RPW;
    const int nchunks = p.nchunks;
    const uint32_t xbytes = static_cast<uint32_t>(nchunks) * XCB;

    // x staging: one bulk copy when x is in its own order in shared memory
    // (one vector per chunk), a cooperative transposing load otherwise.
    constexpr bool XBULK = XMODE == XMODE_BULK && XV == 1;
    constexpr bool XCOOP = (XMODE == XMODE_BULK && XV > 1) || XMODE == XMODE_VEC;
    if constexpr (XBULK) {
        if (threadIdx.x == 0) {
            const uint32_t b = smem_addr(bar);
            mbar_init(b, 1);
            mbar_arrive_expect_tx(b, xbytes);
            if (!(p.skip_copies & SKIP_X)) bulk_copy_g2s(smem_addr(xs), p.x, xbytes, b);
        }
    }

    // Rows of this lane group (clamped to the last row; results of clamped
    // rows are discarded) and the first U chunks of each.
    const bool active = row_base < p.M;
    const int my_chunks = active ? nchunks : 0;
    const unsigned char *rowp[RPW];
    const uint16_t *srow[RPW];
    bool rvalid[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t row = row_base + r;
        rvalid[r] = row < p.M;
        const int64_t rr = row < p.M ? row : p.M - 1;
        rowp[r] = static_cast<const unsigned char *>(p.A) + rr * p.row_bytes;
        srow[r] = F::QUANT ? p.scales + rr * p.groups : nullptr;
    }

    uint4 buf[RPW][U];
    float sbuf[RPW][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = t + u * LPR;
        if (c < my_chunks) {
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                buf[r][u] = ld_stream16(rowp[r] + static_cast<size_t>(c) * 16);
                if constexpr (F::QUANT) sbuf[r][u] = ld_half_as_float(srow[r] + (c >> p.scale_shift));
                else sbuf[r][u] = 0.f;
            }
        }
    }

    if constexpr (XCOOP) stage_x_vmajor<DT>(xs, p.x, nchunks, threadIdx.x, WARPS * 32);
    if constexpr (XMODE == XMODE_BULK || XMODE == XMODE_VEC) __syncthreads();
    if constexpr (XBULK) {
        if (!mbar_wait_bounded(smem_addr(bar), 0, p.wait_limit_ns)) {
            if (threadIdx.x == 0) report_error(p.err, DEVERR_TIMEOUT);
            // A copy that was issued may still land: give it one more bounded
            // wait before the block's shared memory is released.
            if (!(p.skip_copies & SKIP_X) && !mbar_wait_bounded(smem_addr(bar), 0, p.wait_limit_ns))
                report_error(p.err, DEVERR_UNDRAINED);
            return;
        }
    }

    const unsigned char *xsrc =
        (XMODE == XMODE_L1) ? static_cast<const unsigned char *>(p.x) : xs;

    float acc[RPW][NACC];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int k = 0; k < NACC; ++k) acc[r][k] = 0.f;

    for (int c0 = t; c0 < my_chunks; c0 += LPR * U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * LPR;
            if (c < my_chunks) {
                uint4 xv[XV];
#pragma unroll
                for (int v = 0; v < XV; ++v) {
                    if constexpr (XMODE == XMODE_L1)
                        xv[v] = ld_cached16(xsrc + static_cast<size_t>(c) * XCB + 16 * v);
                    else
                        xv[v] = *x_smem_vec(xsrc, nchunks, c, v);
                }
                float xf[EPC];
                x_to_float<DT>(xv, xf);

                uint4 cur[RPW];
                float sc[RPW];
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    cur[r] = buf[r][u];
                    sc[r] = sbuf[r][u];
                }
                const int cn = c + LPR * U;
                if (cn < my_chunks) {
#pragma unroll
                    for (int r = 0; r < RPW; ++r) {
                        buf[r][u] = ld_stream16(rowp[r] + static_cast<size_t>(cn) * 16);
                        if constexpr (F::QUANT)
                            sbuf[r][u] = ld_half_as_float(srow[r] + (cn >> p.scale_shift));
                    }
                }
#pragma unroll
                for (int r = 0; r < RPW; ++r) {
                    float wf[EPC];
                    chunk_to_float<DT>(cur[r], wf);
                    chunk_fma<DT>(wf, xf, sc[r], acc[r]);
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        float s = (acc[r][0] + acc[r][1]) + (acc[r][2] + acc[r][3]);
        s = group_sum<LPR>(s);
        if (t == (r % LPR) && rvalid[r]) p.y[row_base + r] = s;
    }
}

// ---------------------------------------------------------------------------
// Row-tile kernel
// ---------------------------------------------------------------------------
//
// G threads share one row and request all of it at once: thread g of the
// group loads chunks g, g+G, ..., g+(CPT-1)*G (so G*CPT*16 bytes must cover
// the row).  A block of T threads holds T/G consecutive rows (a tile); the
// grid is persistent and walks tiles in grid-stride order, issuing the loads
// of its next tile before it reduces the current one.  At any moment the
// loads in flight therefore cover a dense band of consecutive rows, which is
// how HBM3e delivers its bandwidth (scattered per-warp streams reach far
// less).  Lane partials are summed with an XOR butterfly; groups wider than a
// warp combine their warps' partials through shared memory, one block barrier
// per batch of tiles (every thread of a block walks the same tiles)
// ("llama.cpp GEMV CUDA": a block-wide row with a warp reduction, warp sums
// in shared memory and a second warp reduction).
template <int DT, int G, int CPT, int T, int XMODE, int MATH>
__global__ void __launch_bounds__(T) mbg_rowtile_kernel(const GemvArgs p)
{
    using F = Fmt<DT>;
    constexpr int EPC = F::EPC;
    constexpr int XCB = x_chunk_bytes<DT>();
    constexpr int XV = x_chunk_vecs<DT>();
    constexpr int RT = T / G;                       // rows per tile
    constexpr bool WIDE = G > 32;                   // group spans several warps
    constexpr int GW = WIDE ? G / 32 : 1;           // warps per group
    constexpr int LW = WIDE ? 32 : G;               // shuffle width
    constexpr int NW = T / 32;
    constexpr int KB = kTileBatch;                  // tiles per deferred reduction
    constexpr int PART_BYTES = WIDE ? 2 * KB * NW * 4 : 0;
    constexpr int X_OFFSET = (16 + PART_BYTES + 15) / 16 * 16;
    static_assert(T % G == 0 && (G <= 32 ? 32 % G == 0 : G % 32 == 0), "group shape");
    static_assert(XMODE == XMODE_BULK || XMODE == XMODE_L1, "xmode");
    static_assert(MATH == MATH_F32 || Fmt<DT>::XB == 2, "an FP32 x uses FP32 math");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    float *part = reinterpret_cast<float *>(smem + 16);
    unsigned char *xs = smem + X_OFFSET;

    const int tid = threadIdx.x;
    const int grp = tid / G;
    const int tg = tid % G;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nchunks = p.nchunks;
    const int64_t ntiles = (p.M + RT - 1) / RT;
    const uint32_t xbytes = static_cast<uint32_t>(nchunks) * XCB;

    // x staging: one bulk copy when x is in its own order in shared memory
    // (one vector per chunk), a cooperative transposing load otherwise.
    constexpr bool XBULK = XMODE == XMODE_BULK && XV == 1;
    constexpr bool XCOOP = XMODE == XMODE_BULK && XV > 1;
    // INT4 x staged for the mixed-precision products: paired layout
    constexpr bool PAIRED = DT == DT_Q4 && MATH == MATH_MIXED && XCOOP;
    // The kernel is always launched with programmatic stream serialisation.
    // With p.pdl the first tile of weights is requested before waiting for
    // the preceding kernel (x is read and y written only after that wait);
    // without it the kernel waits before it touches any memory, so only its
    // scheduling overlaps the preceding kernel's drain.
    pdl_trigger();
    const bool pdl = p.pdl != 0;
    // this block's first two tiles into L2 while the preceding kernel drains
    // (a hint only: without p.pdl the loads of the tiles come after the wait;
    // measured: one tile +3-12 %, the second +6 % more at 4096x14336)
    for (int k = 0; k < 2; ++k) {
        const int64_t row0 = (static_cast<int64_t>(blockIdx.x) + k * static_cast<int64_t>(gridDim.x)) * RT + grp;
        if (tg == 0 && row0 < p.M)
            prefetch_l2(static_cast<const unsigned char *>(p.A) + row0 * p.row_bytes,
                        static_cast<uint32_t>(p.row_bytes));
    }
    if (!pdl) pdl_wait();
    auto stage_x_bulk = [&]() {
        if (tid == 0) {
            const uint32_t b = smem_addr(bar);
            mbar_init(b, 1);
            mbar_arrive_expect_tx(b, xbytes);
            if (!(p.skip_copies & SKIP_X)) bulk_copy_g2s(smem_addr(xs), p.x, xbytes, b);
        }
    };
    if constexpr (XBULK) {
        if (!pdl) stage_x_bulk();
    }

    uint4 cur[CPT], nxt[CPT];
    float scur[CPT], snxt[CPT];

    // Addresses: one row pointer per tile, then compile-time offsets k*G*16.
    auto load_tile = [&](int64_t tile, uint4 (&buf)[CPT], float (&sb)[CPT]) {
        const int64_t row = tile * RT + grp;
        if (row < p.M) {
            const unsigned char *rp =
                static_cast<const unsigned char *>(p.A) + row * p.row_bytes + tg * 16;
            const uint16_t *sp = F::QUANT ? p.scales + row * p.groups : nullptr;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                if (tg + k * G < nchunks) {
                    buf[k] = ld_stream16(rp + k * G * 16);
                    if constexpr (F::QUANT) sb[k] = ld_half_as_float(sp + ((tg + k * G) >> p.scale_shift));
                }
            }
        }
    };

    int64_t tile = blockIdx.x;
    if (tile < ntiles) load_tile(tile, cur, scur);
    if (pdl) {
        pdl_wait();
        if constexpr (XBULK) stage_x_bulk();
    }

    if constexpr (XCOOP) stage_x_vmajor<DT, PAIRED>(xs, p.x, nchunks, tid, T);
    if constexpr (XMODE == XMODE_BULK) __syncthreads();
    if constexpr (XBULK) {
        if (!mbar_wait_bounded(smem_addr(bar), 0, p.wait_limit_ns)) {
            if (tid == 0) report_error(p.err, DEVERR_TIMEOUT);
            if (!(p.skip_copies & SKIP_X) && !mbar_wait_bounded(smem_addr(bar), 0, p.wait_limit_ns))
                report_error(p.err, DEVERR_UNDRAINED);
            return;
        }
    }
    // x addresses of this thread's first chunk: global (through L1) or 32-bit
    // shared-space addresses of each vector-major x plane
    const unsigned char *xg = static_cast<const unsigned char *>(p.x) + tg * XCB;
    uint32_t xb[XV];
#pragma unroll
    for (int v = 0; v < XV; ++v)
        xb[v] = smem_addr(xs) + static_cast<uint32_t>(v) * static_cast<uint32_t>(nchunks) * 16u + tg * 16u;

    // Groups wider than a warp leave one partial per warp and tile in shared
    // memory; every KB tiles (kTileBatch) one block barrier makes a batch
    // visible and the warps finish those rows (two batch buffers alternate, so
    // the next batch can be written while the previous one is read).
    int half = 0, fill = 0;
    int64_t batch_tile0 = tile;
    auto flush = [&](int count) {
        __syncthreads();
        const float *pb = part + half * KB * NW;
        for (int e = warp; e < count * RT; e += NW) {
            const int k = e / RT, g = e - k * RT;
            const int64_t r = (batch_tile0 + static_cast<int64_t>(k) * gridDim.x) * RT + g;
            float v = lane < GW ? pb[k * NW + g * GW + lane] : 0.f;
            v = group_sum<32>(v);
            if (lane == 0 && r < p.M) p.y[r] = v;
        }
        half ^= 1;
        fill = 0;
    };

    const bool full_slots = tg + (CPT - 1) * G < nchunks;
    for (; tile < ntiles; tile += gridDim.x) {
        const int64_t next = tile + gridDim.x;
        if (next < ntiles) load_tile(next, nxt, snxt);

        const int64_t row = tile * RT + grp;
        const bool valid = row < p.M;
        float acc[NACC] = {0.f, 0.f, 0.f, 0.f};
        // FULL: every chunk slot of this thread lies inside the row (no checks)
        auto dot = [&](auto full) {
            constexpr bool FULL = decltype(full)::value;
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = tg + k * G;
                if (FULL || c < nchunks) {
                    uint4 xv[XV];
#pragma unroll
                    for (int v = 0; v < XV; ++v) {
                        if constexpr (XMODE == XMODE_L1)
                            xv[v] = ld_cached16(xg + k * G * XCB + 16 * v);
                        else
                            xv[v] = lds128(xb[v] + k * G * 16);
                    }
                    if constexpr (MATH == MATH_MIXED) {
                        chunk_dot_mixed<DT, PAIRED>(cur[k], xv, F::QUANT ? scur[k] : 0.f, acc);
                    } else {
                        float xf[EPC];
                        x_to_float<DT>(xv, xf);
                        float wf[EPC];
                        chunk_to_float<DT>(cur[k], wf);
                        chunk_fma<DT>(wf, xf, F::QUANT ? scur[k] : 0.f, acc);
                    }
                }
            }
        };
        if (valid) {
            // the check-free copy pays for the instruction-bound quantised
            // types; for the others the second copy only costs registers
            if constexpr (F::QUANT) {
                if (full_slots) dot(std::true_type{});
                else dot(std::false_type{});
            } else {
                dot(std::false_type{});
            }
        }
        float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        s = group_sum<LW>(s);
        if constexpr (WIDE) {
            if (fill == 0) batch_tile0 = tile;
            if (lane == 0) part[(half * KB + fill) * NW + warp] = s;
            if (++fill == KB) flush(KB);
        } else {
            if (tg == 0 && valid) p.y[row] = s;
        }
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            cur[k] = nxt[k];
            scur[k] = snxt[k];
        }
    }
    if constexpr (WIDE) {
        if (fill > 0) flush(fill);
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy pipeline kernel (warp-specialised)
// ---------------------------------------------------------------------------
//
// A tile of RS consecutive rows is one contiguous byte range of A, so one
// bulk async copy (cp.async.bulk, completion counted on an mbarrier) moves a
// whole tile into shared memory.  Each block of the persistent grid keeps S
// tiles in flight in a ring of stages: memory-level parallelism comes from
// the copy engine, not from registers, and the tiles in flight across the
// grid form one dense band of consecutive rows.
//
// Warp roles.  T/32 consumer warps wait on a stage's "full" barrier, read the
// tile from shared memory (thread t takes chunks t, t+T, ... of every row of
// the tile and loads each x chunk once for all RS rows), store one partial sum
// per thread and row, and arrive on the stage's "reduced" barrier.  One
// producer warp waits on "reduced", adds the partials of each row (a fixed
// order, then an XOR butterfly), writes y and refills the stage with the tile
// S positions ahead.  No block-wide barrier sits in the
// loop, so consumer warps never wait for one another.  Quantised tiles bring
// their rows' scales along in a second bulk copy on the same barrier.
//
// Every wait is bounded.  A thread whose wait gives up reports the status
// word and raises the block's abort flag; every warp then leaves its loop
// (each decision made warp-uniform first), and the producer first waits
// (bounded) for the copies it still has in flight, so no copy can land in
// shared memory after the block has exited.
// XR: with a fixed chunk count per consumer thread, consumer thread t only
// ever reads the x of chunks t, t + T, ...; XR keeps those vectors in its
// registers (loaded once), so x takes no shared memory and no staging barrier.
template <int DT, int T, int RS, int S, int MATH, int CF, bool XR>
__global__ void __launch_bounds__(T + 32) mbg_bulkpipe_kernel(const GemvArgs p)
{
    using F = Fmt<DT>;
    constexpr int XCB = x_chunk_bytes<DT>();
    constexpr int XV = x_chunk_vecs<DT>();
    constexpr int NW = T / 32;  // consumer warps
    static_assert(MATH == MATH_F32 || Fmt<DT>::XB == 2, "an FP32 x uses FP32 math");
    static_assert(NW <= 32, "the producer warp adds one partial per consumer warp");
    constexpr bool PAIRED = DT == DT_Q4 && MATH == MATH_MIXED;  // see stage_x_vmajor
    constexpr bool XREG = XR;
    static_assert(!XR || (CF > 0 && XV > 1), "x in registers: fixed chunk count, several x vectors");

    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunks = p.nchunks;
    const uint32_t xbytes = static_cast<uint32_t>(nchunks) * XCB;
    const BulkLayout L = bulk_layout(S, RS, T, p.row_bytes, XREG ? 0u : xbytes, p.groups, F::QUANT);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *red = full + S;
    uint64_t *xbar = red + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(xbar + 1);
    float *part = reinterpret_cast<float *>(smem + L.part);
    const unsigned char *xs = smem + L.x;
    const int64_t ntiles = (p.M + RS - 1) / RS;
    const int64_t grid = gridDim.x;
    // iterations of this block: tiles blockIdx.x, blockIdx.x + grid, ...
    const int64_t iters = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / grid + 1 : 0;

    auto issue = [&](int64_t it) {
        const int slot = static_cast<int>(it % S);
        const int64_t r0 = (blockIdx.x + it * grid) * RS;
        const int rows = static_cast<int>(min(static_cast<int64_t>(RS), p.M - r0));
        const uint32_t bytes = static_cast<uint32_t>(rows * p.row_bytes);
        const bool stage_scales = F::QUANT && p.groups > 1;
        const uint32_t sbytes = stage_scales ? static_cast<uint32_t>(rows * 2 * p.groups) : 0u;
        const uint32_t b = smem_addr(&full[slot]);
        mbar_arrive_expect_tx(b, bytes + sbytes);
        if (it == 0 && (p.skip_copies & SKIP_STAGE)) return;  // test hook: the wait must run out
        bulk_copy_g2s(smem_addr(smem + L.stage + slot * L.stage_bytes),
                      static_cast<const unsigned char *>(p.A) + r0 * p.row_bytes, bytes, b);
        if (stage_scales)
            bulk_copy_g2s(smem_addr(smem + L.scale + slot * L.scale_bytes), p.scales + r0 * p.groups,
                          sbytes, b);
    };
    auto fail = [&]() {
        report_error(p.err, DEVERR_TIMEOUT);
        *abort_flag = 1;
    };

    pdl_trigger();
    if (!p.pdl) {
        // the first tile into L2 while the preceding kernel drains (a hint
        // only; see the row-tile kernel).  Only the first: the x loads that
        // follow the wait would queue behind a larger burst (measured: S
        // tiles cost INT8 at 14336 columns 9 %, one tile gains 4-9 %)
        if (tid == 0 && iters > 0) {
            const int64_t r0 = static_cast<int64_t>(blockIdx.x) * RS;
            const int64_t rows = min(static_cast<int64_t>(RS), p.M - r0);
            prefetch_l2(static_cast<const unsigned char *>(p.A) + r0 * p.row_bytes,
                        static_cast<uint32_t>(rows * p.row_bytes));
        }
        pdl_wait();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&red[s]), NW);
        }
        mbar_init(smem_addr(xbar), 1);
        *abort_flag = 0;
    }
    __syncthreads();

    if (warp == NW) {
        // ---------------- producer warp ----------------
        int64_t issued = 0;
        // with programmatic dependent launch the weights stream in before the
        // wait for the preceding kernel; x only after it
        if (p.pdl) {
            if (lane == 0)
                for (; issued < S && issued < iters; ++issued) issue(issued);
            pdl_wait();  // the whole producer warp writes y only after the wait
        }
        if constexpr (XV == 1) {
            if (lane == 0) {
                mbar_arrive_expect_tx(smem_addr(xbar), xbytes);
                if (!(p.skip_copies & SKIP_X)) bulk_copy_g2s(smem_addr(xs), p.x, xbytes, smem_addr(xbar));
            }
        } else {
            // the consumer warps load x: the first stage goes out at once, the
            // other stages only once the x loads have been issued (queued
            // behind a burst of S stages from every block, x would arrive only
            // when the whole burst has, and no consumer can start before it)
            if (lane == 0 && issued == 0 && iters > 0) issue(issued++);
            asm volatile("bar.sync 2, %0;" ::"r"(T + 32) : "memory");
        }
        if (lane == 0)
            for (; issued < S && issued < iters; ++issued) issue(issued);
        issued = __shfl_sync(0xffffffffu, issued, 0);
        int64_t done = 0;
        for (; done < iters; ++done) {
            const int slot = static_cast<int>(done % S);
            bool ok = mbar_wait_bounded(smem_addr(&red[slot]), static_cast<uint32_t>((done / S) & 1),
                                        p.wait_limit_ns);
            ok = __all_sync(0xffffffffu, ok) && !__any_sync(0xffffffffu, *abort_flag != 0);
            if (!ok) {
                if (lane == 0 && !*abort_flag) fail();
                break;
            }
            const int64_t r0 = (blockIdx.x + done * grid) * RS;
            const int rows = static_cast<int>(min(static_cast<int64_t>(RS), p.M - r0));
            // one partial per consumer thread and row: each lane adds T/32 of
            // them (in a fixed order), then the warp butterfly
            const float *pp = part + slot * T * RS;
#pragma unroll
            for (int r = 0; r < RS; ++r) {
                float v = 0.f;
#pragma unroll
                for (int i = lane; i < T; i += 32) v += pp[r * T + i];
                v = group_sum<32>(v);
                if (lane == 0 && r < rows) p.y[r0 + r] = v;
            }
            __syncwarp();
            if (lane == 0 && issued < iters) issue(issued);
            ++issued;
            if (issued > iters) issued = iters;
        }
        if (lane == 0) {
            // copies issued for iterations [done, issued) may still be in flight
            bool drained = true;
            for (int64_t j = done; j < issued; ++j) {
                if (j == 0 && (p.skip_copies & SKIP_STAGE)) continue;  // never issued
                drained &= mbar_wait_bounded(smem_addr(&full[j % S]), static_cast<uint32_t>((j / S) & 1),
                                             p.wait_limit_ns);
            }
            if (XV == 1 && *abort_flag) {
                // the x copy, too, may still be in flight
                if (!(p.skip_copies & SKIP_X)) drained &= mbar_wait_bounded(smem_addr(xbar), 0, p.wait_limit_ns);
            }
            if (!drained) report_error(p.err, DEVERR_UNDRAINED);
        }
        return;
    }

    // ---------------- consumer warps ----------------
    // (every exit decision is made warp-uniform before the warp's shuffles)
    if (p.pdl) pdl_wait();
    // XREG: this thread's x vectors (chunks tid + j T), loaded with ordinary
    // loads that go out before the barrier arrive (see stage_x_vmajor), and
    // re-paired for INT4 once they have arrived
    uint4 xr[XREG ? CF : 1][XV];
    if constexpr (XV == 1) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(xbar), 0, p.wait_limit_ns))) {
            if (lane == 0) fail();
            return;
        }
    } else if constexpr (XREG) {
        const uint4 *src = static_cast<const uint4 *>(p.x);
#pragma unroll
        for (int j = 0; j < CF; ++j)
#pragma unroll
            for (int v = 0; v < XV; ++v) xr[j][v] = ld_l2_16(src + (tid + j * T) * XV + v);
        asm volatile("bar.arrive 2, %0;" ::"r"(T + 32) : "memory");
        if constexpr (PAIRED) {
#pragma unroll
            for (int j = 0; j < CF; ++j)
#pragma unroll
                for (int v = 0; v < XV; ++v) xr[j][v] = pair_x_vec(xr[j][v]);
        }
    } else {
        // several vectors of x per chunk: transpose x into shared memory,
        // then a named barrier of the consumer warps only
        // (every consumer warp arrives on barrier 2 once its first x loads
        // are out; the producer warp waits there before copying weights)
        stage_x_vmajor<DT, PAIRED, true>(const_cast<unsigned char *>(xs), p.x, nchunks, tid, T, [] {
            asm volatile("bar.arrive 2, %0;" ::"r"(T + 32) : "memory");
        });
        asm volatile("bar.sync 1, %0;" ::"r"(T) : "memory");
    }
    // x plane bases (vector-major x), and with a fixed chunk count this
    // thread's x addresses and scale offsets
    const uint32_t t16 = static_cast<uint32_t>(tid) * 16u;
    uint32_t xbase[XV], xthr[XV];
#pragma unroll
    for (int v = 0; v < XV; ++v) {
        xbase[v] = smem_addr(xs) + static_cast<uint32_t>(v) * static_cast<uint32_t>(nchunks) * 16u;
        xthr[v] = xbase[v] + t16;
    }
    uint32_t sgrp[CF > 0 ? CF : 1];
#pragma unroll
    for (int j = 0; j < (CF > 0 ? CF : 1); ++j) sgrp[j] = 2u * static_cast<uint32_t>((tid + j * T) >> p.scale_shift);
    for (int64_t it = 0; it < iters; ++it) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return;
        const int slot = static_cast<int>(it % S);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&full[slot]),
                                                        static_cast<uint32_t>((it / S) & 1),
                                                        p.wait_limit_ns))) {
            if (lane == 0) fail();
            return;
        }
        const int64_t r0 = (blockIdx.x + it * grid) * RS;
        const int rows = static_cast<int>(min(static_cast<int64_t>(RS), p.M - r0));
        // 32-bit shared-space addresses, per-row offsets hoisted out of the loop
        const uint32_t st = smem_addr(smem + L.stage + slot * L.stage_bytes);
        const uint32_t ss = smem_addr(smem + L.scale + slot * L.scale_bytes);
        const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
        const uint32_t gb = static_cast<uint32_t>(2 * p.groups);
        float acc[RS][NACC];
#pragma unroll
        for (int r = 0; r < RS; ++r)
#pragma unroll
            for (int k = 0; k < NACC; ++k) acc[r][k] = 0.f;
        // ROW_SCALE: one scale per row, read once per tile from global memory;
        // FULL: all RS rows of the tile exist (no per-row checks in the loop)
        auto dot_rows = [&](auto row_scale, auto full_tile) {
            constexpr bool ROW_SCALE = decltype(row_scale)::value;
            constexpr bool FULL = decltype(full_tile)::value;
            float rsc[ROW_SCALE ? RS : 1];
            if constexpr (ROW_SCALE) {
#pragma unroll
                for (int r = 0; r < RS; ++r) rsc[r] = r < rows ? ld_half_as_float(p.scales + r0 + r) : 0.f;
            }
            // one chunk of every row of the tile: x vectors xv, row r of the
            // stage at arow[r] + off, its scale at srow[r] + soff
            auto chunk_x = [&](const uint4 (&xv)[XV], const uint32_t (&arow)[RS],
                               const uint32_t (&srow)[RS], uint32_t off, uint32_t soff) {
                [[maybe_unused]] float xf[MATH == MATH_F32 ? F::EPC : 1];
                if constexpr (MATH == MATH_F32) x_to_float<DT>(xv, xf);
#pragma unroll
                for (int r = 0; r < RS; ++r) {
                    if (FULL || r < rows) {
                        const uint4 a = lds128(arow[r] + off);
                        float sc = 0.f;
                        if constexpr (ROW_SCALE)
                            sc = rsc[r];
                        else if constexpr (F::QUANT)
                            sc = lds_half_as_float(srow[r] + soff);
                        if constexpr (MATH == MATH_MIXED) {
                            chunk_dot_mixed<DT, PAIRED>(a, xv, sc, acc[r]);
                        } else {
                            float wf[F::EPC];
                            chunk_to_float<DT>(a, wf);
                            chunk_fma<DT>(wf, xf, sc, acc[r]);
                        }
                    }
                }
            };
            // the same with the x vectors at xrow[v] + off in shared memory
            auto chunk = [&](const uint32_t (&xrow)[XV], const uint32_t (&arow)[RS],
                             const uint32_t (&srow)[RS], uint32_t off, uint32_t soff) {
                uint4 xv[XV];
#pragma unroll
                for (int v = 0; v < XV; ++v) xv[v] = lds128(xrow[v] + off);
                chunk_x(xv, arow, srow, off, soff);
            };
            uint32_t arow[RS], srow[RS];
#pragma unroll
            for (int r = 0; r < RS; ++r) {
                arow[r] = st + r * rb;
                srow[r] = ss + r * gb;
            }
            if constexpr (CF > 0) {
                // exactly CF chunks per thread and row: fixed offsets from
                // per-thread bases (no address arithmetic in the loop)
#pragma unroll
                for (int r = 0; r < RS; ++r) arow[r] += t16;
#pragma unroll
                for (int j = 0; j < CF; ++j) {
                    if constexpr (XREG) chunk_x(xr[j], arow, srow, j * T * 16u, sgrp[j]);
                    else chunk(xthr, arow, srow, j * T * 16u, sgrp[j]);
                }
            } else {
#pragma unroll 2
                for (int c = tid; c < nchunks; c += T)
                    chunk(xbase, arow, srow, static_cast<uint32_t>(c) * 16u,
                          2u * static_cast<uint32_t>(c >> p.scale_shift));
            }
        };
        if constexpr (F::QUANT) {
            if (p.groups == 1) dot_rows(std::true_type{}, std::false_type{});
            else if (rows == RS) dot_rows(std::false_type{}, std::true_type{});
            else dot_rows(std::false_type{}, std::false_type{});
        } else {
            dot_rows(std::false_type{}, std::false_type{});
        }
        // each thread leaves its row sums for the producer warp to add up
        // (no butterfly in the consumer warps)
        float *pp = part + slot * T * RS;
#pragma unroll
        for (int r = 0; r < RS; ++r) pp[r * T + tid] = (acc[r][0] + acc[r][1]) + (acc[r][2] + acc[r][3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&red[slot]));
    }
}

// ---------------------------------------------------------------------------
// Row-band kernel (x held in registers)
// ---------------------------------------------------------------------------
//
// For rows of exactly T * CPT chunks.  Thread t of a block always multiplies
// the chunks t, t + T, ..., t + (CPT - 1) T of a row, so it loads the x
// vectors of those chunks into registers once and never reads x again (for
// INT4 that is 64 bytes of x per 16-byte chunk of A, which from shared
// memory would cost four loads per chunk and row).  Block b of the
// persistent grid takes rows b, b + grid, b + 2 grid, ...: every block owns
// floor(M / grid) or ceil(M / grid) rows, and at any moment the grid as a
// whole streams one dense band of consecutive rows.  Each thread keeps its
// chunks of the next U rows in flight in a rolling window of registers: the
// loads of row j + U are issued as soon as row j has been taken out of its
// slot, before row j is multiplied.  Per row, the lane partials meet in a
// warp butterfly and the warps' partials in shared memory, one block barrier
// per U rows ("llama.cpp GEMV CUDA": warp reduction, warp sums through shared
// memory, a second reduction).  Quantised chunks are summed into two FP32
// partials of exact binary16 products and scaled once per chunk (a chunk
// never straddles a 128-column group).
//
// The products are volatile asm: the compiler keeps them in program order
// relative to the (volatile) loads, so the loads of row j + U are issued
// before row j is multiplied and each slot's registers are reused at once
// (otherwise the scheduler hoists all U loads of the next rows above the
// products and needs a second window of registers).
__device__ __forceinline__ void mfma_pair_ordered(uint32_t a, uint32_t b, float &c0, float &c1)
{
    asm volatile("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
                 " fma.rn.f32.f16 %0, a0, b0, %0;\n fma.rn.f32.f16 %1, a1, b1, %1;\n}"
                 : "+f"(c0), "+f"(c1)
                 : "r"(a), "r"(b));
}

template <int DT, bool PAIRED>
__device__ __forceinline__ void band_chunk(const uint4 a, const uint4 (&xv)[x_chunk_vecs<DT>()],
                                           float &c0, float &c1)
{
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    if constexpr (DT == DT_F32) {
        c0 = fmaf(__uint_as_float(w[0]), __uint_as_float(xv[0].x), c0);
        c1 = fmaf(__uint_as_float(w[1]), __uint_as_float(xv[0].y), c1);
        c0 = fmaf(__uint_as_float(w[2]), __uint_as_float(xv[0].z), c0);
        c1 = fmaf(__uint_as_float(w[3]), __uint_as_float(xv[0].w), c1);
    } else if constexpr (DT == DT_F16) {
        mfma_pair_ordered(w[0], xv[0].x, c0, c1);
        mfma_pair_ordered(w[1], xv[0].y, c0, c1);
        mfma_pair_ordered(w[2], xv[0].z, c0, c1);
        mfma_pair_ordered(w[3], xv[0].w, c0, c1);
    } else if constexpr (DT == DT_Q8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t h[2];
            q8_codes_h2(w[k], h);
            const uint4 &x = xv[k >> 1];
            mfma_pair_ordered(h[0], (k & 1) ? x.z : x.x, c0, c1);
            mfma_pair_ordered(h[1], (k & 1) ? x.w : x.y, c0, c1);
        }
    } else {
        static_assert(DT == DT_Q4 && PAIRED, "INT4 takes x in the paired order");
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t h[4];
            q4_codes_h2(w[k], h);
            const uint4 &x = xv[k];
            mfma_pair_ordered(h[0], x.x, c0, c1);
            mfma_pair_ordered(h[1], x.y, c0, c1);
            mfma_pair_ordered(h[2], x.z, c0, c1);
            mfma_pair_ordered(h[3], x.w, c0, c1);
        }
    }
}

// The G rows of a tile times one x chunk, word by word with the rows
// innermost, into two FP32 partials per row: 2 G independent accumulation
// chains, so the half-rate mixed-precision FMAs of different rows overlap.
template <int DT, bool PAIRED, int G>
__device__ __forceinline__ void tile_chunk(const uint4 (&a)[G], const uint4 (&xv)[x_chunk_vecs<DT>()],
                                           float (&c0)[G], float (&c1)[G])
{
    if constexpr (DT == DT_F16X32) {
        // binary16 weights widened to FP32 (exact), FP32 x, FP32 FMAs: word q
        // of a chunk holds columns 2q and 2q + 1, whose x sit in vector q / 2
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 &x = xv[q >> 1];
            const float xa = __uint_as_float((q & 1) ? x.z : x.x);
            const float xb = __uint_as_float((q & 1) ? x.w : x.y);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t w = q == 0 ? a[g].x : q == 1 ? a[g].y : q == 2 ? a[g].z : a[g].w;
                const float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&w));
                c0[g] = fmaf(wf.x, xa, c0[g]);
                c1[g] = fmaf(wf.y, xb, c1[g]);
            }
        }
    } else if constexpr (DT == DT_F32) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            c0[g] = fmaf(__uint_as_float(a[g].x), __uint_as_float(xv[0].x), c0[g]);
            c1[g] = fmaf(__uint_as_float(a[g].y), __uint_as_float(xv[0].y), c1[g]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            c0[g] = fmaf(__uint_as_float(a[g].z), __uint_as_float(xv[0].z), c0[g]);
            c1[g] = fmaf(__uint_as_float(a[g].w), __uint_as_float(xv[0].w), c1[g]);
        }
    } else if constexpr (DT == DT_F16) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t xw = q == 0 ? xv[0].x : q == 1 ? xv[0].y : q == 2 ? xv[0].z : xv[0].w;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t w = q == 0 ? a[g].x : q == 1 ? a[g].y : q == 2 ? a[g].z : a[g].w;
                mfma_pair(w, xw, c0[g], c1[g]);
            }
        }
    } else if constexpr (DT == DT_Q8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 &x = xv[q >> 1];
            const uint32_t x01 = (q & 1) ? x.z : x.x;
            const uint32_t x23 = (q & 1) ? x.w : x.y;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t w = q == 0 ? a[g].x : q == 1 ? a[g].y : q == 2 ? a[g].z : a[g].w;
                uint32_t h[2];
                q8_codes_h2(w, h);
                mfma_pair(h[0], x01, c0[g], c1[g]);
                mfma_pair(h[1], x23, c0[g], c1[g]);
            }
        }
    } else {
        static_assert(DT == DT_Q4 && PAIRED, "INT4 takes x in the paired order");
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 &x = xv[q];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t w = q == 0 ? a[g].x : q == 1 ? a[g].y : q == 2 ? a[g].z : a[g].w;
                uint32_t h[4];
                q4_codes_h2(w, h);
                mfma_pair(h[0], x.x, c0[g], c1[g]);
                mfma_pair(h[1], x.y, c0[g], c1[g]);
                mfma_pair(h[2], x.z, c0[g], c1[g]);
                mfma_pair(h[3], x.w, c0[g], c1[g]);
            }
        }
    }
}

// Predicated loads that leave the destination unchanged when the predicate is
// false (the same registers either way, so a rolling window needs no copies).
__device__ __forceinline__ void ld_stream16_if(uint4 &v, const void *p, bool pred)
{
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %5, 0;\n"
                 " @q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];\n}"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                 : "l"(p), "r"(static_cast<int>(pred)));
}

// 16-bit load into the low half of a 32-bit register (zero-extended); the
// binary16 value is converted only where it is used, so the load stays in
// flight.
__device__ __forceinline__ void ld_u16_if(uint32_t &v, const void *p, bool pred)
{
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q ld.global.nc.u16 %0, [%1];\n}"
                 : "+r"(v)
                 : "l"(p), "r"(static_cast<int>(pred)));
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// 16-byte streaming load into registers that already hold the slot's
// previous data (the same registers, so a rolling window needs no copies).
__device__ __forceinline__ void ld_stream16_into(uint4 &v, const void *p)
{
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                 : "l"(p));
}

__device__ __forceinline__ void ld_u16_into(uint32_t &v, const void *p)
{
    asm volatile("ld.global.nc.u16 %0, [%1];" : "+r"(v) : "l"(p));
}

// Sums U values (U a power of two, at most 32) over the 32 lanes of a warp:
// afterwards lane l holds the warp sum of value l >> (5 - log2 U).  At each
// of the first log2 U steps a lane keeps half of its values (the upper half
// when its lane bit at that distance is set) and adds its partner's copy of
// them (one shuffle per kept value); the remaining steps are a plain XOR
// butterfly.  U - 1 + 5 - log2 U shuffles instead of 5 U.
template <int U>
__device__ __forceinline__ float warp_sum_rows(float (&v)[U], int lane)
{
    static_assert(U >= 1 && U <= 32 && (U & (U - 1)) == 0, "U: a power of two up to 32");
    float w[U];
#pragma unroll
    for (int i = 0; i < U; ++i) w[i] = v[i];
    int d = 16;
#pragma unroll
    for (int k = U; k > 1; k >>= 1, d >>= 1) {
        const bool up = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < k / 2; ++i) {
            const float keep = up ? w[i + k / 2] : w[i];
            const float send = up ? w[i] : w[i + k / 2];
            w[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
    }
    float s = w[0];
#pragma unroll
    for (; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
    return s;
}

// G consecutive rows form a tile; tiles are dealt to blocks in grid-stride
// order (tile b, b + grid, ...), TW tiles (U = G * TW rows) in flight per
// thread.  Rows of a tile are ROWB bytes apart, so their addresses are
// immediate offsets of one pointer per tile.
template <int DT, int T, int CPT, int G, int TW, int MINB>
__global__ void __launch_bounds__(T, MINB) mbg_rowband_kernel(const GemvArgs p)
{
    using F = Fmt<DT>;
    constexpr int XV = x_chunk_vecs<DT>();
    constexpr int NW = T / 32;
    constexpr int U = G * TW;           // rows in flight per thread
    constexpr int ROWB = T * CPT * 16;  // bytes per row
    constexpr bool PAIRED = DT == DT_Q4;
    static_assert(T % 32 == 0 && NW <= 32, "block shape");
    static_assert(F::XB == 2 || DT == DT_F32 || DT == DT_F16X32,
                  "binary16 x (mixed-precision products), FP32, or binary16 weights with an FP32 x");
    static_assert((U & (U - 1)) == 0 && U <= 32, "rows in flight: a power of two up to 32");

    __shared__ float part[2][U][NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t grid = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t ntiles = (p.M + G - 1) / G;
    // tiles of this block: b + i * grid for 0 <= i < I
    const int64_t I = b < ntiles ? (ntiles - 1 - b) / grid + 1 : 0;
    const unsigned char *abase = static_cast<const unsigned char *>(p.A) + tid * 16;

    pdl_trigger();
    // the first tiles of this block into L2 while the preceding kernel
    // drains (a hint only: it changes no value a later load returns)
    if (tid < TW && tid < I) {
        const int64_t row0 = (b + tid * grid) * G;
        const int64_t rows = p.M - row0 < G ? p.M - row0 : G;
        prefetch_l2(static_cast<const unsigned char *>(p.A) + row0 * ROWB, static_cast<uint32_t>(rows * ROWB));
    }
    if (!p.pdl) pdl_wait();

    // scale of chunk c of a row: scales[row * groups + (c >> scale_shift)]
    int soff[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) soff[k] = (tid + k * T) >> p.scale_shift;
    const int64_t sgrp = p.groups;  // scales per row

    uint4 a[U][CPT];
    uint32_t sc[U][CPT];  // binary16 scale bits
#pragma unroll
    for (int r = 0; r < U; ++r)
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            a[r][k] = make_uint4(0u, 0u, 0u, 0u);
            sc[r][k] = 0u;
        }
    // tiles are loaded strictly in the order i = 0, 1, 2, ...: one pointer per
    // operand walks them (grid tiles apart; both steps in bytes, advanced by
    // a volatile add so that the compiler keeps no address per slot)
    int64_t in = 0;
    const unsigned char *an = abase + b * G * ROWB;
    const int64_t astep = grid * G * ROWB;
    const unsigned char *sn = F::QUANT ? reinterpret_cast<const unsigned char *>(p.scales + b * G * sgrp) : nullptr;
    const int64_t sstep = grid * G * sgrp * 2;
    // FULL: the tile and all its rows exist (no predicates)
    auto load_tile = [&](int w, auto full) {
        constexpr bool FULL = decltype(full)::value;
        const int64_t row0 = (b + in * grid) * G;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const bool ok = FULL || (in < I && row0 + g < p.M);
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                        if constexpr (FULL) ld_stream16_into(a[w * G + g][k], an + g * ROWB + k * T * 16);
                else ld_stream16_if(a[w * G + g][k], an + g * ROWB + k * T * 16, ok);
            }
            if constexpr (F::QUANT) {
#pragma unroll
                for (int k = 0; k < CPT; ++k) {
                    const void *sp = sn + (g * sgrp + soff[k]) * 2;
                    if constexpr (FULL) ld_u16_into(sc[w * G + g][k], sp);
                    else ld_u16_if(sc[w * G + g][k], sp, ok);
                }
            }
        }
        if constexpr (F::QUANT) asm volatile("add.s64 %0, %0, %1;" : "+l"(sn) : "l"(sstep));
        asm volatile("add.s64 %0, %0, %1;" : "+l"(an) : "l"(astep));
        ++in;
    };
#pragma unroll
    for (int w = 0; w < TW; ++w) load_tile(w, std::false_type{});
    if (p.pdl) pdl_wait();

    // this thread's x vectors (read after the wait: the preceding kernel may
    // have written x); re-paired for INT4 so that every product takes the
    // same half of both operands
    uint4 xr[CPT][XV];
    {
        const uint4 *xs = static_cast<const uint4 *>(p.x);
#pragma unroll
        for (int k = 0; k < CPT; ++k)
#pragma unroll
            for (int v = 0; v < XV; ++v) xr[k][v] = ld_l2_16(xs + (tid + k * T) * XV + v);
        if constexpr (PAIRED) {
#pragma unroll
            for (int k = 0; k < CPT; ++k)
#pragma unroll
                for (int v = 0; v < XV; ++v) xr[k][v] = pair_x_vec(xr[k][v]);
        }
    }

    // the products of the G row slots of tile slot w into acc (rows of tiles
    // that do not exist give values that are never stored)
    auto tile_dot = [&](int w, float (&acc)[U]) {
        float c0[G], c1[G];
#pragma unroll
        for (int g = 0; g < G; ++g) c0[g] = c1[g] = 0.f;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            uint4 ak[G];
#pragma unroll
            for (int g = 0; g < G; ++g) ak[g] = a[w * G + g][k];
            if constexpr (F::QUANT) {
                float d0[G], d1[G];
#pragma unroll
                for (int g = 0; g < G; ++g) d0[g] = d1[g] = 0.f;
                tile_chunk<DT, PAIRED, G>(ak, xr[k], d0, d1);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float s = half_bits_to_float(sc[w * G + g][k]);
                    c0[g] = fmaf(s, d0[g], c0[g]);
                    c1[g] = fmaf(s, d1[g], c1[g]);
                }
            } else {
                tile_chunk<DT, PAIRED, G>(ak, xr[k], c0, c1);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) acc[w * G + g] = c0[g] + c1[g];
    };

    int half = 0;
    for (int64_t i0 = 0; i0 < I; i0 += TW) {
        // every tile of this window and of the next one exists in full
        const int64_t last = i0 + 2 * TW - 1;
        const bool full = last < I && (b + last * grid) * G + G <= p.M;
        float acc[U];
        auto window = [&](auto fl) {
#pragma unroll
            for (int w = 0; w < TW; ++w) {
                // rows of tile i0 + w are multiplied straight from their
                // slots, which are then refilled in place with tile i0 + TW + w
                tile_dot(w, acc);
                load_tile(w, fl);
            }
        };
        if (full) window(std::true_type{});
        else window(std::false_type{});
        // lane l ends with the warp's share of row slot l >> (5 - log2 U)
        const float s = warp_sum_rows<U>(acc, lane);
        constexpr int LPR = 32 / U;  // lanes holding each row's sum
        if ((lane & (LPR - 1)) == 0) part[half][lane / LPR][warp] = s;
        __syncthreads();
        if (tid < U) {
            const int64_t i = i0 + tid / G;
            const int64_t row = (b + i * grid) * G + tid % G;
            if (i < I && row < p.M) {
                float v = 0.f;
#pragma unroll
                for (int q = 0; q < NW; ++q) v += part[half][tid][q];
                p.y[row] = v;
            }
        }
        half ^= 1;
    }
}

// ---------------------------------------------------------------------------
// MMA row-band kernel (INT8 / INT4: products on the warp-level MMA unit)
// ---------------------------------------------------------------------------
//
// The quantised row bands spend most of their issue slots on products: one
// mixed-precision FMA per weight on top of the unpacking (one LOP3 and one
// binary16 pair operation per two codes).  Here the exact binary16 codes that
// the unpacking leaves in registers go straight into
// mma.sync.m16n8k16.f32.f16.f16.f32 as the A fragment: one instruction takes
// eight codes per lane (256 per warp), multiplies them exactly (binary16 x
// binary16 products are exact) and accumulates in FP32.  The MMA unit is used
// as a dot-product engine; the weights still stream from HBM into registers
// with 16-byte read-only loads, like every other row band.
//
// Layout of one step (512 bytes of each of the 2 rows of a tile): a "slot" is
// 64 contiguous bytes of a row (one 128-column scale group for INT4, half of
// one for INT8).  The 16 rows of the MMA's A operand are 16 (row, slot)
// pairs: A-row i < 8 is row i & 1 of the tile, slot 2 (i >> 1); A-row i + 8
// is the same row, slot 2 (i >> 1) + 1.  Lane (g, t) (g = lane / 4,
// t = lane % 4) loads the 16-byte chunk t of A-rows g and g + 8 — chunk t of
// two adjacent slots of row g & 1.  The eight columns of the B operand carry
// eight slices of x: column n holds the x of slot n (lane (n, t) supplies
// its chunk t), so A-row g meets its own x in column 2 (g >> 1) and A-row
// g + 8 in column 2 (g >> 1) + 1: both land in lane (g, g >> 1) of the
// result, in registers d[0] and d[3].  The other 48 values of the 16 x 8
// result are products with foreign slices and are never read.  A lane's two
// slots are adjacent, so their scales are one 4-byte load (INT4: two
// neighbouring groups) or one scale (INT8: the two halves of one group).
// The useful values are scaled, summed over the warp per row and over the
// warps of the block per row.
//
// Thread t of the block always multiplies the same slots of every row, so its
// x fragments are loaded into registers once.  Tiles of 2 consecutive rows are
// dealt to the blocks of a persistent grid in grid-stride order; each lane
// keeps its chunks of the next TW tiles in flight in a rolling window of
// registers (refilled in place, as in the row-band kernel).  Warp w takes the
// steps w, w + NW, ..., so for every step index the block reads NW * 512
// contiguous bytes of each row.  The MMAs of a step alternate between two
// accumulators, each started from zero by its first MMA.  Rows must be
// exactly NW * SPW * 512 bytes.
__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                 uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B (the accumulator input is zero)
__device__ __forceinline__ void mma_m16n8k16_f16_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                       uint32_t a3, uint32_t b0, uint32_t b1)
{
    const float z = 0.f;
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%10, %10, %10, %10};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// The code unpacking of q8_codes_h2 / q4_codes_h2 as volatile asm: kept in
// program order between the (volatile) MMAs, so that a step's codes are
// unpacked right before its MMAs and only one step's codes are live at a time.
__device__ __forceinline__ uint32_t vlop3_sel_xor(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm volatile("lop3.b32 %0, %1, %2, %3, 0x6C;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t vhsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm volatile("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t vhfma2(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm volatile("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t vprmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm volatile("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// Two words of codes at once (the A fragments of one MMA step): all the
// integer operations first, then the binary16 pair operations, so that no
// pair operation issues right behind the integer operation it reads.
__device__ __forceinline__ void q4_codes_h2_two(uint32_t wa, uint32_t wb, uint32_t (&ha)[4], uint32_t (&hb)[4])
{
    uint32_t va, vb;
    asm volatile("shr.b32 %0, %1, 8;" : "=r"(va) : "r"(wa));
    asm volatile("shr.b32 %0, %1, 8;" : "=r"(vb) : "r"(wb));
    ha[0] = vlop3_sel_xor(wa, 0x64086408u, 0x000F000Fu);
    hb[0] = vlop3_sel_xor(wb, 0x64086408u, 0x000F000Fu);
    ha[1] = vlop3_sel_xor(wa, 0x64806480u, 0x00F000F0u);
    hb[1] = vlop3_sel_xor(wb, 0x64806480u, 0x00F000F0u);
    ha[2] = vlop3_sel_xor(va, 0x64086408u, 0x000F000Fu);
    hb[2] = vlop3_sel_xor(vb, 0x64086408u, 0x000F000Fu);
    ha[3] = vlop3_sel_xor(va, 0x64806480u, 0x00F000F0u);
    hb[3] = vlop3_sel_xor(vb, 0x64806480u, 0x00F000F0u);
    ha[0] = vhsub2(ha[0], 0x64086408u);
    hb[0] = vhsub2(hb[0], 0x64086408u);
    ha[1] = vhfma2(ha[1], 0x2C002C00u, 0xD480D480u);
    hb[1] = vhfma2(hb[1], 0x2C002C00u, 0xD480D480u);
    ha[2] = vhsub2(ha[2], 0x64086408u);
    hb[2] = vhsub2(hb[2], 0x64086408u);
    ha[3] = vhfma2(ha[3], 0x2C002C00u, 0xD480D480u);
    hb[3] = vhfma2(hb[3], 0x2C002C00u, 0xD480D480u);
}
__device__ __forceinline__ void q8_codes_h2_two(uint32_t wa, uint32_t wb, uint32_t (&ha)[2], uint32_t (&hb)[2])
{
    uint32_t ua, ub;
    asm volatile("xor.b32 %0, %1, 0x80808080;" : "=r"(ua) : "r"(wa));
    asm volatile("xor.b32 %0, %1, 0x80808080;" : "=r"(ub) : "r"(wb));
    ha[0] = vprmt(ua, 0x64646464u, 0x4140u);
    hb[0] = vprmt(ub, 0x64646464u, 0x4140u);
    ha[1] = vprmt(ua, 0x64646464u, 0x4342u);
    hb[1] = vprmt(ub, 0x64646464u, 0x4342u);
    ha[0] = vhsub2(ha[0], 0x64806480u);
    hb[0] = vhsub2(hb[0], 0x64806480u);
    ha[1] = vhsub2(ha[1], 0x64806480u);
    hb[1] = vhsub2(hb[1], 0x64806480u);
}

// A lane's two 16-byte chunks (one per slot) times its x fragments: eight
// MMAs (INT4) or four (INT8) that alternate between two accumulators, each
// started from zero by its first MMA, so that no MMA follows the one whose
// result it adds to.  The slot sums are d[0][0] + d[1][0] (first slot) and
// d[0][3] + d[1][3] (second slot) of a lane that holds results.
template <int DT>
__device__ __forceinline__ void mma_chunk_pair(const uint4 &c0, const uint4 &c1,
                                               const uint4 (&x)[DT == DT_Q4 ? 4 : 2], float (&d)[2][4])
{
    const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w};
    const uint32_t w1[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (DT == DT_Q4) {
            uint32_t h[4], h8[4];
            q4_codes_h2_two(w0[k], w1[k], h, h8);
            if (k == 0) {
                mma_m16n8k16_f16_first(d[0], h[0], h8[0], h[1], h8[1], x[k].x, x[k].y);
                mma_m16n8k16_f16_first(d[1], h[2], h8[2], h[3], h8[3], x[k].z, x[k].w);
            } else {
                mma_m16n8k16_f16(d[0], h[0], h8[0], h[1], h8[1], x[k].x, x[k].y);
                mma_m16n8k16_f16(d[1], h[2], h8[2], h[3], h8[3], x[k].z, x[k].w);
            }
        } else {
            uint32_t h[2], h8[2];
            q8_codes_h2_two(w0[k], w1[k], h, h8);
            const uint4 &xv = x[k >> 1];
            const uint32_t b0 = (k & 1) ? xv.z : xv.x, b1 = (k & 1) ? xv.w : xv.y;
            if (k < 2) mma_m16n8k16_f16_first(d[k & 1], h[0], h8[0], h[1], h8[1], b0, b1);
            else mma_m16n8k16_f16(d[k & 1], h[0], h8[0], h[1], h8[1], b0, b1);
        }
    }
}

// Sums each of the TW values over the 16 lanes that share lane bit 2 (lanes
// of one tile row).  The first log2 TW lane bits of (4, 3, 1) split the
// values (a lane keeps half of them at each of those steps and adds its
// partner's copy), the remaining bits of (4, 3, 1, 0) are a plain XOR
// butterfly.  Afterwards the lanes whose remaining bits are 0 hold the sums;
// the value a lane holds belongs to tile (bit 4, bit 3, bit 1) of its lane
// index, taken in that order.
template <int TW>
__device__ __forceinline__ float mma_rows_sum(float (&v)[TW], int lane)
{
    static_assert(TW == 1 || TW == 2 || TW == 4 || TW == 8, "tiles per window: 1, 2, 4 or 8");
    constexpr int kDist[4] = {16, 8, 2, 1};
    float w[TW];
#pragma unroll
    for (int i = 0; i < TW; ++i) w[i] = v[i];
    int step = 0;
#pragma unroll
    for (int k = TW; k > 1; k >>= 1, ++step) {
        const int d = kDist[step];
        const bool up = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < k / 2; ++i) {
            const float keep = up ? w[i + k / 2] : w[i];
            const float send = up ? w[i] : w[i + k / 2];
            w[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
    }
    float s = w[0];
#pragma unroll
    for (; step < 4; ++step) s += __shfl_xor_sync(0xffffffffu, s, kDist[step]);
    return s;
}

// Tile index within a window of TW tiles held by a lane after mma_rows_sum,
// and the lane bits that must be 0 for the lane to hold a sum.
template <int TW>
__device__ __forceinline__ int mma_rows_tile(int lane)
{
    if constexpr (TW == 8) return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 1) & 1);
    if constexpr (TW == 4) return ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
    if constexpr (TW == 2) return (lane >> 4) & 1;
    return 0;
}
template <int TW>
constexpr int mma_rows_rest()
{
    return TW == 8 ? 0x1 : TW == 4 ? 0x3 : TW == 2 ? 0xB : 0x1B;
}

// 32-bit load into a register that already holds the slot's previous value.
__device__ __forceinline__ void ld_u32_into(uint32_t &v, const void *p)
{
    asm volatile("ld.global.nc.u32 %0, [%1];" : "+r"(v) : "l"(p));
}
__device__ __forceinline__ void ld_u32_if(uint32_t &v, const void *p, bool pred)
{
    asm volatile("{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n @q ld.global.nc.u32 %0, [%1];\n}"
                 : "+r"(v)
                 : "l"(p), "r"(static_cast<int>(pred)));
}

template <int DT, int NW, int SPW, int TW, int MINB, bool RC>
__global__ void __launch_bounds__(NW * 32, MINB) mbg_mmaband_kernel(const GemvArgs p)
{
    static_assert(DT == DT_Q8 || DT == DT_Q4, "quantised weights only");
    static_assert(NW >= 1 && NW <= 32, "block shape");
    constexpr int XV = DT == DT_Q4 ? 4 : 2;  // 16-byte x vectors per 16-byte chunk of codes
    constexpr int ROWB = NW * SPW * 512;     // bytes per row
    constexpr int U = 2 * TW;                // rows per window
    // Two lane layouts.  RC = false: lane (g, t) loads chunk t of the slots
    // 2(g/2) and 2(g/2) + 1 of tile row g % 2 (A-rows g and g + 8; results in
    // d[0] and d[3]); INT4: the two slots are neighbouring scale groups (one
    // 4-byte load, groups a multiple of 8); INT8: both halves of one group, or
    // the row's one scale.  RC = true: lane (g, t) loads chunk t of slot g of
    // both tile rows, so each load instruction of a warp reads 512 contiguous
    // bytes of one row (A-rows g and g + 8 are rows 0 and 1; results in
    // d[g % 2] and d[2 + g % 2]); one scale per row, and one exchange across
    // lane bit 2 per tile leaves each lane the sums of row g % 2 over the
    // slots g and g ^ 1, as in the first layout.
    constexpr bool PAIR = DT == DT_Q4 && !RC;

    __shared__ float part[2][U][NW];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int rsel = g & 1;          // tile row whose sums this lane keeps
    const bool use = t == (g >> 1);  // this lane holds its A-rows' results

    const int64_t grid = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t ntiles = (p.M + 1) / 2;
    const int I = static_cast<int>(b < ntiles ? (ntiles - 1 - b) / grid + 1 : 0);

    pdl_trigger();
    if (tid < TW && tid < I) {
        const int64_t row0 = (b + tid * grid) * 2;
        const int64_t rows = p.M - row0 < 2 ? p.M - row0 : 2;
        prefetch_l2(static_cast<const unsigned char *>(p.A) + row0 * ROWB, static_cast<uint32_t>(rows * ROWB));
    }
    if (!p.pdl) pdl_wait();

    // byte offset of this lane's scale(s) of step s within the scales of a row
    int sidx[SPW];
#pragma unroll
    for (int s = 0; s < SPW; ++s)
        sidx[s] = (((((warp + s * NW) * 8 + (RC ? g : 2 * (g >> 1))) * 4) >> p.scale_shift) * 2);
    const int64_t sgrp = p.groups;

    uint4 a[TW][SPW][2];
    uint32_t sc[TW][SPW];           // binary16 scale bits (a pair, or one in the low half)
    uint32_t sc1[RC ? TW : 1][SPW];  // RC: the scale of tile row 1
#pragma unroll
    for (int w = 0; w < TW; ++w)
#pragma unroll
        for (int s = 0; s < SPW; ++s) {
            a[w][s][0] = a[w][s][1] = make_uint4(0u, 0u, 0u, 0u);
            sc[w][s] = 0u;
            if constexpr (RC) sc1[w][s] = 0u;
        }
    int in = 0;
    // RC: tile row 0 (row 1 lies ROWB further); else this lane's tile row
    const int64_t arow = RC ? 0 : rsel;
    const unsigned char *an = static_cast<const unsigned char *>(p.A) + (b * 2 + arow) * ROWB + warp * 512 +
                              (RC ? g * 64 : (g >> 1) * 128) + t * 16;
    constexpr int SECOND = RC ? ROWB : 64;  // offset of the second load
    const int64_t astep = grid * 2 * ROWB;
    const unsigned char *sn = reinterpret_cast<const unsigned char *>(p.scales + (b * 2 + arow) * sgrp);
    const int64_t srow = sgrp * 2;  // bytes of scales per row
    const int64_t sstep = grid * 2 * sgrp * 2;
    // FULL: the tile and both its rows exist (no predicates)
    auto load_tile = [&](int w, auto full) {
        constexpr bool FULL = decltype(full)::value;
        const int64_t row0 = (b + static_cast<int64_t>(in) * grid) * 2;
        const bool ok0 = FULL || (in < I && row0 + arow < p.M);
        const bool ok1 = FULL || (in < I && row0 + 1 < p.M);
#pragma unroll
        for (int s = 0; s < SPW; ++s) {
            const unsigned char *q = an + s * NW * 512;
            if constexpr (FULL) {
                ld_stream16_into(a[w][s][0], q);
                ld_stream16_into(a[w][s][1], q + SECOND);
                if constexpr (PAIR) ld_u32_into(sc[w][s], sn + sidx[s]);
                else ld_u16_into(sc[w][s], sn + sidx[s]);
                if constexpr (RC) ld_u16_into(sc1[w][s], sn + srow + sidx[s]);
            } else {
                ld_stream16_if(a[w][s][0], q, ok0);
                ld_stream16_if(a[w][s][1], q + SECOND, RC ? ok1 : ok0);
                if constexpr (PAIR) ld_u32_if(sc[w][s], sn + sidx[s], ok0);
                else ld_u16_if(sc[w][s], sn + sidx[s], ok0);
                if constexpr (RC) ld_u16_if(sc1[w][s], sn + srow + sidx[s], ok1);
            }
        }
        asm volatile("add.s64 %0, %0, %1;" : "+l"(sn) : "l"(sstep));
        asm volatile("add.s64 %0, %0, %1;" : "+l"(an) : "l"(astep));
        ++in;
    };
#pragma unroll
    for (int w = 0; w < TW; ++w) load_tile(w, std::false_type{});
    if (p.pdl) pdl_wait();

    // B fragments: chunk t of x slot g of each of this lane's steps (read
    // after the wait: the preceding kernel may have written x); INT4
    // re-paired four columns apart, the order in which the codes unpack
    uint4 xr[SPW][XV];
    {
        const unsigned char *xs = static_cast<const unsigned char *>(p.x);
#pragma unroll
        for (int s = 0; s < SPW; ++s) {
            // first code of the chunk: byte (step * 512 + slot * 64 + t * 16) of the row
            const int64_t cbyte = static_cast<int64_t>(warp + s * NW) * 512 + g * 64 + t * 16;
            const int64_t col = DT == DT_Q4 ? cbyte * 2 : cbyte;
#pragma unroll
            for (int v = 0; v < XV; ++v) {
                xr[s][v] = ld_l2_16(xs + col * 2 + v * 16);
                if constexpr (DT == DT_Q4) xr[s][v] = pair_x_vec(xr[s][v]);
            }
        }
    }

    // tile slot w times x: this lane's share of its row.  Every lane applies
    // its scales (no divergent branch); the lanes that hold no result (their
    // sums mix foreign slices) give 0 through one select per tile.
    auto tile_dot = [&](int w) -> float {
        if constexpr (RC) {
            float acc0 = 0.f, acc1 = 0.f;  // tile rows 0 and 1, slot g
#pragma unroll
            for (int s = 0; s < SPW; ++s) {
                float d[2][4];
                mma_chunk_pair<DT>(a[w][s][0], a[w][s][1], xr[s], d);
                const float r0 = rsel ? d[0][1] + d[1][1] : d[0][0] + d[1][0];
                const float r1 = rsel ? d[0][3] + d[1][3] : d[0][2] + d[1][2];
                acc0 = fmaf(half_bits_to_float(sc[w][s]), r0, acc0);
                acc1 = fmaf(half_bits_to_float(sc1[w][s]), r1, acc1);
            }
            // keep row g % 2, hand the other row to lane bit 2's partner
            // (slot g ^ 1, which keeps the other row)
            const float keep = rsel ? acc1 : acc0, send = rsel ? acc0 : acc1;
            const float acc = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            return use ? acc : 0.f;
        } else {
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < SPW; ++s) {
                float d[2][4];
                mma_chunk_pair<DT>(a[w][s][0], a[w][s][1], xr[s], d);
                const float r0 = d[0][0] + d[1][0], r3 = d[0][3] + d[1][3];
                if constexpr (PAIR) {
                    const float2 sf = __half22float2(*reinterpret_cast<const __half2 *>(&sc[w][s]));
                    acc = fmaf(sf.x, r0, acc);
                    acc = fmaf(sf.y, r3, acc);
                } else {
                    acc = fmaf(half_bits_to_float(sc[w][s]), r0 + r3, acc);
                }
            }
            return use ? acc : 0.f;
        }
    };

    int half = 0;
    for (int i0 = 0; i0 < I; i0 += TW) {
        // every tile of this window and of the next one exists in full
        const int last = i0 + 2 * TW - 1;
        const bool full = last < I && (b + static_cast<int64_t>(last) * grid) * 2 + 2 <= p.M;
        float acc[TW];
        auto window = [&](auto fl) {
#pragma unroll
            for (int w = 0; w < TW; ++w) {
                acc[w] = tile_dot(w);
                load_tile(w, fl);
            }
        };
        if (full) window(std::true_type{});
        else window(std::false_type{});
        const float s = mma_rows_sum<TW>(acc, lane);
        // lanes whose butterfly bits are all 0 hold (tile, row) sums
        if ((lane & mma_rows_rest<TW>()) == 0) part[half][mma_rows_tile<TW>(lane) * 2 + rsel][warp] = s;
        __syncthreads();
        if (tid < U) {
            const int i = i0 + tid / 2;
            const int64_t row = (b + static_cast<int64_t>(i) * grid) * 2 + (tid & 1);
            if (i < I && row < p.M) {
                float v = 0.f;
#pragma unroll
                for (int q = 0; q < NW; ++q) v += part[half][tid][q];
                p.y[row] = v;
            }
        }
        half ^= 1;
    }
}

// ---------------------------------------------------------------------------
// Staged row-band kernel (x in registers, tiles of A staged by bulk copies)
// ---------------------------------------------------------------------------
//
// The row-band kernel's work split (thread t multiplies chunks t, t + T, ...
// of every row with x held in registers; tiles of G consecutive rows dealt
// to blocks in grid-stride order), but the tiles reach the block through a
// ring of (PF + 1) TW shared-memory stages filled by bulk async copies, so
// the bytes in flight cost no registers: PF windows of TW tiles are in flight
// while one is multiplied.  Thread 0 issues the copies; everybody reads the
// stage (one 16-byte shared load per chunk and row).  The block barrier that
// closes each window of TW tiles (after the warp partials are written) also
// tells thread 0 that the window's stages have been read, and it refills them
// with the tiles (PF + 1) TW ahead.  Every wait is bounded: a thread
// whose wait gives up carries that into the window's barrier
// (__syncthreads_or), so the whole block leaves together; thread 0 first
// waits (bounded) for the copies it still has in flight.
template <int DT, int T, int CPT, int G, int TW, int PF, int MINB>
__global__ void __launch_bounds__(T, MINB) mbg_stageband_kernel(const GemvArgs p)
{
    using F = Fmt<DT>;
    constexpr int XV = x_chunk_vecs<DT>();
    constexpr int NW = T / 32;
    constexpr int U = G * TW;           // rows per window
    constexpr int S = (PF + 1) * TW;    // stages
    constexpr int ROWB = T * CPT * 16;  // bytes per row
    constexpr bool PAIRED = DT == DT_Q4;
    static_assert(T % 32 == 0 && NW <= 32, "block shape");
    static_assert(F::XB == 2 || DT == DT_F32, "binary16 x (mixed-precision products) or FP32");
    static_assert((U & (U - 1)) == 0 && U <= 32, "rows per window: a power of two up to 32");

    extern __shared__ __align__(128) unsigned char smem[];
    const StageBandLayout L = stageband_layout(S, U, NW, G, ROWB, p.groups, F::QUANT);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    float *part = reinterpret_cast<float *>(smem + L.part);  // [2][U][NW]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t grid = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t ntiles = (p.M + G - 1) / G;
    const int64_t I = b < ntiles ? (ntiles - 1 - b) / grid + 1 : 0;  // tiles b + i * grid
    const int64_t sgrp = p.groups;

    int64_t issued = 0;  // thread 0: tiles whose copies have been issued
    auto issue = [&](int64_t i) {
        const int s = static_cast<int>(i % S);
        const int64_t row0 = (b + i * grid) * G;
        const int64_t rows = p.M - row0 < G ? p.M - row0 : G;
        const uint32_t abytes = static_cast<uint32_t>(rows * ROWB);
        const uint32_t sbytes = F::QUANT ? static_cast<uint32_t>(rows * sgrp * 2) : 0u;
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, abytes + sbytes);
        if (i == 0 && (p.skip_copies & SKIP_STAGE)) return;  // test hook: the wait must run out
        bulk_copy_g2s(smem_addr(smem + L.stage + s * L.stage_bytes),
                      static_cast<const unsigned char *>(p.A) + row0 * ROWB, abytes, bar);
        if constexpr (F::QUANT)
            bulk_copy_g2s(smem_addr(smem + L.stage + s * L.stage_bytes + L.scale_off), p.scales + row0 * sgrp,
                          sbytes, bar);
    };

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_addr(&full[s]), 1);
        if (I > 0) {
            // the first tile into L2 while the preceding kernel drains (a hint)
            const int64_t row0 = b * G;
            const int64_t rows = p.M - row0 < G ? p.M - row0 : G;
            prefetch_l2(static_cast<const unsigned char *>(p.A) + row0 * ROWB, static_cast<uint32_t>(rows * ROWB));
        }
    }
    if (!p.pdl) pdl_wait();
    if (tid == 0)
        for (; issued < S && issued < I; ++issued) issue(issued);
    __syncthreads();  // barriers initialised before anyone waits on them
    if (p.pdl) pdl_wait();

    // this thread's x vectors (after the wait: the preceding kernel may have
    // written x), re-paired for INT4
    uint4 xr[CPT][XV];
    {
        const uint4 *xs = static_cast<const uint4 *>(p.x);
#pragma unroll
        for (int k = 0; k < CPT; ++k)
#pragma unroll
            for (int v = 0; v < XV; ++v) xr[k][v] = ld_l2_16(xs + (tid + k * T) * XV + v);
        if constexpr (PAIRED) {
#pragma unroll
            for (int k = 0; k < CPT; ++k)
#pragma unroll
                for (int v = 0; v < XV; ++v) xr[k][v] = pair_x_vec(xr[k][v]);
        }
    }
    // shared-space offsets of this thread's chunks and scales within a row
    const uint32_t stage0 = smem_addr(smem + L.stage);
    uint32_t soff[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) soff[k] = 2u * static_cast<uint32_t>((tid + k * T) >> p.scale_shift);

    int half = 0;
    for (int64_t i0 = 0; i0 < I; i0 += TW) {
        bool ok = true;
        float acc[U];
#pragma unroll
        for (int w = 0; w < TW; ++w) {
            const int64_t i = i0 + w;
#pragma unroll
            for (int g = 0; g < G; ++g) acc[w * G + g] = 0.f;
            if (i < I) {
                const int s = static_cast<int>(i % S);
                ok &= mbar_wait_bounded(smem_addr(&full[s]), static_cast<uint32_t>((i / S) & 1), p.wait_limit_ns);
                const uint32_t st = stage0 + static_cast<uint32_t>(s) * L.stage_bytes;
                // rows past the end of A hold stale bytes: their sums are never stored
                float c0[G], c1[G];
#pragma unroll
                for (int g = 0; g < G; ++g) c0[g] = c1[g] = 0.f;
#pragma unroll
                for (int k = 0; k < CPT; ++k) {
                    uint4 ak[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) ak[g] = lds128(st + g * ROWB + (tid + k * T) * 16);
                    if constexpr (F::QUANT) {
                        float d0[G], d1[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) d0[g] = d1[g] = 0.f;
                        tile_chunk<DT, PAIRED, G>(ak, xr[k], d0, d1);
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float sc = lds_half_as_float(st + L.scale_off + g * sgrp * 2 + soff[k]);
                            c0[g] = fmaf(sc, d0[g], c0[g]);
                            c1[g] = fmaf(sc, d1[g], c1[g]);
                        }
                    } else {
                        tile_chunk<DT, PAIRED, G>(ak, xr[k], c0, c1);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) acc[w * G + g] = c0[g] + c1[g];
            }
        }
        // lane l ends with the warp's share of row slot l >> (5 - log2 U)
        const float sum = warp_sum_rows<U>(acc, lane);
        constexpr int LPR = 32 / U;
        if ((lane & (LPR - 1)) == 0) part[(half * U + lane / LPR) * NW + warp] = sum;
        // every thread has read the window's stages and written its partials;
        // a wait that gave up anywhere makes the whole block leave here
        if (__syncthreads_or(ok ? 0 : 1)) {
            if (tid == 0) {
                report_error(p.err, DEVERR_TIMEOUT);
                bool drained = true;
                for (int64_t j = i0; j < issued; ++j) {
                    if (j == 0 && (p.skip_copies & SKIP_STAGE)) continue;  // never issued
                    drained &= mbar_wait_bounded(smem_addr(&full[j % S]), static_cast<uint32_t>((j / S) & 1),
                                                 p.wait_limit_ns);
                }
                if (!drained) report_error(p.err, DEVERR_UNDRAINED);
            }
            return;
        }
        if (tid == 0)
            for (; issued < i0 + S + TW && issued < I; ++issued) issue(issued);  // into the window's stages
        if (tid < U) {
            const int64_t i = i0 + tid / G;
            const int64_t row = (b + i * grid) * G + tid % G;
            if (i < I && row < p.M) {
                float v = 0.f;
#pragma unroll
                for (int q = 0; q < NW; ++q) v += part[(half * U + tid) * NW + q];
                p.y[row] = v;
            }
        }
        half ^= 1;
    }
}

// ---------------------------------------------------------------------------
// Staged MMA row-band kernel (INT8 / INT4)
// ---------------------------------------------------------------------------
//
// The MMA row band's arithmetic (exact binary16 codes into
// mma.sync.m16n8k16, eight slices of x in the eight B columns), with tiles of
// RP row pairs streamed into a ring of (PF + 1) TW shared-memory stages by
// bulk async copies (the staged row band's pipeline: thread 0 issues, every
// wait bounded, the block barrier that closes a window of TW tiles frees its
// stages).  The bytes in flight cost no registers, so the lookahead (PF
// windows) does not compete with the arithmetic for registers; the row pairs
// of a tile share the B fragments and the per-tile bookkeeping.  (Measured
// no faster than the register-resident band or the bulk pipeline on the
// decode shapes: an explicit option.)
//
// Slots in a stage: lane (g, t) reads chunk t of slots k and 4 + k of row
// g & 1 of each row pair, with k = (g >> 1) ^ (g & 1): the two rows of a
// pair sit a multiple of 128 bytes apart, and the odd row's lanes taking the
// neighbouring slot of their even-row partners puts the eight lanes of every
// quarter-warp on 128 distinct bytes of bank space (no bank conflicts).  B column 2k carries the x of slot k and
// column 2k + 1 that of slot 4 + k, so the results of A-rows g and g + 8 land
// in lane (g, k), registers d[0] and d[3].
template <int DT, int NW, int SPW, int RP, int TW, int PF, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB) mbg_mmastage_kernel(const GemvArgs p)
{
    static_assert(DT == DT_Q8 || DT == DT_Q4, "quantised weights only");
    static_assert(NW >= 1 && NW <= 32, "block shape");
    constexpr int G = 2 * RP;                // rows per tile
    constexpr int XV = DT == DT_Q4 ? 4 : 2;  // 16-byte x vectors per 16-byte chunk of codes
    constexpr int ROWB = NW * SPW * 512;     // bytes per row
    constexpr int U = G * TW;                // rows per window
    constexpr int V = RP * TW;               // row-pair partials per lane and window
    constexpr int S = (PF + 1) * TW;         // stages
    static_assert(V == 1 || V == 2 || V == 4 || V == 8, "row pairs per window: 1, 2, 4 or 8");

    extern __shared__ __align__(128) unsigned char smem[];
    const StageBandLayout L = stageband_layout(S, U, NW, G, ROWB, p.groups, true);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    float *part = reinterpret_cast<float *>(smem + L.part);  // [2][U][NW]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int rsel = g & 1;                    // row of each pair this lane reads
    const int kslot = (g >> 1) ^ rsel;         // its slots: kslot and 4 + kslot
    const bool use = t == kslot;               // this lane holds its A-rows' results
    const int xslot = (g >> 1) + 4 * (g & 1);  // slot of x in B column g
    const int64_t grid = gridDim.x;
    const int64_t b = blockIdx.x;
    const int64_t ntiles = (p.M + G - 1) / G;
    const int I = static_cast<int>(b < ntiles ? (ntiles - 1 - b) / grid + 1 : 0);  // tiles b + i * grid
    const int64_t sgrp = p.groups;

    int issued = 0;  // thread 0: tiles whose copies have been issued
    auto issue = [&](int i) {
        const int s = i % S;
        const int64_t row0 = (b + i * grid) * G;
        const int64_t rows = p.M - row0 < G ? p.M - row0 : G;
        const uint32_t abytes = static_cast<uint32_t>(rows * ROWB);
        const uint32_t sbytes = static_cast<uint32_t>(rows * sgrp * 2);
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, abytes + sbytes);
        if (i == 0 && (p.skip_copies & SKIP_STAGE)) return;  // test hook: the wait must run out
        bulk_copy_g2s(smem_addr(smem + L.stage + s * L.stage_bytes),
                      static_cast<const unsigned char *>(p.A) + row0 * ROWB, abytes, bar);
        bulk_copy_g2s(smem_addr(smem + L.stage + s * L.stage_bytes + L.scale_off), p.scales + row0 * sgrp,
                      sbytes, bar);
    };

    pdl_trigger();
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_addr(&full[s]), 1);
        if (I > 0) {
            // the first tile into L2 while the preceding kernel drains (a hint)
            const int64_t row0 = b * G;
            const int64_t rows = p.M - row0 < G ? p.M - row0 : G;
            prefetch_l2(static_cast<const unsigned char *>(p.A) + row0 * ROWB, static_cast<uint32_t>(rows * ROWB));
        }
    }
    if (!p.pdl) pdl_wait();
    if (tid == 0)
        for (; issued < S && issued < I; ++issued) issue(issued);
    __syncthreads();  // barriers initialised before anyone waits on them
    if (p.pdl) pdl_wait();

    // B fragments: chunk t of x slot `xslot` of each of this lane's steps
    // (after the wait: the preceding kernel may have written x); INT4
    // re-paired four columns apart, the order in which the codes unpack
    uint4 xr[SPW][XV];
    {
        const unsigned char *xs = static_cast<const unsigned char *>(p.x);
#pragma unroll
        for (int s = 0; s < SPW; ++s) {
            const int64_t cbyte = static_cast<int64_t>(warp + s * NW) * 512 + xslot * 64 + t * 16;
            const int64_t col = DT == DT_Q4 ? cbyte * 2 : cbyte;
#pragma unroll
            for (int v = 0; v < XV; ++v) {
                xr[s][v] = ld_l2_16(xs + col * 2 + v * 16);
                if constexpr (DT == DT_Q4) xr[s][v] = pair_x_vec(xr[s][v]);
            }
        }
    }
    // shared-space offsets within a stage (row pair 0): this lane's chunk of
    // slot kslot of step s (slot 4 + kslot is 256 bytes further), its two scales
    const uint32_t stage0 = smem_addr(smem + L.stage);
    uint32_t aoff[SPW], soff[SPW][2];
#pragma unroll
    for (int s = 0; s < SPW; ++s) {
        const int slot0 = (warp + s * NW) * 8 + kslot;
        aoff[s] = static_cast<uint32_t>(rsel * ROWB + (warp + s * NW) * 512 + kslot * 64 + t * 16);
        soff[s][0] = static_cast<uint32_t>(L.scale_off + rsel * sgrp * 2 + ((slot0 * 4) >> p.scale_shift) * 2);
        soff[s][1] = static_cast<uint32_t>(L.scale_off + rsel * sgrp * 2 + (((slot0 + 4) * 4) >> p.scale_shift) * 2);
    }
    const uint32_t pair_a = 2u * ROWB;                          // next row pair's weights
    const uint32_t pair_s = static_cast<uint32_t>(4 * sgrp);    // and scales

    int half = 0;
    for (int i0 = 0; i0 < I; i0 += TW) {
        bool ok = true;
        float acc[V];
#pragma unroll
        for (int w = 0; w < TW; ++w) {
            const int i = i0 + w;
#pragma unroll
            for (int r = 0; r < RP; ++r) acc[w * RP + r] = 0.f;
            if (i < I) {
                const int s = i % S;
                ok &= mbar_wait_bounded(smem_addr(&full[s]), static_cast<uint32_t>((i / S) & 1), p.wait_limit_ns);
                const uint32_t st = stage0 + static_cast<uint32_t>(s) * L.stage_bytes;
                // a row past the end of A holds stale bytes: its sum is never stored
#pragma unroll
                for (int q = 0; q < SPW; ++q) {
#pragma unroll
                    for (int r = 0; r < RP; ++r) {
                        const uint4 a0 = lds128(st + aoff[q] + r * pair_a);
                        const uint4 a1 = lds128(st + aoff[q] + r * pair_a + 256);
                        float d[2][4];
                        mma_chunk_pair<DT>(a0, a1, xr[q], d);
                        const uint32_t sp = st + r * pair_s;
                        float &av = acc[w * RP + r];
                        av = fmaf(lds_half_as_float(sp + soff[q][0]), d[0][0] + d[1][0], av);
                        av = fmaf(lds_half_as_float(sp + soff[q][1]), d[0][3] + d[1][3], av);
                    }
                }
            }
        }
        // lanes that hold no result (their sums mix foreign slices) give 0
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = use ? acc[v] : 0.f;
        // value v of a lane: row 2 (v % RP) + rsel of tile v / RP of the window
        const float sum = mma_rows_sum<V>(acc, lane);
        if ((lane & mma_rows_rest<V>()) == 0) {
            const int v = mma_rows_tile<V>(lane);
            part[(half * U + (v / RP) * G + 2 * (v % RP) + rsel) * NW + warp] = sum;
        }
        // every thread has read the window's stages and written its partials;
        // a wait that gave up anywhere makes the whole block leave here
        if (__syncthreads_or(ok ? 0 : 1)) {
            if (tid == 0) {
                report_error(p.err, DEVERR_TIMEOUT);
                bool drained = true;
                for (int j = i0; j < issued; ++j) {
                    if (j == 0 && (p.skip_copies & SKIP_STAGE)) continue;  // never issued
                    drained &= mbar_wait_bounded(smem_addr(&full[j % S]), static_cast<uint32_t>((j / S) & 1),
                                                 p.wait_limit_ns);
                }
                if (!drained) report_error(p.err, DEVERR_UNDRAINED);
            }
            return;
        }
        if (tid == 0)
            for (; issued < i0 + S + TW && issued < I; ++issued) issue(issued);  // into the window's stages
        if (tid < U) {
            const int i = i0 + tid / G;
            const int64_t row = (b + static_cast<int64_t>(i) * grid) * G + tid % G;
            if (i < I && row < p.M) {
                float v = 0.f;
#pragma unroll
                for (int q = 0; q < NW; ++q) v += part[(half * U + tid) * NW + q];
                p.y[row] = v;
            }
        }
        half ^= 1;
    }
}

template <int DT, int G, int CPT, int T>
constexpr int tile_x_offset()
{
    return (16 + (G > 32 ? 2 * kTileBatch * (T / 32) * 4 : 0) + 15) / 16 * 16;
}

// Element weight (i, j) as FP32; the quantised types return FP32(s) * q,
// which is exact.
template <int DT>
__device__ __forceinline__ float elem_weight(const GemvArgs &p, int64_t i, int64_t j)
{
    const unsigned char *row = static_cast<const unsigned char *>(p.A) + i * p.row_bytes;
    if constexpr (DT == DT_F32) {
        return __ldg(reinterpret_cast<const float *>(row) + j);
    } else if constexpr (DT == DT_F16 || DT == DT_F16X32) {
        return ld_half_as_float(reinterpret_cast<const uint16_t *>(row) + j);
    } else {
        const float s = ld_half_as_float(p.scales + i * p.groups + (j >> p.scale_elem_shift));
        int q;
        if constexpr (DT == DT_Q8) {
            q = static_cast<int>(static_cast<signed char>(__ldg(reinterpret_cast<const char *>(row) + j)));
        } else {
            const unsigned b = __ldg(row + (j >> 1));
            const unsigned nib = (j & 1) ? (b >> 4) : (b & 0xFu);
            q = static_cast<int>(nib) - ((nib & 8u) ? 16 : 0);
        }
        return s * static_cast<float>(q);
    }
}

template <int DT>
__device__ __forceinline__ float elem_x(const GemvArgs &p, int64_t j)
{
    if constexpr (Fmt<DT>::XB == 4) return __ldg(static_cast<const float *>(p.x) + j);
    else return ld_half_as_float(static_cast<const uint16_t *>(p.x) + j);
}

template <int DT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) mbg_elem_kernel(const GemvArgs p)
{
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
    if (row >= p.M) return;  // whole warp leaves together
    float acc[NACC] = {0.f, 0.f, 0.f, 0.f};
    int k = 0;
    for (int64_t j = lane; j < p.N; j += 32, ++k) {
        acc[k & (NACC - 1)] = fmaf(elem_weight<DT>(p, row, j), elem_x<DT>(p, j), acc[k & (NACC - 1)]);
    }
    float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    s = group_sum<32>(s);
    if (lane == 0) p.y[row] = s;
}

// ---------------------------------------------------------------------------
// Variant-table glue
// ---------------------------------------------------------------------------

template <int DT, int LPR, int RPW, int U, int WARPS, int XMODE>
void launch_vec(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool)
{
    mbg_warprow_kernel<DT, LPR, RPW, U, WARPS, XMODE><<<grid, WARPS * 32, smem, s>>>(a);
}

template <int DT, int LPR, int RPW, int U, int WARPS, int XMODE>
cudaError_t smem_limit_vec(int bytes)
{
    return cudaFuncSetAttribute(mbg_warprow_kernel<DT, LPR, RPW, U, WARPS, XMODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DT, int WARPS>
void launch_elem(const GemvArgs &a, unsigned grid, size_t, cudaStream_t s, bool)
{
    mbg_elem_kernel<DT, WARPS><<<grid, WARPS * 32, 0, s>>>(a);
}

template <int DT, int WARPS>
cudaError_t smem_limit_elem(int)
{
    return cudaSuccess;
}

// Launch, optionally with programmatic stream serialisation (the kernel may
// start before the preceding kernel on the stream has finished).
template <typename Kernel>
void launch_maybe_pdl(Kernel k, const GemvArgs &a, unsigned grid, unsigned block, size_t smem,
                      cudaStream_t s, bool pdl)
{
    if (!pdl) {
        k<<<grid, block, smem, s>>>(a);
        return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, k, a);  // errors surface through cudaGetLastError
}

template <int DT, int G, int CPT, int T, int XMODE, int MATH>
void launch_tile(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool pdl)
{
    launch_maybe_pdl(mbg_rowtile_kernel<DT, G, CPT, T, XMODE, MATH>, a, grid, T, smem, s, pdl);
}

template <int DT, int G, int CPT, int T, int XMODE, int MATH>
cudaError_t smem_limit_tile(int bytes)
{
    return cudaFuncSetAttribute(mbg_rowtile_kernel<DT, G, CPT, T, XMODE, MATH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DT, int G, int CPT, int T, int XMODE, int MATH>
cudaError_t occupancy_tile(int *blocks, size_t smem)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks, mbg_rowtile_kernel<DT, G, CPT, T, XMODE, MATH>, T, smem);
}

#define MBG_TILE_M(DT, G, CPT, T, XM, MATH, NAME)                                              \
    Variant{DT, G, 1, CPT, T / 32, XM, NAME, &launch_tile<DT, G, CPT, T, XM, MATH>,             \
            &smem_limit_tile<DT, G, CPT, T, XM, MATH>, KIND_TILE, tile_x_offset<DT, G, CPT, T>(), \
            &occupancy_tile<DT, G, CPT, T, XM, MATH>, MATH, 0}
// An FP32 x uses FP32 arithmetic; binary16 x defaults to the mixed path.
#define MBG_TILE(DT, G, CPT, T, XM, NAME) \
    MBG_TILE_M(DT, G, CPT, T, XM, ((DT) == DT_F32 || (DT) == DT_F16X32 ? MATH_F32 : MATH_MIXED), NAME)

template <int DT, int T, int RS, int S, int MATH, int CF, bool XR>
void launch_bulk(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool pdl)
{
    launch_maybe_pdl(mbg_bulkpipe_kernel<DT, T, RS, S, MATH, CF, XR>, a, grid, T + 32, smem, s, pdl);
}

template <int DT, int T, int RS, int S, int MATH, int CF, bool XR>
cudaError_t smem_limit_bulk(int bytes)
{
    return cudaFuncSetAttribute(mbg_bulkpipe_kernel<DT, T, RS, S, MATH, CF, XR>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DT, int T, int RS, int S, int MATH, int CF, bool XR>
cudaError_t occupancy_bulk(int *blocks, size_t smem)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mbg_bulkpipe_kernel<DT, T, RS, S, MATH, CF, XR>,
                                                         T + 32, smem);
}

// unroll = CF: chunks per consumer thread and row when fixed (0: any row
// length); XR: x in registers (MBG_BULK_FX)
#define MBG_BULK_MFX(DT, T, RS, S, MATH, CF, XR, NAME)                                             \
    Variant{DT, T, RS, CF, T / 32, XMODE_BULK, NAME, &launch_bulk<DT, T, RS, S, MATH, CF, XR>,     \
            &smem_limit_bulk<DT, T, RS, S, MATH, CF, XR>, KIND_BULK, 0,                             \
            &occupancy_bulk<DT, T, RS, S, MATH, CF, XR>, MATH, S, XR}
#define MBG_BULK_MF(DT, T, RS, S, MATH, CF, NAME) MBG_BULK_MFX(DT, T, RS, S, MATH, CF, false, NAME)
#define MBG_BULK_M(DT, T, RS, S, MATH, NAME) MBG_BULK_MF(DT, T, RS, S, MATH, 0, NAME)
#define MBG_BULK(DT, T, RS, S, NAME) \
    MBG_BULK_M(DT, T, RS, S, ((DT) == DT_F32 || (DT) == DT_F16X32 ? MATH_F32 : MATH_MIXED), NAME)
#define MBG_BULK_F(DT, T, RS, S, CF, NAME) \
    MBG_BULK_MF(DT, T, RS, S, ((DT) == DT_F32 || (DT) == DT_F16X32 ? MATH_F32 : MATH_MIXED), CF, NAME)
#define MBG_BULK_FX(DT, T, RS, S, CF, NAME) MBG_BULK_MFX(DT, T, RS, S, MATH_MIXED, CF, true, NAME)

template <int DT, int T, int CPT, int G, int TW, int MINB>
void launch_band(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool pdl)
{
    launch_maybe_pdl(mbg_rowband_kernel<DT, T, CPT, G, TW, MINB>, a, grid, T, smem, s, pdl);
}

template <int DT, int T, int CPT, int G, int TW, int MINB>
cudaError_t smem_limit_band(int)
{
    return cudaSuccess;  // static shared memory only
}

template <int DT, int T, int CPT, int G, int TW, int MINB>
cudaError_t occupancy_band(int *blocks, size_t smem)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mbg_rowband_kernel<DT, T, CPT, G, TW, MINB>,
                                                         T, smem);
}

// band_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles in flight>:
// rows of exactly threads * chunks 16-byte chunks; x in registers
#define MBG_BAND_CAP(DT, T, CPT, G, TW, MINB, CAP, NAME)                                          \
    Variant{DT, T, (G) * (TW), CPT, T / 32, XMODE_REG, NAME, &launch_band<DT, T, CPT, G, TW, MINB>, \
            &smem_limit_band<DT, T, CPT, G, TW, MINB>, KIND_BAND, 0,                               \
            &occupancy_band<DT, T, CPT, G, TW, MINB>,                                               \
            ((DT) == DT_F32 || (DT) == DT_F16X32) ? MATH_F32 : MATH_MIXED, 0, false, G, CAP}
#define MBG_BAND(DT, T, CPT, G, TW, MINB, NAME) MBG_BAND_CAP(DT, T, CPT, G, TW, MINB, 0, NAME)

template <int DT, int NW, int SPW, int TW, int MINB, bool RC>
void launch_mmaband(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool pdl)
{
    launch_maybe_pdl(mbg_mmaband_kernel<DT, NW, SPW, TW, MINB, RC>, a, grid, NW * 32, smem, s, pdl);
}

template <int DT, int NW, int SPW, int TW, int MINB, bool RC>
cudaError_t smem_limit_mmaband(int)
{
    return cudaSuccess;  // static shared memory only
}

template <int DT, int NW, int SPW, int TW, int MINB, bool RC>
cudaError_t occupancy_mmaband(int *blocks, size_t smem)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mbg_mmaband_kernel<DT, NW, SPW, TW, MINB, RC>,
                                                         NW * 32, smem);
}

// mma_w<warps>_s<steps per warp>_t<tiles in flight>_m<min blocks per SM>[_rc]:
// rows of exactly warps * steps * 512 bytes; x in registers; products on the
// MMA unit; _rc: each load instruction of a warp reads 512 contiguous bytes of
// one row
#define MBG_MMA_L(DT, NW, SPW, TW, MINB, RC, NAME)                                                         \
    Variant{DT, (NW) * 32, 2 * (TW), SPW, NW, XMODE_REG, NAME, &launch_mmaband<DT, NW, SPW, TW, MINB, RC>, \
            &smem_limit_mmaband<DT, NW, SPW, TW, MINB, RC>, KIND_MMA, 0,                                   \
            &occupancy_mmaband<DT, NW, SPW, TW, MINB, RC>, MATH_MIXED, 0, false, 2, 0,                  \
            ((DT) == DT_Q4 && !(RC)) ? 4 : 2}
#define MBG_MMA(DT, NW, SPW, TW, MINB, NAME) MBG_MMA_L(DT, NW, SPW, TW, MINB, false, NAME)

template <int DT, int T, int CPT, int G, int TW, int PF, int MINB>
void launch_stageband(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool pdl)
{
    launch_maybe_pdl(mbg_stageband_kernel<DT, T, CPT, G, TW, PF, MINB>, a, grid, T, smem, s, pdl);
}

template <int DT, int T, int CPT, int G, int TW, int PF, int MINB>
cudaError_t smem_limit_stageband(int bytes)
{
    return cudaFuncSetAttribute(mbg_stageband_kernel<DT, T, CPT, G, TW, PF, MINB>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DT, int T, int CPT, int G, int TW, int PF, int MINB>
cudaError_t occupancy_stageband(int *blocks, size_t smem)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mbg_stageband_kernel<DT, T, CPT, G, TW, PF, MINB>,
                                                         T, smem);
}

// sband_t<threads>_c<chunks per thread>_g<rows per tile>_w<tiles per window>_p<windows
// in flight>: rows of exactly threads * chunks 16-byte chunks; x in registers;
// (p + 1) w stages
#define MBG_SBAND(DT, T, CPT, G, TW, PF, MINB, NAME)                                                   \
    Variant{DT, T, (G) * (TW), CPT, T / 32, XMODE_REG, NAME,                                          \
            &launch_stageband<DT, T, CPT, G, TW, PF, MINB>, &smem_limit_stageband<DT, T, CPT, G, TW, PF, MINB>, \
            KIND_SBAND, 0, &occupancy_stageband<DT, T, CPT, G, TW, PF, MINB>,                           \
            (DT) == DT_F32 ? MATH_F32 : MATH_MIXED, ((PF) + 1) * (TW), false, G}

template <int DT, int NW, int SPW, int RP, int TW, int PF, int MINB>
void launch_mmastage(const GemvArgs &a, unsigned grid, size_t smem, cudaStream_t s, bool pdl)
{
    launch_maybe_pdl(mbg_mmastage_kernel<DT, NW, SPW, RP, TW, PF, MINB>, a, grid, NW * 32, smem, s, pdl);
}

template <int DT, int NW, int SPW, int RP, int TW, int PF, int MINB>
cudaError_t smem_limit_mmastage(int bytes)
{
    return cudaFuncSetAttribute(mbg_mmastage_kernel<DT, NW, SPW, RP, TW, PF, MINB>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DT, int NW, int SPW, int RP, int TW, int PF, int MINB>
cudaError_t occupancy_mmastage(int *blocks, size_t smem)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks, mbg_mmastage_kernel<DT, NW, SPW, RP, TW, PF, MINB>, NW * 32, smem);
}

// smma_w<warps>_s<steps per warp>_r<row pairs per tile>_t<tiles per
// window>_p<windows in flight>_m<min blocks per SM>: rows of exactly warps *
// steps * 512 bytes; (p + 1) t stages of 2 r rows and their scales
#define MBG_SMMA(DT, NW, SPW, RP, TW, PF, MINB, NAME)                                                     \
    Variant{DT, (NW) * 32, 2 * (RP) * (TW), SPW, NW, XMODE_REG, NAME,                                    \
            &launch_mmastage<DT, NW, SPW, RP, TW, PF, MINB>, &smem_limit_mmastage<DT, NW, SPW, RP, TW, PF, MINB>, \
            KIND_SMMA, 0, &occupancy_mmastage<DT, NW, SPW, RP, TW, PF, MINB>, MATH_MIXED, ((PF) + 1) * (TW),  \
            false, 2 * (RP), 0}

#define MBG_VEC(DT, LPR, RPW, U, W, XM, NAME)                                              \
    Variant{DT, LPR, RPW, U, W, XM, NAME, &launch_vec<DT, LPR, RPW, U, W, XM>,              \
            &smem_limit_vec<DT, LPR, RPW, U, W, XM>, KIND_VEC, 16, nullptr, MATH_F32, 0}
#define MBG_ELEM(DT, W, NAME) \
    Variant{DT, 32, 1, 1, W, XMODE_ELEM, NAME, &launch_elem<DT, W>, &smem_limit_elem<DT, W>, \
            KIND_ELEM, 0, nullptr, MATH_F32, 0}

}  // namespace mbg
