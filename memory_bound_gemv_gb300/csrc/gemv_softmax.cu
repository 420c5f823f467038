// Row softmax of binary16 data ("membound", section "Bonus kernel: online
// softmax": y_j = exp(x_j - m) / sum_k exp(x_k - m) with m the row maximum,
// combined with the online update m' = max(m, m2), d' = d e^(m - m') +
// d2 e^(m2 - m')), and a copy probe for its read + write ceiling.
//
// mbg_softmax_vec_kernel: a row is read once into registers (16-byte loads; the
// persistent grid loads the next row while it finishes the current one), each
// thread keeps exp(x_j - m_t) for its own maximum m_t and its partial sum,
// the (max, sum) pairs are combined across the warp, the block and -- for
// rows wider than one block holds -- the thread-block cluster through
// distributed shared memory, and the row is written once.  HBM traffic is one
// read and one write per element (the page's version re-reads the row through
// L2 for a second pass; with the row in registers there is no second read).
//
// mbg_softmax_cluster_kernel: the same single read and write, with the row segments
// staged by bulk async copies into a ring of shared-memory buffers instead of
// register prefetch, so a persistent grid of blocks (or clusters) keeps the
// next rows in flight without spending registers on them.  Each thread keeps
// exp(x - m_t) for its own maximum; the (max, sum) pairs meet in one
// exchange per row (one barrier of the block or cluster), which also frees
// the row's buffer for the next copy.
//
// mbg_softmax_elem_kernel: any layout or length.  One block per row, the page's
// two passes: the online update over the row, then exp(x - m) / d re-reading
// the row.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <mutex>

#include "gemv_device.cuh"

namespace cg = cooperative_groups;

namespace mbg {

// e^t computed as 2^(t log2 e) by the ex2.approx instruction (PTX ISA: at
// most 2^-22 relative error; results below the FP32 normal range flush to
// zero, far below anything a binary16 output can hold).  t = x - m is formed
// first, so the scaling never multiplies a large |m| on its own.
__device__ __forceinline__ float exp_approx(float t)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t * 1.4426950408889634f));
    return r;
}

// (m, d) pairs: running maximum and sum of exp(x - m).  An empty side has
// m = -inf and d = 0.
struct MaxSum {
    float m, d;
};

__device__ __forceinline__ MaxSum combine(MaxSum a, MaxSum b)
{
    if (a.m == -INFINITY) return b;
    if (b.m == -INFINITY) return a;
    const float m = fmaxf(a.m, b.m);
    return {m, a.d * exp_approx(a.m - m) + b.d * exp_approx(b.m - m)};
}

// (max, sum) over a warp: the maximum first, then every lane's sum rescaled
// to it once and added up (one exponential per lane instead of one per
// butterfly level).
__device__ __forceinline__ MaxSum warp_combine(MaxSum v)
{
    float m = v.m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float d = (v.m == -INFINITY) ? 0.f : v.d * exp_approx(v.m - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    return {m, d};
}

// Combine over the block; every thread receives the result.  `red` holds at
// least 33 MaxSum entries of shared memory.
template <int T>
__device__ __forceinline__ MaxSum block_combine(MaxSum v, MaxSum *red)
{
    constexpr int NW = T / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_combine(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        MaxSum w = lane < NW ? red[lane] : MaxSum{-INFINITY, 0.f};
        w = warp_combine(w);
        if (lane == 0) red[32] = w;
    }
    __syncthreads();
    return red[32];
}

__device__ __forceinline__ void st_stream16(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Two floats -> binary16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// C CTAs (a cluster) per row, T threads per CTA, EPT elements per thread.
// Requires N % 8 == 0, 16-byte aligned x and y, and N <= C * T * EPT.
// Cluster k handles rows k, k + nclusters, ... and loads its segment of the
// next row into registers before it reduces and writes the current one, so a
// persistent grid keeps reads in flight while it finishes a row.  All CTAs of
// a cluster walk the same rows, so they meet the same cluster barriers.
template <int T, int EPT, int C>
__global__ void __launch_bounds__(T) mbg_softmax_vec_kernel(const uint16_t *x, uint16_t *y, int64_t M, int N)
{
    constexpr int VPT = EPT / 8;  // 16-byte vectors per thread
    __shared__ MaxSum red[33];
    __shared__ MaxSum cta_result;

    const int tid = threadIdx.x;
    const int rank = C > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int64_t nclusters = gridDim.x / C;
    const int seg = rank * T * EPT;

    auto load = [&](int64_t row, uint4 (&raw)[VPT]) {
        const uint16_t *xr = x + row * N;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int e0 = seg + 8 * (k * T + tid);
            raw[k] = e0 < N ? ld_stream16(xr + e0) : make_uint4(0, 0, 0, 0);
        }
    };

    // Only single-block rows prefetch (a persistent grid); the extra registers
    // would halve the occupancy of the cluster variants, which run one
    // cluster per row instead.
    constexpr bool PREFETCH = C == 1;
    uint4 nxt[PREFETCH ? VPT : 1];
    int64_t row = blockIdx.x / C;
    if constexpr (PREFETCH) {
        if (row < M) load(row, nxt);
    }
    for (; row < M; row += nclusters) {
        uint4 raw[VPT];
        if constexpr (PREFETCH) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) raw[k] = nxt[k];
            if (row + nclusters < M) load(row + nclusters, nxt);
        } else {
            load(row, raw);
        }

        float v[EPT];
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int e0 = seg + 8 * (k * T + tid);
            half2_bits_to_float(raw[k].x, v[8 * k + 0], v[8 * k + 1]);
            half2_bits_to_float(raw[k].y, v[8 * k + 2], v[8 * k + 3]);
            half2_bits_to_float(raw[k].z, v[8 * k + 4], v[8 * k + 5]);
            half2_bits_to_float(raw[k].w, v[8 * k + 6], v[8 * k + 7]);
            if (e0 < N) {
#pragma unroll
                for (int e = 0; e < 8; ++e) m = fmaxf(m, v[8 * k + e]);
            }
        }
        // e_j = exp(x_j - m_t) for this thread's maximum; kept for the output
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int e0 = seg + 8 * (k * T + tid);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[8 * k + e] = e0 < N ? exp_approx(v[8 * k + e] - m) : 0.f;
                d += v[8 * k + e];
            }
        }
        MaxSum mine{m, d};
        if (m == -INFINITY) mine = {-INFINITY, 0.f};
        MaxSum tot = block_combine<T>(mine, red);

        if constexpr (C > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            if (tid == 0) cta_result = tot;
            cluster.sync();  // every CTA's partial is written
            MaxSum all{-INFINITY, 0.f};
#pragma unroll
            for (int r = 0; r < C; ++r) all = combine(all, *cluster.map_shared_rank(&cta_result, r));
            cluster.sync();  // no CTA moves on while another still reads its partial
            tot = all;
        }

        const float scale = (mine.m == -INFINITY) ? 0.f : exp_approx(mine.m - tot.m) / tot.d;
        uint16_t *yr = y + row * N;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int e0 = seg + 8 * (k * T + tid);
            if (e0 < N) {
                uint4 o;
                o.x = pack_half2(v[8 * k + 0] * scale, v[8 * k + 1] * scale);
                o.y = pack_half2(v[8 * k + 2] * scale, v[8 * k + 3] * scale);
                o.z = pack_half2(v[8 * k + 4] * scale, v[8 * k + 5] * scale);
                o.w = pack_half2(v[8 * k + 6] * scale, v[8 * k + 7] * scale);
                st_stream16(yr + e0, o);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy staged rows
// ---------------------------------------------------------------------------

// Max or sum of one value per thread over the block (C == 1) or the cluster:
// warp butterfly, then lane 0 of each warp writes its value into slot
// [rank * NW + warp] of every block of the cluster, one barrier, and every
// warp reduces the C * NW slots in the same order (all blocks get the same
// bits).
template <int T, int C, bool MAX>
__device__ __forceinline__ float row_reduce(float v, float *slots, int rank)
{
    constexpr int NW = T / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = MAX ? fmaxf(v, o) : v + o;
    }
    if (lane == 0) {
        if constexpr (C == 1) {
            slots[warp] = v;
        } else {
            cg::cluster_group cluster = cg::this_cluster();
#pragma unroll
            for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&slots[rank * NW + warp], r) = v;
        }
    }
    if constexpr (C == 1) __syncthreads();
    else cg::this_cluster().sync();
    float w = MAX ? -INFINITY : 0.f;
    for (int i = lane; i < C * NW; i += 32) w = MAX ? fmaxf(w, slots[i]) : w + slots[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, w, off);
        w = MAX ? fmaxf(w, o) : w + o;
    }
    return w;
}

// (max, sum) of the row from one pair per thread: inside a warp the maximum
// first, then the sums rescaled to it; lane 0 of each warp writes the warp's
// pair into slot [rank * NW + warp] of every block of the cluster; one barrier
// (of the block, or of the cluster); then every warp combines the C * NW pairs
// in the same order, so all blocks of a cluster get the same bits.  A side
// with no elements has m = -inf and d = 0.
template <int T, int C>
__device__ __forceinline__ MaxSum row_exchange(MaxSum v, float2 *slots, int rank)
{
    constexpr int NW = T / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float m = v.m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float d = (v.m == -INFINITY) ? 0.f : v.d * exp_approx(v.m - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) {
        const float2 pr = make_float2(m, d);
        if constexpr (C == 1) {
            slots[warp] = pr;
        } else {
            cg::cluster_group cluster = cg::this_cluster();
#pragma unroll
            for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&slots[rank * NW + warp], r) = pr;
        }
    }
    if constexpr (C == 1) __syncthreads();
    else cg::this_cluster().sync();
    constexpr int PER = (C * NW + 31) / 32;
    float2 e[PER];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int idx = lane + 32 * k;
        e[k] = idx < C * NW ? slots[idx] : make_float2(-INFINITY, 0.f);
        M = fmaxf(M, e[k].x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float D = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k)
        if (e[k].x != -INFINITY) D += e[k].y * exp_approx(e[k].x - M);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) D += __shfl_xor_sync(0xffffffffu, D, off);
    return {M, D};
}

__host__ __device__ constexpr int softmax_bulk_smem(int T, int EPT, int C, int NB)
{
    // NB row-segment buffers, NB mbarriers + the abort flag, slots [2 rows][C * T/32] of
    // (max, sum) pairs (or of a max and a sum)
    return NB * T * EPT * 2 + NB * 8 + 16 + 2 * C * (T / 32) * 8;
}

// C blocks (a cluster) per row, T threads per block, EPT elements per thread,
// NB staged rows per block.  PAIR: one exchange of (max, sum) pairs per row;
// else the row maximum first, then the sum of exp(x - max) (two barriers, but
// fewer live registers across them).  Requires N % 8 == 0, 16-byte aligned x and y and
// N <= C * T * EPT.  Cluster k handles rows k, k + nclusters, ...; its blocks
// walk the same rows and meet the same barriers.  A wait that gives up sets
// the status word and the block's abort flag; the block then runs on without
// writing y, so that the barriers of the cluster still match.
template <int T, int EPT, int C, int NB, bool PAIR>
__global__ void __launch_bounds__(T) mbg_softmax_cluster_kernel(const uint16_t *x, uint16_t *y, int64_t M, int N,
                                                         unsigned int *err, uint64_t wait_limit_ns,
                                                         unsigned int skip)
{
    constexpr int VPT = EPT / 8;
    constexpr int NW = T / 32;
    constexpr int SEGE = T * EPT;  // elements of a block's segment
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *bufs = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + NB * SEGE * 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + NB);
    float2 *slots = reinterpret_cast<float2 *>(smem + NB * SEGE * 2 + NB * 8 + 16);

    const int tid = threadIdx.x;
    const int rank = C > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int64_t cid = blockIdx.x / C;
    const int64_t ncl = gridDim.x / C;
    const int seg0 = rank * SEGE;
    const int segn = N - seg0 < 0 ? 0 : (N - seg0 < SEGE ? N - seg0 : SEGE);
    const uint32_t seg_bytes = static_cast<uint32_t>(segn) * 2u;

    if (tid == 0) {
        for (int b = 0; b < NB; ++b) mbar_init(smem_addr(&full[b]), 1);
        *abort_flag = 0;
    }
    __syncthreads();
    if constexpr (C > 1) cg::this_cluster().sync();  // every block of the cluster has started

    // thread 0 issues the copies and remembers, per buffer, the phase of a
    // copy not yet waited for (only needed when the block gives up)
    uint32_t issued[NB], pending[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) issued[b] = pending[b] = 0;
    auto issue = [&](int64_t row, int b, bool skip_copy) {
        const uint32_t bar = smem_addr(&full[b]);
        mbar_arrive_expect_tx(bar, seg_bytes);
        ++issued[b];
        if (skip_copy) return;  // test hook: armed, never filled, so the wait runs out
        bulk_copy_g2s(smem_addr(bufs + b * SEGE * 2), x + row * N + seg0, seg_bytes, bar);
        pending[b] = 1;
    };
    if (tid == 0 && seg_bytes) {
        for (int b = 0; b < NB; ++b) {
            const int64_t row = cid + b * ncl;
            if (row < M) issue(row, b, b == 0 && (skip & SKIP_SEGMENT));
        }
    }

    int64_t i = 0;
    for (int64_t row = cid; row < M; row += ncl, ++i) {
        const int b = static_cast<int>(i % NB);
        if (seg_bytes && !*abort_flag) {
            if (mbar_wait_bounded(smem_addr(&full[b]), static_cast<uint32_t>((i / NB) & 1), wait_limit_ns)) {
                if (tid == 0) pending[b] = 0;
            } else {
                report_error(err, DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        // this block's segment into registers; -inf beyond the row end
        uint4 raw[VPT];
        const uint32_t bb = smem_addr(bufs + b * SEGE * 2);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int e0 = seg0 + 8 * (k * T + tid);
            raw[k] = e0 < N ? lds128(bb + (k * T + tid) * 16) : make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);
        }
        if constexpr (!PAIR) {
            // every thread has read buffer b: refill it with a later row
            __syncthreads();
            if (tid == 0 && seg_bytes && !*abort_flag && row + NB * ncl < M) issue(row + NB * ncl, b, false);
        }
        // this thread's maximum (on binary16 pairs, then one conversion)
        __half2 hm = __halves2half2(__ushort_as_half(0xFC00u), __ushort_as_half(0xFC00u));
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            hm = __hmax2(hm, *reinterpret_cast<const __half2 *>(&raw[k].x));
            hm = __hmax2(hm, *reinterpret_cast<const __half2 *>(&raw[k].y));
            hm = __hmax2(hm, *reinterpret_cast<const __half2 *>(&raw[k].z));
            hm = __hmax2(hm, *reinterpret_cast<const __half2 *>(&raw[k].w));
        }
        const float mt = fmaxf(__low2float(hm), __high2float(hm));
        float *sl = reinterpret_cast<float *>(slots + static_cast<int>(i & 1) * (C * NW));
        float m = mt;  // the maximum the exponentials are taken against
        if constexpr (!PAIR) m = row_reduce<T, C, true>(mt, sl, rank);

        // exp(x - m) kept for the output, and its sum
        float e[EPT];
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            half2_bits_to_float(raw[k].x, e[8 * k + 0], e[8 * k + 1]);
            half2_bits_to_float(raw[k].y, e[8 * k + 2], e[8 * k + 3]);
            half2_bits_to_float(raw[k].z, e[8 * k + 4], e[8 * k + 5]);
            half2_bits_to_float(raw[k].w, e[8 * k + 6], e[8 * k + 7]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                e[8 * k + j] = PAIR && m == -INFINITY ? 0.f : exp_approx(e[8 * k + j] - m);
                d += e[8 * k + j];
            }
        }
        float inv;
        if constexpr (PAIR) {
            // one exchange per row; after it every thread has read buffer b
            const MaxSum tot = row_exchange<T, C>(MaxSum{mt, d}, slots + static_cast<int>(i & 1) * (C * NW), rank);
            if (tid == 0 && seg_bytes && !*abort_flag && row + NB * ncl < M) issue(row + NB * ncl, b, false);
            inv = (mt == -INFINITY) ? 0.f : exp_approx(mt - tot.m) / tot.d;
        } else {
            inv = 1.f / row_reduce<T, C, false>(d, sl + C * NW, rank);
        }
        const bool aborted = *abort_flag != 0;
        if (!aborted) {
            uint16_t *yr = y + row * N;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int e0 = seg0 + 8 * (k * T + tid);
                if (e0 < N) {
                    uint4 o;
                    o.x = pack_half2(e[8 * k + 0] * inv, e[8 * k + 1] * inv);
                    o.y = pack_half2(e[8 * k + 2] * inv, e[8 * k + 3] * inv);
                    o.z = pack_half2(e[8 * k + 4] * inv, e[8 * k + 5] * inv);
                    o.w = pack_half2(e[8 * k + 6] * inv, e[8 * k + 7] * inv);
                    st_stream16(yr + e0, o);
                }
            }
        }
    }
    if (tid == 0 && *abort_flag) {
        // copies issued for rows this block did not take may still land
        bool drained = true;
#pragma unroll
        for (int b = 0; b < NB; ++b)
            if (pending[b]) drained &= mbar_wait_bounded(smem_addr(&full[b]), (issued[b] - 1) & 1u, wait_limit_ns);
        if (!drained) report_error(err, DEVERR_UNDRAINED);
    }
}

// Any layout, any length: one block per row, two passes over the row.
template <int T>
__global__ void __launch_bounds__(T) mbg_softmax_elem_kernel(const uint16_t *x, uint16_t *y, int64_t N)
{
    __shared__ MaxSum red[33];
    const int64_t row = blockIdx.x;
    const uint16_t *xr = x + row * N;
    uint16_t *yr = y + row * N;
    MaxSum acc{-INFINITY, 0.f};
    for (int64_t j = threadIdx.x; j < N; j += T) {
        const float v = ld_half_as_float(xr + j);
        if (v == -INFINITY) continue;  // contributes exp(-inf) = 0
        if (v > acc.m) {
            acc.d = acc.d * exp_approx(acc.m - v) + 1.f;  // acc.m = -inf gives 0 * 0
            acc.m = v;
        } else {
            acc.d += exp_approx(v - acc.m);
        }
    }
    const MaxSum tot = block_combine<T>(acc, red);
    const float inv = 1.f / tot.d;
    for (int64_t j = threadIdx.x; j < N; j += T) {
        const float v = ld_half_as_float(xr + j);
        reinterpret_cast<__half *>(yr)[j] = __float2half_rn(exp_approx(v - tot.m) * inv);
    }
}

// ---------------------------------------------------------------------------
// Copy probe (read + write ceiling)
// ---------------------------------------------------------------------------

template <int THREADS, int U>
__global__ void __launch_bounds__(THREADS) mbg_probe_copy_kernel(const uint4 *src, uint4 *dst, size_t n16)
{
    const size_t tile = static_cast<size_t>(THREADS) * U;
    for (size_t t0 = static_cast<size_t>(blockIdx.x) * tile; t0 < n16; t0 += static_cast<size_t>(gridDim.x) * tile) {
        uint4 b[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t c = t0 + static_cast<size_t>(u) * THREADS + threadIdx.x;
            if (c < n16) b[u] = ld_stream16(src + c);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t c = t0 + static_cast<size_t>(u) * THREADS + threadIdx.x;
            if (c < n16) st_stream16(dst + c, b[u]);
        }
    }
}

// ---------------------------------------------------------------------------
// Launch glue
// ---------------------------------------------------------------------------

// A value computed once per device (with that device current): launch set-up
// such as shared-memory limits and persistent grid sizes, which belong to the
// device's context.  0 when the device index is out of range.
constexpr int kSoftmaxMaxDevices = 64;

template <typename F>
int per_device_once(std::once_flag (&once)[kSoftmaxMaxDevices], int (&val)[kSoftmaxMaxDevices], F compute)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSoftmaxMaxDevices) return 0;
    std::call_once(once[dev], [&] { val[dev] = compute(dev); });
    return val[dev];
}

template <int T, int EPT, int C>
int count_resident_clusters(int dev)
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int n = 0;
    if constexpr (C == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mbg_softmax_vec_kernel<T, EPT, 1>, T, 0) ==
            cudaSuccess)
            n = per_sm * sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * sms);
        cfg.blockDim = dim3(T);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, mbg_softmax_vec_kernel<T, EPT, C>, &cfg) != cudaSuccess) n = 0;
    }
    return n > 0 ? n : sms;
}

// Resident clusters (of C blocks) for this kernel: the persistent grid size.
template <int T, int EPT, int C>
int resident_clusters()
{
    static std::once_flag once[kSoftmaxMaxDevices];
    static int val[kSoftmaxMaxDevices];
    return per_device_once(once, val, [](int dev) { return count_resident_clusters<T, EPT, C>(dev); });
}

template <int T, int EPT, int C>
cudaError_t launch_softmax_vec(const uint16_t *x, uint16_t *y, int64_t M, int N, cudaStream_t s)
{
    // single-block rows: a persistent grid that prefetches the next row;
    // cluster rows: one cluster per row (measured faster: the scheduler keeps
    // more clusters in flight than a persistent grid of resident clusters)
    int64_t clusters = M;
    if constexpr (C == 1) clusters = M < resident_clusters<T, EPT, C>() ? M : resident_clusters<T, EPT, C>();
    const unsigned grid = static_cast<unsigned>(clusters * C);
    if constexpr (C == 1) {
        mbg_softmax_vec_kernel<T, EPT, 1><<<grid, T, 0, s>>>(x, y, M, N);
        return cudaGetLastError();
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(T);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, mbg_softmax_vec_kernel<T, EPT, C>, x, y, M, N);
    }
}

// Persistent grid of the bulk-staged kernel: resident clusters (of C
// blocks), at most one per row.
template <int T, int EPT, int C, int NB, bool PAIR>
cudaError_t launch_softmax_bulk(const uint16_t *x, uint16_t *y, int64_t M, int N, unsigned int *err,
                                uint64_t wait_limit_ns, unsigned int skip, cudaStream_t s)
{
    constexpr int SMEM = softmax_bulk_smem(T, EPT, C, NB);
    static std::once_flag once[kSoftmaxMaxDevices];
    static int val[kSoftmaxMaxDevices];
    const int resident = per_device_once(once, val, [](int dev) {
        // raise the dynamic shared memory limit once per device, then ask for the occupancy
        if (cudaFuncSetAttribute(mbg_softmax_cluster_kernel<T, EPT, C, NB, PAIR>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
            return 0;
        int sms = 0, n = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if constexpr (C == 1) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mbg_softmax_cluster_kernel<T, EPT, 1, NB, PAIR>, T,
                                                              SMEM) != cudaSuccess)
                return 0;
            return n * sms;
        } else {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(C * sms);
            cfg.blockDim = dim3(T);
            cfg.dynamicSmemBytes = SMEM;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = C;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, mbg_softmax_cluster_kernel<T, EPT, C, NB, PAIR>, &cfg) != cudaSuccess)
                return 0;
            return n;
        }
    });
    if (resident <= 0) return cudaErrorNotSupported;
    const int64_t clusters = M < resident ? M : resident;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * C));
    cfg.blockDim = dim3(T);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mbg_softmax_cluster_kernel<T, EPT, C, NB, PAIR>, x, y, M, N, err, wait_limit_ns,
                              skip);
}

template <int T, int EPT, int C>
cudaError_t launch_softmax_vec_v(const uint16_t *x, uint16_t *y, int64_t M, int N, unsigned int *,
                                 uint64_t, unsigned int, cudaStream_t s)
{
    return launch_softmax_vec<T, EPT, C>(x, y, M, N, s);
}

struct SoftmaxVariant {
    int threads, ept, cluster;
    const char *name;
    cudaError_t (*launch)(const uint16_t *, uint16_t *, int64_t, int, unsigned int *, uint64_t,
                          unsigned int, cudaStream_t);
    int capacity() const { return threads * ept * cluster; }
};

// The automatic choice is the first entry whose capacity covers the row.
static const SoftmaxVariant kSoftmax[] = {
    // the automatic choice, by capacity (each measured fastest for its widths);
    // smb_: rows staged by bulk copies, t<threads>_e<elements per thread>_c<cluster>
    // _b<staged rows>, _p: one (max, sum) exchange per row instead of a max then a sum;
    // sm_: rows held in registers with a register prefetch of the next row
    {128, 8, 1, "sm_t128_e8_c1", &launch_softmax_vec_v<128, 8, 1>},
    {256, 16, 1, "sm_t256_e16_c1", &launch_softmax_vec_v<256, 16, 1>},
    {256, 32, 1, "sm_t256_e32_c1", &launch_softmax_vec_v<256, 32, 1>},
    {512, 32, 1, "sm_t512_e32_c1", &launch_softmax_vec_v<512, 32, 1>},
    {512, 32, 2, "smb_t512_e32_c2_b2_p", &launch_softmax_bulk<512, 32, 2, 2, true>},
    {512, 32, 4, "smb_t512_e32_c4_b2_p", &launch_softmax_bulk<512, 32, 4, 2, true>},
    {512, 32, 8, "smb_t512_e32_c8_b2_p", &launch_softmax_bulk<512, 32, 8, 2, true>},
    // alternatives
    {128, 8, 1, "smb_t128_e8_c1_b3", &launch_softmax_bulk<128, 8, 1, 3, false>},
    {256, 16, 1, "smb_t256_e16_c1_b3", &launch_softmax_bulk<256, 16, 1, 3, false>},
    {256, 32, 1, "smb_t256_e32_c1_b2", &launch_softmax_bulk<256, 32, 1, 2, false>},
    {256, 32, 1, "smb_t256_e32_c1_b2_p", &launch_softmax_bulk<256, 32, 1, 2, true>},
    {512, 32, 1, "smb_t512_e32_c1_b2", &launch_softmax_bulk<512, 32, 1, 2, false>},
    {256, 32, 4, "smb_t256_e32_c4_b2_p", &launch_softmax_bulk<256, 32, 4, 2, true>},
    {512, 32, 8, "smb_t512_e32_c8_b2", &launch_softmax_bulk<512, 32, 8, 2, false>},
    {512, 32, 8, "smb_t512_e32_c8_b3_p", &launch_softmax_bulk<512, 32, 8, 3, true>},
    {512, 32, 2, "sm_t512_e32_c2", &launch_softmax_vec_v<512, 32, 2>},
    {512, 32, 8, "sm_t512_e32_c8", &launch_softmax_vec_v<512, 32, 8>},
};
constexpr int kSoftmaxVariants = static_cast<int>(sizeof(kSoftmax) / sizeof(kSoftmax[0]));

int softmax_variant_count() { return kSoftmaxVariants + 1; }

const char *softmax_variant_name(int v)
{
    if (v >= 0 && v < kSoftmaxVariants) return kSoftmax[v].name;
    return v == kSoftmaxVariants ? "sm_elem_t256" : nullptr;
}

// Chooses (variant < 0) or runs a given variant; returns a CUDA error, or
// cudaErrorNotSupported when the variant cannot serve the shape.
cudaError_t launch_softmax(const uint16_t *x, uint16_t *y, int64_t M, int64_t N, int variant,
                           unsigned int *err, uint64_t wait_limit_ns, unsigned int skip,
                           cudaStream_t s)
{
    const bool vec_ok = N % 8 == 0 && N <= (1 << 30) &&
                        (reinterpret_cast<uintptr_t>(x) % 16) == 0 &&
                        (reinterpret_cast<uintptr_t>(y) % 16) == 0;
    if (variant < 0) {
        variant = kSoftmaxVariants;
        if (vec_ok) {
            for (int k = 0; k < kSoftmaxVariants; ++k) {
                if (kSoftmax[k].capacity() >= N) {
                    variant = k;
                    break;
                }
            }
        }
    }
    if (variant < kSoftmaxVariants) {
        const SoftmaxVariant &v = kSoftmax[variant];
        if (!vec_ok || N > v.capacity()) return cudaErrorNotSupported;
        return v.launch(x, y, M, static_cast<int>(N), err, wait_limit_ns, skip, s);
    }
    if (M > 0x7fffffffLL) return cudaErrorNotSupported;
    mbg_softmax_elem_kernel<256><<<static_cast<unsigned>(M), 256, 0, s>>>(x, y, N);
    return cudaGetLastError();
}

struct CopyVariant {
    const char *name;
    int blocks_per_sm;
    void (*launch)(const void *, void *, size_t, unsigned, cudaStream_t);
};

template <int THREADS, int U>
void launch_copy(const void *src, void *dst, size_t n16, unsigned grid, cudaStream_t s)
{
    mbg_probe_copy_kernel<THREADS, U>
        <<<grid, THREADS, 0, s>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
}

static const CopyVariant kCopy[] = {
    {"copy_t256_u4_b4", 4, &launch_copy<256, 4>},
    {"copy_t256_u8_b4", 4, &launch_copy<256, 8>},
    {"copy_t512_u4_b2", 2, &launch_copy<512, 4>},
    {"copy_t256_u8_b2", 2, &launch_copy<256, 8>},
};

int copy_variant_count() { return static_cast<int>(sizeof(kCopy) / sizeof(kCopy[0])); }
const char *copy_variant_name(int v) { return (v >= 0 && v < copy_variant_count()) ? kCopy[v].name : nullptr; }

cudaError_t launch_copy_probe(const void *src, void *dst, size_t bytes, int variant, int sm_count,
                              cudaStream_t s)
{
    const CopyVariant &c = kCopy[variant];
    c.launch(src, dst, bytes / 16, static_cast<unsigned>(sm_count * c.blocks_per_sm), s);
    return cudaGetLastError();
}

}  // namespace mbg
