// Pure-read bandwidth probe ("membound", section "Why GEMV, and why MBU": the
// read ceiling measured on the same card is the denominator for a GEMV,
// whose traffic is almost all reads).
//
// The probe uses the GEMV kernels' load instruction (16-byte, read-only, L1
// no-allocate, 256-byte L2 fetch) and their rolling buffer of U loads in
// flight per lane.  Three read patterns:
//   segment: each warp streams one contiguous stretch of the buffer with its
//            lanes 16 bytes apart -- the access pattern of a warp-per-row GEMV;
//   stride:  blocks walk tiles of THREADS*U vectors in grid-stride order;
//   tile:    the row-tile GEMV's pattern: a persistent grid walks tiles of
//            THREADS*U vectors in grid-stride order and requests the next tile
//            before folding the current one;
//   bulk:    bulk async copies (cp.async.bulk) of large chunks into
//            shared-memory rings -- the bulk pipeline's way of reading weights
//            (measured a little above the load-based patterns).
// Every loaded word is XOR-folded; each warp XORs its fold into *sink, so no
// load can be dropped as dead code.
#include "gemv_device.cuh"

namespace mbg {

template <int THREADS, int U, int SEGMENT>
__global__ void __launch_bounds__(THREADS) mbg_probe_read_kernel(const uint4 *buf, size_t n16,
                                                             unsigned long long *sink)
{
    uint32_t fold = 0;
    const int lane = threadIdx.x & 31;
    if constexpr (SEGMENT) {
        const size_t warps = static_cast<size_t>(gridDim.x) * (THREADS / 32);
        const size_t w = static_cast<size_t>(blockIdx.x) * (THREADS / 32) + (threadIdx.x >> 5);
        size_t seg = (n16 + warps - 1) / warps;
        seg = (seg + 31) & ~static_cast<size_t>(31);
        const size_t begin = w * seg;
        const size_t end = begin + seg < n16 ? begin + seg : n16;
        if (begin < end) {
            const uint4 *base = buf + begin;
            const size_t n = end - begin;
            uint4 b[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t c = lane + static_cast<size_t>(u) * 32;
                if (c < n) b[u] = ld_stream16(base + c);
            }
            for (size_t c0 = lane; c0 < n; c0 += 32 * U) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const size_t c = c0 + static_cast<size_t>(u) * 32;
                    if (c < n) {
                        const uint4 v = b[u];
                        const size_t cn = c + 32 * U;
                        if (cn < n) b[u] = ld_stream16(base + cn);
                        fold ^= v.x ^ v.y ^ v.z ^ v.w;
                    }
                }
            }
        }
    } else {
        const size_t tile = static_cast<size_t>(THREADS) * U;
        const size_t step = static_cast<size_t>(gridDim.x) * tile;
        for (size_t t0 = static_cast<size_t>(blockIdx.x) * tile; t0 < n16; t0 += step) {
            uint4 b[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t c = t0 + static_cast<size_t>(u) * THREADS + threadIdx.x;
                b[u] = c < n16 ? ld_stream16(buf + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) fold ^= b[u].x ^ b[u].y ^ b[u].z ^ b[u].w;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) fold ^= __shfl_xor_sync(0xffffffffu, fold, off);
    if (lane == 0 && fold) atomicXor(sink, static_cast<unsigned long long>(fold));
}

template <int THREADS, int U>
__global__ void __launch_bounds__(THREADS) mbg_probe_tile_kernel(const uint4 *buf, size_t n16,
                                                             unsigned long long *sink)
{
    uint32_t fold = 0;
    const size_t tile = static_cast<size_t>(THREADS) * U;
    const size_t ntiles = (n16 + tile - 1) / tile;
    uint4 cur[U], nxt[U];
    auto load = [&](size_t t, uint4 (&b)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t c = t * tile + static_cast<size_t>(u) * THREADS + threadIdx.x;
            b[u] = c < n16 ? ld_stream16(buf + c) : make_uint4(0, 0, 0, 0);
        }
    };
    size_t t = blockIdx.x;
    if (t < ntiles) load(t, cur);
    for (; t < ntiles; t += gridDim.x) {
        if (t + gridDim.x < ntiles) load(t + gridDim.x, nxt);
#pragma unroll
        for (int u = 0; u < U; ++u) fold ^= cur[u].x ^ cur[u].y ^ cur[u].z ^ cur[u].w;
#pragma unroll
        for (int u = 0; u < U; ++u) cur[u] = nxt[u];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) fold ^= __shfl_xor_sync(0xffffffffu, fold, off);
    if ((threadIdx.x & 31) == 0 && fold) atomicXor(sink, static_cast<unsigned long long>(fold));
}

// Bulk-copy read probe: one warp per block streams chunks of B bytes (grid-
// stride order) through an S-deep ring of shared-memory stages with
// cp.async.bulk, waits on each stage's mbarrier (bounded), and XOR-folds the
// chunk before the stage is refilled.  On a timeout it waits (bounded) for the
// copies still in flight and sets bit 63 of *sink, and bit 62 as well if that
// wait gave up too.  skip_first (test hook): the first chunk's barrier is
// armed but no copy is issued, so its wait runs out.
template <int B, int S>
__global__ void __launch_bounds__(32) mbg_probe_bulk_kernel(const uint4 *buf, size_t n16,
                                                        unsigned long long *sink, uint64_t limit_ns,
                                                        int skip_first)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + 128;
    const int lane = threadIdx.x & 31;
    const size_t nbytes = n16 * 16;
    const size_t nchunks = (nbytes + B - 1) / B;
    const size_t grid = gridDim.x;
    const size_t iters = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / grid + 1 : 0;
    if (lane == 0)
        for (int s = 0; s < S; ++s) mbar_init(smem_addr(&bar[s]), 1);
    __syncwarp();
    auto chunk_bytes = [&](size_t k) {
        const size_t off = (blockIdx.x + k * grid) * static_cast<size_t>(B);
        return static_cast<uint32_t>(nbytes - off < static_cast<size_t>(B) ? nbytes - off : B);
    };
    auto issue = [&](size_t k) {
        if (lane == 0) {
            const uint32_t b = smem_addr(&bar[k % S]);
            const uint32_t n = chunk_bytes(k);
            mbar_arrive_expect_tx(b, n);
            if (k == 0 && skip_first) return;
            bulk_copy_g2s(smem_addr(ring + (k % S) * B),
                          reinterpret_cast<const unsigned char *>(buf) + (blockIdx.x + k * grid) * static_cast<size_t>(B),
                          n, b);
        }
    };
    size_t issued = 0;
    for (; issued < S && issued < iters; ++issued) issue(issued);
    uint32_t fold = 0;
    bool ok = true;
    size_t k = 0;
    for (; k < iters; ++k) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(smem_addr(&bar[k % S]), static_cast<uint32_t>((k / S) & 1), limit_ns));
        if (!ok) break;
        const uint4 *r = reinterpret_cast<const uint4 *>(ring + (k % S) * B);
        const uint32_t n = chunk_bytes(k) / 16;
        for (uint32_t i = lane; i < n; i += 32) {
            const uint4 v = r[i];
            fold ^= v.x ^ v.y ^ v.z ^ v.w;
        }
        __syncwarp();  // every lane has read the stage before it is refilled
        if (issued < iters) issue(issued++);
    }
    if (!ok) {
        if (lane == 0) {
            bool drained = true;
            for (size_t j = k; j < issued; ++j) {
                if (j == 0 && skip_first) continue;  // never issued
                drained &= mbar_wait_bounded(smem_addr(&bar[j % S]), static_cast<uint32_t>((j / S) & 1), limit_ns);
            }
            atomicOr(sink, drained ? (1ull << 63) : (3ull << 62));
        }
        return;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) fold ^= __shfl_xor_sync(0xffffffffu, fold, off);
    if (lane == 0 && fold) atomicXor(sink, static_cast<unsigned long long>(fold));
}

template <int B, int S>
void launch_probe_bulk(const void *buf, size_t n16, unsigned long long *sink, unsigned grid,
                       uint64_t limit_ns, bool skip_first, cudaStream_t s)
{
    const int smem = 128 + S * B;
    cudaFuncSetAttribute(mbg_probe_bulk_kernel<B, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    mbg_probe_bulk_kernel<B, S><<<grid, 32, smem, s>>>(static_cast<const uint4 *>(buf), n16, sink, limit_ns,
                                                       skip_first ? 1 : 0);
}

template <int THREADS, int U>
void launch_probe_tile(const void *buf, size_t n16, unsigned long long *sink, unsigned grid,
                       uint64_t, bool, cudaStream_t s)
{
    mbg_probe_tile_kernel<THREADS, U><<<grid, THREADS, 0, s>>>(static_cast<const uint4 *>(buf), n16, sink);
}

template <int THREADS, int U, int SEGMENT>
void launch_probe(const void *buf, size_t n16, unsigned long long *sink, unsigned grid,
                  uint64_t, bool, cudaStream_t s)
{
    mbg_probe_read_kernel<THREADS, U, SEGMENT>
        <<<grid, THREADS, 0, s>>>(static_cast<const uint4 *>(buf), n16, sink);
}

// pattern field: 0 grid-stride tiles, 1 one segment per warp, 2 tiles with
// the next requested early, 3 bulk copies (threads 32, unroll = stages)
static const ProbeVariant kProbes[] = {
    {"segment_t128_u8_b8", 128, 8, 8, 1, &launch_probe<128, 8, 1>},
    {"segment_t256_u8_b4", 256, 8, 4, 1, &launch_probe<256, 8, 1>},
    {"segment_t128_u16_b6", 128, 16, 6, 1, &launch_probe<128, 16, 1>},
    {"stride_t256_u8_b4", 256, 8, 4, 0, &launch_probe<256, 8, 0>},
    {"stride_t512_u4_b4", 512, 4, 4, 0, &launch_probe<512, 4, 0>},
    {"stride_t256_u16_b4", 256, 16, 4, 0, &launch_probe<256, 16, 0>},
    {"tile_t256_u8_b2", 256, 8, 2, 2, &launch_probe_tile<256, 8>},
    {"tile_t512_u4_b2", 512, 4, 2, 2, &launch_probe_tile<512, 4>},
    {"tile_t256_u8_b4", 256, 8, 4, 2, &launch_probe_tile<256, 8>},
    {"tile_t512_u8_b1", 512, 8, 1, 2, &launch_probe_tile<512, 8>},
    {"bulk_b32k_s2_x2", 32, 2, 2, 3, &launch_probe_bulk<32768, 2>},
    {"bulk_b32k_s4_x1", 32, 4, 1, 3, &launch_probe_bulk<32768, 4>},
    {"bulk_b16k_s4_x2", 32, 4, 2, 3, &launch_probe_bulk<16384, 4>},
};

const ProbeVariant *probe_variants(int *count)
{
    *count = static_cast<int>(sizeof(kProbes) / sizeof(kProbes[0]));
    return kProbes;
}

}  // namespace mbg
