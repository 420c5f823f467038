// x from page-locked host memory into device memory, as a kernel.
//
// On a GB300 the GPU reads page-locked host memory directly over the
// coherent CPU-GPU link, so the input vector of a host-side call can be
// fetched by a few blocks instead of a DMA copy.  Being a kernel, the copy
// takes part in programmatic dependent launch: it is always launched with
// programmatic stream serialisation (its blocks are scheduled while the
// preceding kernel drains) and waits for that kernel before it touches any
// memory; when the caller allows it (early), it reads x before that wait and
// only writes the device buffer after it.  The GEMV after it starts
// streaming its weights while x is still in flight.
//
// Ordering.  The copy lets the GEMV after it start at once, and the GEMV
// orders itself after the copy with its own wait (griddepcontrol.wait), which
// returns only once the copy grid has completed -- and the copy completes
// only after its own wait for the kernel before the call.  Unless the caller
// has promised that the kernel before the call leaves the weights, scales and
// x alone (early), the GEMV therefore touches no memory before that wait
// (only L2 prefetch hints); with the promise it streams its weights at once
// and reads x after the wait.
#include "gemv_kernels.cuh"

namespace mbg {

namespace {

__global__ void __launch_bounds__(256) mbg_copy_in_kernel(const unsigned char *src, unsigned char *dst,
                                                      int64_t bytes, int vec, int early)
{
    pdl_trigger();
    if (!early) pdl_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t n16 = vec ? bytes / 16 : 0;
    const uint4 *s16 = reinterpret_cast<const uint4 *>(src);
    uint4 *d16 = reinterpret_cast<uint4 *>(dst);
    // first vector read (before the wait for the preceding kernel when early),
    // written after it
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    const bool have = t0 < n16;
    if (have) v = s16[t0];
    pdl_wait();
    if (have) d16[t0] = v;
    for (int64_t i = t0 + stride; i < n16; i += stride) d16[i] = s16[i];
    for (int64_t b = n16 * 16 + t0; b < bytes; b += stride) dst[b] = src[b];
}

// Test helper: lets the next kernel start at once, then after delay_ns
// fills dst with a 32-bit pattern (a preceding kernel that writes a GEMV's
// operands late).  The delay is a spin on the global timer that ends by
// itself.
__global__ void __launch_bounds__(256) mbg_late_fill_kernel(uint32_t *dst, size_t words, uint32_t word,
                                                            uint64_t delay_ns)
{
    pdl_trigger();
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < delay_ns) {
    }
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words; i += stride)
        dst[i] = word;
}

}  // namespace

void launch_late_fill(void *dst, size_t bytes, uint32_t word, uint64_t delay_ns, cudaStream_t s)
{
    const size_t words = bytes / 4;
    size_t blocks = (words + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    mbg_late_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<uint32_t *>(dst), words,
                                                                        word, delay_ns);
}

void launch_copy_in(const void *src, void *dst, int64_t bytes, bool early, cudaStream_t s)
{
    const bool vec = (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
    const int64_t units = vec ? (bytes + 15) / 16 : bytes;
    int64_t blocks = (units + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    const auto *sp = static_cast<const unsigned char *>(src);
    auto *dp = static_cast<unsigned char *>(dst);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, mbg_copy_in_kernel, sp, dp, bytes, vec ? 1 : 0, early ? 1 : 0);
}

}  // namespace mbg
