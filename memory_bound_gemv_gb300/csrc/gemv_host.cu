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
#include "gemv_kernels.cuh"

namespace mbg {

namespace {

__global__ void __launch_bounds__(256) copy_in_kernel(const unsigned char *src, unsigned char *dst,
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

}  // namespace

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
    (void)cudaLaunchKernelEx(&cfg, copy_in_kernel, sp, dp, bytes, vec ? 1 : 0, early ? 1 : 0);
}

}  // namespace mbg
