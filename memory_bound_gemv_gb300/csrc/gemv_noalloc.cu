// gemv_ex_host without a caller-provided device buffer for x.
//
// Some callers cannot allocate device memory when they need a GEMV: code
// that runs after start-up under a rule of no further allocations (real-time
// or safety-checked loops), plug-ins that live inside a host program which
// owns the device allocator and gives them none, and callers that reach this
// library only through its C ABI with no CUDA allocation routine at hand.
// For them the device copy of x lives in this file: one fixed array per GPU,
// loaded with the library and held until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gemv.h"

namespace {

// Device copy of x for gemv_ex_host_noalloc (GEMV_NOALLOC_X_MAX_BYTES).
static __device__ __align__(256) unsigned char g_noalloc_x[GEMV_NOALLOC_X_MAX_BYTES];

constexpr int kMaxNoAllocDevices = 64;

struct NoAllocDevice {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void *x = nullptr;  // device address of g_noalloc_x on this device
};

NoAllocDevice g_noalloc_devices[kMaxNoAllocDevices];

// Device address of the array on the current device, looked up once per
// device (with that device current); nullptr on failure.
void *noalloc_x_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices) return nullptr;
    NoAllocDevice &d = g_noalloc_devices[dev];
    std::call_once(d.once, [&d] {
        d.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.x), g_noalloc_x);
    });
    return d.err == cudaSuccess ? d.x : nullptr;
}

}  // namespace

extern "C" gemv_status_t gemv_ex_host_noalloc(int dtype, const void *A, const void *x_host,
                                              float *y_host, int64_t M, int64_t N,
                                              const uint16_t *scales, unsigned flags, void *stream)
{
    const int64_t x_bytes = (dtype == GEMV_F32 || dtype == GEMV_F16_X32) ? 4 : 2;
    if (N > GEMV_NOALLOC_X_MAX_BYTES / x_bytes) return GEMV_ERR_UNSUPPORTED;
    void *x_dev = noalloc_x_address();
    if (!x_dev) return GEMV_ERR_CUDA;
    return gemv_ex_host(dtype, A, x_host, x_dev, y_host, M, N, scales, flags, stream);
}
