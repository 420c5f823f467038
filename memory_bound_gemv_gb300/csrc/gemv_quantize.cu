// Symmetric weight quantisation to the INT8 / INT4 operands of the GEMV
// ("membound", section "The kernel decode actually runs: dequant GEMV": INT8
// with a symmetric scale per row, INT4 with a symmetric scale per group of 128
// columns; the quantisation RMSE reported there for U[-1,1] weights, 2.3e-3
// and 4.1e-2, fixes the scales as max|w| / 127 and max|w| / 7).
//
// One warp per (row, group), FP32 arithmetic:
//   a = max |w|, s = a / qmax (IEEE division), s16 = binary16(s) rounded to
//   nearest even (+inf replaced by 65504), q = clamp(rint(w / s16), +-qmax),
//   q = 0 where s16 == 0 or w is NaN.
// The squared error (w - s16 q)^2 is summed in double, per warp, then per
// block, and added to *sq_err with one atomic per block.
#include "gemv_kernels.cuh"

namespace mbg {

namespace {

struct QuantArgs {
    const void *W;
    void *A;
    uint16_t *scales;
    double *sq_err;
    int64_t M, N;
    int64_t width;   // columns per group (128, or N for one scale per row)
    int64_t groups;  // groups per row
};

template <bool F16IN>
__device__ __forceinline__ float load_w(const QuantArgs &p, int64_t k)
{
    if constexpr (F16IN)
        return __half2float(__ushort_as_half(__ldg(static_cast<const unsigned short *>(p.W) + k)));
    else
        return __ldg(static_cast<const float *>(p.W) + k);
}

template <int QMAX, bool F16IN, bool PACK4>
__global__ void __launch_bounds__(256) mbg_quantize_kernel(const QuantArgs p)
{
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t items = p.M * p.groups;
    double err = 0.0;
    for (int64_t item = warp_id; item < items; item += nwarps) {
        const int64_t i = item / p.groups;
        const int64_t g = item - i * p.groups;
        const int64_t j0 = g * p.width;
        const int64_t j1 = min(j0 + p.width, p.N);
        const int64_t row = i * p.N;
        // group maximum of |w| (a NaN never compares greater, so it is skipped)
        float a = 0.f;
        for (int64_t j = j0 + lane; j < j1; j += 32) {
            const float m = fabsf(load_w<F16IN>(p, row + j));
            a = m > a ? m : a;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(full, a, off);
            a = o > a ? o : a;
        }
        const float s = __fdiv_rn(a, static_cast<float>(QMAX));
        unsigned short s16 = __half_as_ushort(__float2half_rn(s));
        if (s16 == 0x7C00u) s16 = 0x7BFFu;
        const float sf = __half2float(__ushort_as_half(s16));
        if (lane == 0) p.scales[i * p.groups + g] = s16;
        for (int64_t base = j0; base < j1; base += 32) {
            const int64_t j = base + lane;
            int code = 0;
            if (j < j1) {
                const float w = load_w<F16IN>(p, row + j);
                if (sf != 0.f && w == w) {
                    float q = rintf(__fdiv_rn(w, sf));
                    q = fminf(fmaxf(q, -static_cast<float>(QMAX)), static_cast<float>(QMAX));
                    code = static_cast<int>(q);
                }
                const double d = static_cast<double>(w) - static_cast<double>(sf) * code;
                err += d * d;
            }
            if constexpr (PACK4) {
                // even column in the low nibble: the even lane writes the byte
                const int odd = __shfl_down_sync(full, code, 1);
                if (!(lane & 1) && j < j1)
                    static_cast<uint8_t *>(p.A)[i * (p.N / 2) + j / 2] =
                        static_cast<uint8_t>((code & 0xF) | ((odd & 0xF) << 4));
            } else if (j < j1) {
                static_cast<int8_t *>(p.A)[row + j] = static_cast<int8_t>(code);
            }
        }
    }
    if (p.sq_err) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) err += __shfl_xor_sync(full, err, off);
        __shared__ double part[8];
        if (lane == 0) part[threadIdx.x >> 5] = err;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += part[w];
            atomicAdd(p.sq_err, t);
        }
    }
}

template <int QMAX, bool PACK4>
void launch_q(const QuantArgs &p, bool f16in, unsigned blocks, cudaStream_t s)
{
    if (f16in) mbg_quantize_kernel<QMAX, true, PACK4><<<blocks, 256, 0, s>>>(p);
    else mbg_quantize_kernel<QMAX, false, PACK4><<<blocks, 256, 0, s>>>(p);
}

}  // namespace

void launch_quantize(int bits, bool per_row, bool f16in, const void *W, void *A, uint16_t *scales,
                     double *sq_err, int64_t M, int64_t N, int sm_count, cudaStream_t s)
{
    QuantArgs p{};
    p.W = W;
    p.A = A;
    p.scales = scales;
    p.sq_err = sq_err;
    p.M = M;
    p.N = N;
    p.width = per_row ? N : kGroup;
    p.groups = per_row ? 1 : (N + kGroup - 1) / kGroup;
    const int64_t warps = M * p.groups;
    int64_t blocks = (warps + 7) / 8;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (bits == 8) launch_q<127, false>(p, f16in, static_cast<unsigned>(blocks), s);
    else launch_q<7, true>(p, f16in, static_cast<unsigned>(blocks), s);
}

}  // namespace mbg
