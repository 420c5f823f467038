// Dequantisation to FP32 with the GEMV kernels' own unpacking code (the
// binary16 codes of the mixed-precision path), so that comparing its output
// bit for bit with the oracle's q * s checks that code
// ("membound", section "dequant GEMV": the reference is computed on the
// dequantised weights, q * s exactly).  Also the N == 0 fill.
#include "gemv_kernels.cuh"

namespace mbg {

// One thread per 16-byte chunk (vector layout) -> EPC outputs.
template <int DT>
__global__ void mbg_dequant_vec_kernel(const unsigned char *A, const uint16_t *scales, float *W,
                                   int64_t M, int64_t N, int64_t row_bytes, int64_t groups)
{
    constexpr int EPC = Fmt<DT>::EPC;
    const int64_t nchunks = row_bytes / 16;
    const int64_t total = M * nchunks;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < total;
         k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = k / nchunks;
        const int64_t c = k - i * nchunks;
        const uint4 a = ld_stream16(A + i * row_bytes + c * 16);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
        float wf[EPC];
        // the binary16 codes of the mixed-precision GEMV path, widened exactly
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (DT == DT_Q8) {
                uint32_t h[2];
                q8_codes_h2(w[k], h);
                half2_bits_to_float(h[0], wf[4 * k + 0], wf[4 * k + 1]);
                half2_bits_to_float(h[1], wf[4 * k + 2], wf[4 * k + 3]);
            } else {
                uint32_t h[4];
                q4_codes_h2(w[k], h);
                half2_bits_to_float(h[0], wf[8 * k + 0], wf[8 * k + 4]);
                half2_bits_to_float(h[1], wf[8 * k + 1], wf[8 * k + 5]);
                half2_bits_to_float(h[2], wf[8 * k + 2], wf[8 * k + 6]);
                half2_bits_to_float(h[3], wf[8 * k + 3], wf[8 * k + 7]);
            }
        }
        const float s = ld_half_as_float(scales + i * groups + (c * EPC) / kGroup);
        float *out = W + i * N + c * EPC;
#pragma unroll
        for (int e = 0; e < EPC; ++e) out[e] = wf[e] * s;
    }
}

// One thread per element (any layout).
template <int DT>
__global__ void mbg_dequant_elem_kernel(GemvArgs p, float *W)
{
    const int64_t total = p.M * p.N;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < total;
         k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = k / p.N;
        W[k] = elem_weight<DT>(p, i, k - i * p.N);
    }
}

static unsigned grid_for(int64_t work, int threads)
{
    int64_t g = (work + threads - 1) / threads;
    if (g > 65535LL * 16) g = 65535LL * 16;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

void launch_dequant(int dtype, const void *A, const uint16_t *scales, float *W, int64_t M,
                    int64_t N, bool vec, cudaStream_t s)
{
    const int64_t row_bytes = dtype == DT_Q4 ? N / 2 : N;
    const int64_t groups = (N + kGroup - 1) / kGroup;
    const auto *a = static_cast<const unsigned char *>(A);
    if (vec) {
        const unsigned g = grid_for(M * (row_bytes / 16), 256);
        if (dtype == DT_Q8) mbg_dequant_vec_kernel<DT_Q8><<<g, 256, 0, s>>>(a, scales, W, M, N, row_bytes, groups);
        else mbg_dequant_vec_kernel<DT_Q4><<<g, 256, 0, s>>>(a, scales, W, M, N, row_bytes, groups);
    } else {
        GemvArgs p{};
        p.A = A;
        p.scales = scales;
        p.M = M;
        p.N = N;
        p.row_bytes = row_bytes;
        p.groups = groups;
        p.scale_elem_shift = 7;  // 128 columns per scale
        const unsigned g = grid_for(M * N, 256);
        if (dtype == DT_Q8) mbg_dequant_elem_kernel<DT_Q8><<<g, 256, 0, s>>>(p, W);
        else mbg_dequant_elem_kernel<DT_Q4><<<g, 256, 0, s>>>(p, W);
    }
}

__global__ void mbg_fill_zero_kernel(float *y, int64_t M)
{
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < M;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        y[i] = 0.0f;
}

void launch_fill_zero(float *y, int64_t M, cudaStream_t s)
{
    mbg_fill_zero_kernel<<<grid_for(M, 256), 256, 0, s>>>(y, M);
}

}  // namespace mbg
