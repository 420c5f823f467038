// Symmetric weight quantisation to the INT8 / INT4 operands of the GEMV
// ("membound", section "The kernel decode actually runs: dequant GEMV": INT8
// with a symmetric scale per row, INT4 with a symmetric scale per group of 128
// columns; the quantisation RMSE reported there for U[-1,1] weights, 2.3e-3
// and 4.1e-2, fixes the scales as max|w| / 127 and max|w| / 7).
//
// FP32 arithmetic for every weight of a group:
//   a = max |w|, s = a / qmax (IEEE division), s16 = binary16(s) rounded to
//   nearest even (+inf replaced by 65504), q = clamp(rint(w / s16), +-qmax),
//   q = 0 where s16 == 0 or w is NaN.
// The squared error (w - s16 q)^2 is summed in double, per thread, then per
// block, and added to *sq_err with one atomic per block; kernels launched
// without an error sum do none of that arithmetic.
//
// Kernels: groups of 128 columns with 16-byte aligned weights take one
// half-warp per group with the group's weights held in registers (read
// once); one scale per row takes one block per row (the row maximum, then
// the codes from a second read of the row, which L2 still holds); any other
// layout takes one warp per (row, group) with 2- or 4-byte loads.
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

// The code of one weight (the rule above; IEEE division, so that the codes
// are those of the definition bit for bit).
template <int QMAX>
__device__ __forceinline__ int quant_code(float w, float sf)
{
    if (!(sf != 0.f && w == w)) return 0;
    float q = rintf(__fdiv_rn(w, sf));
    q = fminf(fmaxf(q, -static_cast<float>(QMAX)), static_cast<float>(QMAX));
    return static_cast<int>(q);
}

// binary16 scale of a group maximum (+inf replaced by 65504)
template <int QMAX>
__device__ __forceinline__ unsigned short scale_bits(float a)
{
    unsigned short s16 = __half_as_ushort(__float2half_rn(__fdiv_rn(a, static_cast<float>(QMAX))));
    return s16 == 0x7C00u ? static_cast<unsigned short>(0x7BFFu) : s16;
}

// FP32 -> FP64, exact: a normal number by re-biasing its exponent (1023 -
// 127 = 896) and moving its significand with integer operations, which keeps
// the (slow) FP64 pipe for the accumulation; zero, subnormal, infinite and
// NaN values take the conversion instruction.
__device__ __forceinline__ double widen_exact(float f)
{
    const uint32_t u = __float_as_uint(f);
    const uint32_t e = u & 0x7F800000u;
    if (e == 0u || e == 0x7F800000u) return static_cast<double>(f);
    const uint32_t hi = (u & 0x80000000u) | (((u >> 3) & 0x0FFFFFFFu) + (896u << 20));
    return __hiloint2double(static_cast<int>(hi), static_cast<int>(u << 29));
}

// err += (w - sf q)^2 with the residual exact: in FP32 when q == 0 or
// |w| <= 2 |sf q| (sf q is exact, 11 x 8 significant bits, and has the sign
// of w; |q| >= 1 puts |w| >= |sf q| / 2, so Sterbenz's lemma makes the
// difference exact), else in double as written; its square is exact in
// double (48 significant bits), so one fused multiply-add adds it.
__device__ __forceinline__ void add_sq_err(double &err, float w, float sf, int code)
{
    const float pr = sf * static_cast<float>(code);
    if (code == 0 || fabsf(w) <= 2.f * fabsf(pr)) {
        const double d = widen_exact(w - pr);
        err = fma(d, d, err);
    } else {
        const double d = static_cast<double>(w) - static_cast<double>(sf) * code;
        err = fma(d, d, err);
    }
}

// Eight consecutive weights (16-byte aligned) as floats; binary16 widens exactly.
template <bool F16IN>
__device__ __forceinline__ void load8(const void *W, int64_t k, float (&w)[8])
{
    if constexpr (F16IN) {
        const uint4 v = ld_stream16(static_cast<const uint16_t *>(W) + k);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[c]));
            w[2 * c] = f.x;
            w[2 * c + 1] = f.y;
        }
    } else {
        const float *f = static_cast<const float *>(W) + k;
        const uint4 v0 = ld_stream16(f), v1 = ld_stream16(f + 4);
        const uint32_t u[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) w[c] = __uint_as_float(u[c]);
    }
}

// Stores the eight codes of weights k .. k + 7 (INT8: 8 bytes; INT4: 4
// bytes, the even column in the low nibble).
template <bool PACK4>
__device__ __forceinline__ void store8(void *A, int64_t k, const int (&c)[8])
{
    if constexpr (PACK4) {
        uint32_t v = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) v |= static_cast<uint32_t>(c[j] & 0xF) << (4 * j);
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(A) + k / 2) = v;
    } else {
        uint32_t lo = 0u, hi = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo |= static_cast<uint32_t>(c[j] & 0xFF) << (8 * j);
            hi |= static_cast<uint32_t>(c[4 + j] & 0xFF) << (8 * j);
        }
        *reinterpret_cast<uint2 *>(static_cast<int8_t *>(A) + k) = make_uint2(lo, hi);
    }
}

__device__ __forceinline__ void add_block_err(double err, double *sq_err)
{
    const unsigned full = 0xffffffffu;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) err += __shfl_xor_sync(full, err, off);
    __shared__ double part[8];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = err;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += part[w];
        atomicAdd(sq_err, t);
    }
}

// Groups of exactly 128 columns (N a multiple of 128), 16-byte aligned W:
// group k of the row-major sequence is W[128 k .. 128 k + 127], handled by
// one half-warp whose lane l holds weights 8 l .. 8 l + 7 of it.  In each
// pass a warp takes 2 UNROLL consecutive groups (group 2 u + h of its run to
// half-warp h, u < UNROLL) and issues all their loads first; consecutive
// warps take consecutive runs, so a pass of the grid reads one contiguous
// span of W.
template <int QMAX, bool F16IN, bool PACK4, bool ERR, int UNROLL>
__global__ void __launch_bounds__(256) mbg_quantize_vec_kernel(const QuantArgs p)
{
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31, hl = lane & 15, h = lane >> 4;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t items = p.M * p.groups;
    double err[2] = {0.0, 0.0};  // two chains of fused multiply-adds
    for (int64_t base = warp_id * 2 * UNROLL; base < items; base += nwarps * 2 * UNROLL) {
        float w[UNROLL][8];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t item = base + 2 * u + h;
            if (item < items) {
                load8<F16IN>(p.W, item * 128 + hl * 8, w[u]);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) w[u][c] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t item = base + 2 * u + h;
            // group maximum of |w| (a NaN never compares greater, so it is skipped)
            float a = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float m = fabsf(w[u][c]);
                a = m > a ? m : a;
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) {
                const float o = __shfl_xor_sync(full, a, off);
                a = o > a ? o : a;
            }
            const unsigned short s16 = scale_bits<QMAX>(a);
            const float sf = __half2float(__ushort_as_half(s16));
            if (item < items) {
                if (hl == 0) p.scales[item] = s16;
                int code[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    code[c] = quant_code<QMAX>(w[u][c], sf);
                    if constexpr (ERR) add_sq_err(err[c & 1], w[u][c], sf, code[c]);
                }
                store8<PACK4>(p.A, item * 128 + hl * 8, code);
            }
        }
    }
    if constexpr (ERR) add_block_err(err[0] + err[1], p.sq_err);
}

// One INT8 scale per row, N a multiple of 8, 16-byte aligned W: a block per
// row (grid-stride), 16-byte loads of eight weights; the row maximum, a
// block reduction, then the codes from a second read of the row.
template <bool F16IN, bool ERR>
__global__ void __launch_bounds__(256) mbg_quantize_row_kernel(const QuantArgs p)
{
    const unsigned full = 0xffffffffu;
    constexpr int QMAX = 127;
    __shared__ float red[2][8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t chunks = p.N / 8;
    double err[2] = {0.0, 0.0};  // two chains of fused multiply-adds
    int buf = 0;
    for (int64_t i = blockIdx.x; i < p.M; i += gridDim.x) {
        const int64_t row = i * p.N;
        float a = 0.f;
#pragma unroll 4
        for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
            float w[8];
            load8<F16IN>(p.W, row + c * 8, w);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float m = fabsf(w[j]);
                a = m > a ? m : a;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(full, a, off);
            a = o > a ? o : a;
        }
        // two buffers: the next row's partial maxima never overwrite ones
        // that a slow thread is still reading
        if (lane == 0) red[buf][warp] = a;
        __syncthreads();
        a = 0.f;
        for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) a = red[buf][k] > a ? red[buf][k] : a;
        buf ^= 1;
        const unsigned short s16 = scale_bits<QMAX>(a);
        const float sf = __half2float(__ushort_as_half(s16));
        if (threadIdx.x == 0) p.scales[i] = s16;
        for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
            float w[8];
            load8<F16IN>(p.W, row + c * 8, w);
            int code[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                code[j] = quant_code<QMAX>(w[j], sf);
                if constexpr (ERR) add_sq_err(err[j & 1], w[j], sf, code[j]);
            }
            store8<false>(p.A, row + c * 8, code);
        }
    }
    if constexpr (ERR) add_block_err(err[0] + err[1], p.sq_err);
}

template <int QMAX, bool PACK4>
void launch_q(const QuantArgs &p, bool f16in, unsigned blocks, cudaStream_t s)
{
    if (f16in) mbg_quantize_kernel<QMAX, true, PACK4><<<blocks, 256, 0, s>>>(p);
    else mbg_quantize_kernel<QMAX, false, PACK4><<<blocks, 256, 0, s>>>(p);
}

template <int QMAX, bool PACK4, bool F16IN>
void launch_vec(const QuantArgs &p, unsigned blocks, cudaStream_t s)
{
    constexpr int UNROLL = F16IN ? 2 : 1;
    if (p.sq_err) mbg_quantize_vec_kernel<QMAX, F16IN, PACK4, true, UNROLL><<<blocks, 256, 0, s>>>(p);
    else mbg_quantize_vec_kernel<QMAX, F16IN, PACK4, false, UNROLL><<<blocks, 256, 0, s>>>(p);
}

template <bool F16IN>
void launch_row(const QuantArgs &p, unsigned blocks, cudaStream_t s)
{
    if (p.sq_err) mbg_quantize_row_kernel<F16IN, true><<<blocks, 256, 0, s>>>(p);
    else mbg_quantize_row_kernel<F16IN, false><<<blocks, 256, 0, s>>>(p);
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
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;  // 2048 threads per SM
    const bool w16 = reinterpret_cast<uintptr_t>(W) % 16 == 0;
    const uintptr_t a_addr = reinterpret_cast<uintptr_t>(A);
    if (!per_row && N % kGroup == 0 && w16 && a_addr % (bits == 8 ? 8 : 4) == 0) {
        // 16 groups per block and pass (8 warps x 2 halves x UNROLL)
        const int64_t per_block = f16in ? 32 : 16;
        const unsigned blocks = static_cast<unsigned>(std::min(cap, (M * p.groups + per_block - 1) / per_block));
        if (bits == 8) {
            if (f16in) launch_vec<127, false, true>(p, blocks, s);
            else launch_vec<127, false, false>(p, blocks, s);
        } else {
            if (f16in) launch_vec<7, true, true>(p, blocks, s);
            else launch_vec<7, true, false>(p, blocks, s);
        }
        return;
    }
    if (per_row && bits == 8 && N % 8 == 0 && w16 && a_addr % 8 == 0) {
        const unsigned blocks = static_cast<unsigned>(std::min(cap, M));
        if (f16in) launch_row<true>(p, blocks, s);
        else launch_row<false>(p, blocks, s);
        return;
    }
    const int64_t warps = M * p.groups;
    int64_t blocks = (warps + 7) / 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (bits == 8) launch_q<127, false>(p, f16in, static_cast<unsigned>(blocks), s);
    else launch_q<7, true>(p, f16in, static_cast<unsigned>(blocks), s);
}

}  // namespace mbg
