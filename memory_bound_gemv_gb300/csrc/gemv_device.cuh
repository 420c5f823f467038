// Device-side building blocks of the GEMV kernels (sm_103a).
//
// Streaming loads of A, bounded mbarrier waits for the bulk copy of x,
// in-register unpacking of INT8 / INT4 codes and the FP32 dot-product
// accumulation.  The kernels themselves are in gemv_kernels.cuh.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "gemv_internal.h"

namespace mbg {

// ---------------------------------------------------------------------------
// Global memory
// ---------------------------------------------------------------------------

// 16-byte read-only load that bypasses L1 and asks L2 to fetch the whole
// 256-byte block: A is read exactly once, so it should not evict x or the
// scales from L1.  ("membound", kernel "vec": one 128-bit load per lane per
// step, so a warp reads 512 contiguous bytes.)
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// An ordinary 16-byte load cached in L2 only (not the read-only path).
__device__ __forceinline__ uint4 ld_l2_16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p)
        : "memory");
    return v;
}

// 16-byte read-only load that may allocate in L1 (x, when it is not staged).
__device__ __forceinline__ uint4 ld_cached16(const void *p)
{
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_half_as_float(const uint16_t *p)
{
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Asks L2 to fetch [p, p + bytes) (16-byte aligned, a multiple of 16 bytes).
// A prefetch is only a hint: it changes no value that a later load returns,
// so it may be issued before the wait for a preceding kernel that could
// still write the range (L2 is where that kernel's writes land).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream (if it was launched with programmatic serialisation) start its
// blocks while this grid still runs; wait blocks until the preceding grid has
// finished and its memory operations are visible.  Both are no-ops for
// kernels launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void report_error(unsigned int *err, unsigned int code)
{
    if (err) atomicOr(err, code);
}

// Shared-memory loads with 32-bit shared-space addresses (keeps the hot loops'
// address arithmetic in 32-bit registers).  Volatile so that they stay after
// the mbarrier waits that make the data visible.
__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_half_as_float(uint32_t addr)
{
    unsigned short b;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(b) : "r"(addr));
    return __half2float(__ushort_as_half(b));
}

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (x staging)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One bulk copy global -> shared that signals `bar` with its byte count.
// Addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Waits for phase `parity` of `bar` to complete, giving up after limit_ns.
// Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(2000u)
            : "memory");
        if (done) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------------
// Unpacking quantised codes (exact)
// ---------------------------------------------------------------------------

// Four int8 codes of a 32-bit word -> four floats, exactly.  Flipping the
// sign bit turns code b into the unsigned byte b + 128; placing that byte in
// the low mantissa bits of 2^23 (bit pattern 0x4B0000uu) gives the float
// 2^23 + b + 128, and subtracting 2^23 + 128 leaves b.
__device__ __forceinline__ void unpack_q8_word(uint32_t w, float (&f)[4])
{
    const uint32_t u = w ^ 0x80808080u;
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - 8388736.0f;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - 8388736.0f;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - 8388736.0f;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - 8388736.0f;
}

// Eight int4 codes of a 32-bit word (nibble k = column k of the word: the
// low nibble of each byte is the even column) -> eight floats, exactly.
// XOR with 8 per nibble maps the two's-complement code q to q + 8 in [0, 15];
// OR-ing that into the mantissa of 2^23 and subtracting 2^23 + 8 leaves q.
__device__ __forceinline__ void unpack_q4_word(uint32_t w, float (&f)[8])
{
    const uint32_t u = w ^ 0x88888888u;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        f[k] = __uint_as_float(0x4B000000u | ((u >> (4 * k)) & 0xFu)) - 8388616.0f;
}

// Two binary16 values packed in a 32-bit word (low half first) -> two floats.
__device__ __forceinline__ void half2_bits_to_float(uint32_t w, float &lo, float &hi)
{
    asm("{\n .reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
}

// ---------------------------------------------------------------------------
// Storage formats
// ---------------------------------------------------------------------------

template <int DT> struct Fmt;

template <> struct Fmt<DT_F32> {
    static constexpr int EPC = 4;   // elements per 16-byte chunk of A
    static constexpr int XB = 4;    // bytes per element of x
    static constexpr bool QUANT = false;
};
template <> struct Fmt<DT_F16> {
    static constexpr int EPC = 8;
    static constexpr int XB = 2;
    static constexpr bool QUANT = false;
};
template <> struct Fmt<DT_Q8> {
    static constexpr int EPC = 16;
    static constexpr int XB = 2;
    static constexpr bool QUANT = true;
};
template <> struct Fmt<DT_Q4> {
    static constexpr int EPC = 32;
    static constexpr int XB = 2;
    static constexpr bool QUANT = true;
};
template <> struct Fmt<DT_F16X32> {
    static constexpr int EPC = 8;
    static constexpr int XB = 4;
    static constexpr bool QUANT = false;
};

// Bytes of x that one 16-byte chunk of A multiplies.
template <int DT> constexpr int x_chunk_bytes() { return Fmt<DT>::EPC * Fmt<DT>::XB; }
template <int DT> constexpr int x_chunk_vecs() { return x_chunk_bytes<DT>() / 16; }

// x in shared memory is kept vector-major: 16-byte vector v of chunk c sits at
// byte (v * nchunks + c) * 16.  Lane t of a warp reading vector v of chunk t
// then touches consecutive 16-byte slots, free of bank conflicts, whatever
// the number of vectors per chunk (INT4 needs four: 32 binary16 values of x
// per 16 bytes of A; read chunk-major they would be 64 bytes apart per lane,
// a 16-way conflict).  For FP32 and FP16 (one vector per chunk) this is
// simply x in its own order, so a plain bulk copy stages it.
__device__ __forceinline__ const uint4 *x_smem_vec(const unsigned char *xs, int nchunks, int c, int v)
{
    return reinterpret_cast<const uint4 *>(xs + (static_cast<size_t>(v) * nchunks + c) * 16);
}

// Cooperative staging of x into the vector-major layout by threads
// t = 0 .. nt-1 (reads are coalesced in x's own order).  Loads are issued in
// batches of eight per thread before any of them is stored, so staging costs
// one memory round trip per batch instead of one per vector.
// ORDERED: the loads are ordinary (not read-only-path) loads, which the
// compiler keeps ahead of a barrier arrive that follows them, and
// after_issue() runs once in every thread, at the same point in all of them,
// as soon as the first batch has been issued (before any of it is used).
// PAIRED (INT4 with the mixed-precision products): each 16-byte vector of x
// is stored re-paired four columns apart, (x0,x4) (x1,x5) (x2,x6) (x3,x7),
// the order in which q4_codes_h2 yields the codes, so that every product
// takes the same half of its two operands.
// One 16-byte vector of x re-paired four columns apart (the PAIRED layout).
__device__ __forceinline__ uint4 pair_x_vec(const uint4 u)
{
    uint4 w;
    w.x = __byte_perm(u.x, u.z, 0x5410);
    w.y = __byte_perm(u.x, u.z, 0x7632);
    w.z = __byte_perm(u.y, u.w, 0x5410);
    w.w = __byte_perm(u.y, u.w, 0x7632);
    return w;
}

struct NoOp {
    __device__ void operator()() const {}
};

template <int DT, bool PAIRED = false, bool ORDERED = false, typename AfterIssue = NoOp>
__device__ __forceinline__ void stage_x_vmajor(unsigned char *xs, const void *x, int nchunks, int t,
                                               int nt, AfterIssue after_issue = AfterIssue{})
{
    constexpr int XV = x_chunk_vecs<DT>();
    constexpr int B = 8;
    const uint4 *src = static_cast<const uint4 *>(x);
    const int n = nchunks * XV;
    auto batch = [&](int base, auto first) {
        uint4 r[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int i = base + j * nt;
            if (i < n) r[j] = ORDERED ? ld_l2_16(src + i) : ld_cached16(src + i);
        }
        if constexpr (decltype(first)::value) after_issue();
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int i = base + j * nt;
            if (i < n) {
                const int c = i / XV;
                const int v = i - c * XV;
                uint4 w = r[j];
                if constexpr (PAIRED) w = pair_x_vec(w);
                *reinterpret_cast<uint4 *>(xs + (static_cast<size_t>(v) * nchunks + c) * 16) = w;
            }
        }
    };
    if constexpr (ORDERED) {
        batch(t, std::true_type{});
        for (int base = t + B * nt; base < n; base += B * nt) batch(base, std::false_type{});
    } else {
        for (int base = t; base < n; base += B * nt) batch(base, std::false_type{});
    }
}

// x chunk (as raw 16-byte vectors) -> floats.
template <int DT>
__device__ __forceinline__ void x_to_float(const uint4 (&xv)[x_chunk_vecs<DT>()],
                                           float (&xf)[Fmt<DT>::EPC])
{
    if constexpr (Fmt<DT>::XB == 4) {
#pragma unroll
        for (int v = 0; v < x_chunk_vecs<DT>(); ++v) {
            xf[4 * v + 0] = __uint_as_float(xv[v].x);
            xf[4 * v + 1] = __uint_as_float(xv[v].y);
            xf[4 * v + 2] = __uint_as_float(xv[v].z);
            xf[4 * v + 3] = __uint_as_float(xv[v].w);
        }
    } else {
#pragma unroll
        for (int v = 0; v < x_chunk_vecs<DT>(); ++v) {
            half2_bits_to_float(xv[v].x, xf[v * 8 + 0], xf[v * 8 + 1]);
            half2_bits_to_float(xv[v].y, xf[v * 8 + 2], xf[v * 8 + 3]);
            half2_bits_to_float(xv[v].z, xf[v * 8 + 4], xf[v * 8 + 5]);
            half2_bits_to_float(xv[v].w, xf[v * 8 + 6], xf[v * 8 + 7]);
        }
    }
}

// One 16-byte chunk of A -> its EPC weights (codes for the quantised types).
template <int DT>
__device__ __forceinline__ void chunk_to_float(const uint4 a, float (&wf)[Fmt<DT>::EPC])
{
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    if constexpr (DT == DT_F32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) wf[k] = __uint_as_float(w[k]);
    } else if constexpr (DT == DT_F16 || DT == DT_F16X32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) half2_bits_to_float(w[k], wf[2 * k], wf[2 * k + 1]);
    } else if constexpr (DT == DT_Q8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float f[4];
            unpack_q8_word(w[k], f);
#pragma unroll
            for (int e = 0; e < 4; ++e) wf[4 * k + e] = f[e];
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float f[8];
            unpack_q4_word(w[k], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) wf[8 * k + e] = f[e];
        }
    }
}

// Number of FP32 accumulators per row and lane.  Each 16-byte chunk feeds
// its elements round-robin into them, so the dependent-add chain of one
// accumulator is (elements per lane) / NACC long; four keep the FP32 chain at
// N/128 for a full warp per row.
constexpr int NACC = 4;

// acc[e % NACC] += w[e] * x[e] over one chunk (unquantised), or
// acc[e % NACC] += s * (sum of the chunk's code * x) (quantised: the scale is
// constant over a chunk because 128 is a multiple of the chunk's width).
template <int DT>
__device__ __forceinline__ void chunk_fma(const float (&wf)[Fmt<DT>::EPC],
                                          const float (&xf)[Fmt<DT>::EPC], float scale,
                                          float (&acc)[NACC])
{
    if constexpr (!Fmt<DT>::QUANT) {
        (void)scale;
#pragma unroll
        for (int e = 0; e < Fmt<DT>::EPC; ++e) acc[e % NACC] = fmaf(wf[e], xf[e], acc[e % NACC]);
    } else {
        float p[NACC] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < Fmt<DT>::EPC; ++e) p[e % NACC] = fmaf(wf[e], xf[e], p[e % NACC]);
#pragma unroll
        for (int k = 0; k < NACC; ++k) acc[k] = fmaf(scale, p[k], acc[k]);
    }
}

// ---------------------------------------------------------------------------
// Mixed-precision path: binary16 operands, FP32 accumulation, no conversions
// ---------------------------------------------------------------------------
//
// fma.rn.f32.f16 (sm_100 and later) multiplies two binary16 values and adds
// an FP32 accumulator.  The product of two binary16 significands (11 bits
// each) is exact in FP32, so c + a*b is rounded once, exactly as
// fmaf(float(a), float(b), c) would be.  On this GPU it issues at the full
// FP32 rate, while a binary16 -> FP32 conversion issues at half rate.

// c0 += lo(a) * lo(b);  c1 += hi(a) * hi(b)
__device__ __forceinline__ void mfma_pair(uint32_t a, uint32_t b, float &c0, float &c1)
{
    asm("{\n .reg .f16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
        " fma.rn.f32.f16 %0, a0, b0, %0;\n fma.rn.f32.f16 %1, a1, b1, %1;\n}"
        : "+f"(c0), "+f"(c1)
        : "r"(a), "r"(b));
}

// c0 += lo(a) * lo(b0);  c1 += hi(a) * lo(b1)  (codes paired across x words)
__device__ __forceinline__ void mfma_cross_lo(uint32_t a, uint32_t b0, uint32_t b1, float &c0,
                                              float &c1)
{
    asm("{\n .reg .f16 a0, a1, p0, p1, q0, q1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {p0, p1}, %3;\n"
        " mov.b32 {q0, q1}, %4;\n fma.rn.f32.f16 %0, a0, p0, %0;\n fma.rn.f32.f16 %1, a1, q0, %1;\n}"
        : "+f"(c0), "+f"(c1)
        : "r"(a), "r"(b0), "r"(b1));
}

// c0 += lo(a) * hi(b0);  c1 += hi(a) * hi(b1)
__device__ __forceinline__ void mfma_cross_hi(uint32_t a, uint32_t b0, uint32_t b1, float &c0,
                                              float &c1)
{
    asm("{\n .reg .f16 a0, a1, p0, p1, q0, q1;\n mov.b32 {a0, a1}, %2;\n mov.b32 {p0, p1}, %3;\n"
        " mov.b32 {q0, q1}, %4;\n fma.rn.f32.f16 %0, a0, p1, %0;\n fma.rn.f32.f16 %1, a1, q1, %1;\n}"
        : "+f"(c0), "+f"(c1)
        : "r"(a), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four int8 codes -> two pairs of exact binary16 values, in column order:
// h[0] = (q0, q1), h[1] = (q2, q3).  The sign flip gives the byte q + 128;
// pairing it with 0x64 forms the binary16 value 1024 + q + 128, and
// subtracting 1152 (0x6480) leaves q.
__device__ __forceinline__ void q8_codes_h2(uint32_t w, uint32_t (&h)[2])
{
    const uint32_t u = w ^ 0x80808080u;
    h[0] = hsub2_bits(__byte_perm(u, 0x64646464u, 0x4140), 0x64806480u);
    h[1] = hsub2_bits(__byte_perm(u, 0x64646464u, 0x4342), 0x64806480u);
}

// d = c ? (a ^ b) : b, bit by bit (one LOP3, lookup table 0x6C).
__device__ __forceinline__ uint32_t lop3_sel_xor(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6C;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Eight int4 codes of a word (nibble k = column k) -> four pairs of exact
// binary16 values, paired four columns apart: h[0] = (q0, q4),
// h[1] = (q1, q5), h[2] = (q2, q6), h[3] = (q3, q7).  One LOP3 per pair
// keeps two nibbles (mask c), flips their top bit (two's complement q ->
// q + 8 in [0, 15]) and fills the rest of each half with 0x6400: a nibble in
// bits 0-3 of a half gives 1024 + (q + 8), minus 1032 (0x6408) is q; a
// nibble in bits 4-7 gives 1024 + 16 (q + 8), times 1/16 (0x2C00) minus 72
// (0xD480) is q.  The XOR constant is the same in every nibble, so the upper
// four nibbles use the word shifted right by 8 with the same constants.
// (ALU cost: one shift and four LOP3 per eight codes.)
__device__ __forceinline__ void q4_codes_h2(uint32_t w, uint32_t (&h)[4])
{
    const uint32_t v = w >> 8;
    h[0] = hsub2_bits(lop3_sel_xor(w, 0x64086408u, 0x000F000Fu), 0x64086408u);
    h[1] = hfma2_bits(lop3_sel_xor(w, 0x64806480u, 0x00F000F0u), 0x2C002C00u, 0xD480D480u);
    h[2] = hsub2_bits(lop3_sel_xor(v, 0x64086408u, 0x000F000Fu), 0x64086408u);
    h[3] = hfma2_bits(lop3_sel_xor(v, 0x64806480u, 0x00F000F0u), 0x2C002C00u, 0xD480D480u);
}

// One 16-byte chunk of A times its x chunk (binary16), accumulated in FP32.
// Quantised chunks are summed into partials and scaled once per chunk
// (the chunk lies inside one 128-column group).
template <int DT, bool PAIRED = false>
__device__ __forceinline__ void chunk_dot_mixed(const uint4 a, const uint4 (&xv)[x_chunk_vecs<DT>()],
                                                float scale, float (&acc)[NACC])
{
    static_assert(Fmt<DT>::XB == 2, "an FP32 x takes the FP32 path");
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    if constexpr (DT == DT_F16) {
        (void)scale;
        mfma_pair(w[0], xv[0].x, acc[0], acc[1]);
        mfma_pair(w[1], xv[0].y, acc[2], acc[3]);
        mfma_pair(w[2], xv[0].z, acc[0], acc[1]);
        mfma_pair(w[3], xv[0].w, acc[2], acc[3]);
    } else if constexpr (DT == DT_Q8) {
        float p[NACC] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t h[2];
            q8_codes_h2(w[k], h);
            const uint4 &x = xv[k >> 1];
            const uint32_t x01 = (k & 1) ? x.z : x.x;
            const uint32_t x23 = (k & 1) ? x.w : x.y;
            mfma_pair(h[0], x01, p[0], p[1]);
            mfma_pair(h[1], x23, p[2], p[3]);
        }
#pragma unroll
        for (int k = 0; k < NACC; ++k) acc[k] = fmaf(scale, p[k], acc[k]);
    } else {
        float p[NACC] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t h[4];
            q4_codes_h2(w[k], h);
            const uint4 &x = xv[k];
            if constexpr (PAIRED) {
                // x words (x0,x4) (x1,x5) (x2,x6) (x3,x7): same halves as the codes
                mfma_pair(h[0], x.x, p[0], p[1]);
                mfma_pair(h[1], x.y, p[2], p[3]);
                mfma_pair(h[2], x.z, p[0], p[1]);
                mfma_pair(h[3], x.w, p[2], p[3]);
            } else {
                // x words (x0,x1) (x2,x3) (x4,x5) (x6,x7)
                mfma_cross_lo(h[0], x.x, x.z, p[0], p[1]);  // q0*x0, q4*x4
                mfma_cross_hi(h[1], x.x, x.z, p[2], p[3]);  // q1*x1, q5*x5
                mfma_cross_lo(h[2], x.y, x.w, p[0], p[1]);  // q2*x2, q6*x6
                mfma_cross_hi(h[3], x.y, x.w, p[2], p[3]);  // q3*x3, q7*x7
            }
        }
#pragma unroll
        for (int k = 0; k < NACC; ++k) acc[k] = fmaf(scale, p[k], acc[k]);
    }
}

template <int WIDTH>
__device__ __forceinline__ float group_sum(float v)
{
    // XOR butterfly inside aligned groups of WIDTH lanes: every lane of the
    // group ends with the group's sum ("llama.cpp GEMV CUDA", warp_reduce_sum
    // with __shfl_xor_sync).
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

}  // namespace mbg
