// Device helpers shared by the quantizer kernels (sm_103a): loads and
// stores, element access, |x| maxima, FP8 / FP4 conversions, the scale
// rules, Philox4x32-10 and stochastic rounding, reductions, the CTA-wide
// maximum, programmatic-dependent-launch waits and the 4x4 byte transpose.
// The tile geometry of the kernels that stream 128-row tiles is in
// q_engine.cuh (a 16-byte chunk of 8 rows per thread, VEC = 8 BF16 or 4 FP32
// elements per chunk).
//
// FP32 arithmetic that decides a code is written with explicit round-to-
// nearest intrinsics (__fmul_rn, __fdiv_rn) so that no product is fused into
// an FMA and no division is approximated; the library is also compiled with
// -fmad=false.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <float.h>

#define QD __device__ __forceinline__

namespace qk {

enum { BF16 = 0, F32 = 1, U8 = 2 };
enum { E4M3 = 0, E5M2 = 1 };

constexpr int32_t kStNonFinite = 1;

template <int DT> struct In;
template <> struct In<BF16> { static constexpr int VEC = 8; static constexpr int BYTES = 2; };
template <> struct In<F32> { static constexpr int VEC = 4; static constexpr int BYTES = 4; };

template <int FMT> struct Fp8;
template <> struct Fp8<E4M3> { static constexpr float FMAX = 448.0f; static constexpr int EMAX = 8; };
template <> struct Fp8<E5M2> { static constexpr float FMAX = 57344.0f; static constexpr int EMAX = 15; };

// ---------------------------------------------------------------------------
// memory
// ---------------------------------------------------------------------------

// Streaming 16-byte load: read-only path, no L1 allocation.
QD uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

QD void stg16(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
// 32 bytes in one store (p 32-byte aligned): a warp's store covers 1 KiB.
QD void stg32(void *p, const uint4 &a, const uint4 &b)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
                 "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w) : "memory");
}
QD void stg8(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(a), "r"(b) : "memory");
}
QD void stg4(void *p, uint32_t a)
{
    asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(a) : "memory");
}

QD uint32_t word(const uint4 &v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------

// Element j (0..VEC-1) of a 16-byte vector as an exact FP32 value.
template <int DT> QD float elem(const uint4 &v, int j);
template <> QD float elem<BF16>(const uint4 &v, int j)
{
    uint32_t w = word(v, j >> 1);
    return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
}
template <> QD float elem<F32>(const uint4 &v, int j) { return __uint_as_float(word(v, j)); }

// |x| maxima.  Packed BF16 pairs use max.NaN.xorsign.abs.bf16x2 (one FP-pipe
// instruction for two magnitudes; the result's sign bits are the XOR of the
// inputs' and are masked off where a value is read).  NaN propagates as the
// canonical NaN, whose bit pattern exceeds every finite value and inf.
QD uint32_t hmax_abs2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
QD float fmax_abs(float a, float b)
{
    float r;
    asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// absmax_bits: FP32 bit pattern of the largest |element| of the vector
// (non-negative FP32 bit patterns compare like the magnitudes they encode).
template <int DT> QD uint32_t absmax_bits(const uint4 &v);
template <> QD uint32_t absmax_bits<BF16>(const uint4 &v)
{
    uint32_t m = hmax_abs2(hmax_abs2(v.x, v.y), hmax_abs2(v.z, v.w));
    m = hmax_abs2(m, __byte_perm(m, 0u, 0x1032));   // both halves now hold the maximum
    return (m << 16) & 0x7FFF0000u;
}
template <> QD uint32_t absmax_bits<F32>(const uint4 &v)
{
    const float m = fmax_abs(fmax_abs(__uint_as_float(v.x), __uint_as_float(v.y)),
                             fmax_abs(__uint_as_float(v.z), __uint_as_float(v.w)));
    return __float_as_uint(m) & 0x7FFFFFFFu;
}

// Per-column running maximum of |x| over rows, kept in the input's packing
// (BF16: two columns per word; FP32: one), sign bits undefined.
template <int DT> QD uint32_t colmax_word(uint32_t acc, uint32_t w);
template <> QD uint32_t colmax_word<BF16>(uint32_t acc, uint32_t w) { return hmax_abs2(acc, w); }
template <> QD uint32_t colmax_word<F32>(uint32_t acc, uint32_t w)
{
    return __float_as_uint(fmax_abs(__uint_as_float(acc), __uint_as_float(w)));
}
// FP32 bits of column j's maximum from the packed accumulators.
template <int DT> QD uint32_t colmax_bits(const uint4 &acc, int j);
template <> QD uint32_t colmax_bits<BF16>(const uint4 &acc, int j)
{
    const uint32_t w = word(acc, j >> 1);
    return ((j & 1) ? w : (w << 16)) & 0x7FFF0000u;
}
template <> QD uint32_t colmax_bits<F32>(const uint4 &acc, int j) { return word(acc, j) & 0x7FFFFFFFu; }

// Maxima of two rows over groups of G consecutive lanes with one shuffle
// chain: BF16 magnitudes (the high halves of their FP32 bit patterns) travel
// packed in one word.  FP32 runs two chains.
template <int DT, int G> QD void group_max2(uint32_t &a, uint32_t &b)
{
    if (DT == BF16) {
        uint32_t p = __byte_perm(a, b, 0x7632);   // a's magnitude low, b's high
#pragma unroll
        for (int o = 1; o < G; o <<= 1) p = hmax_abs2(p, __shfl_xor_sync(0xFFFFFFFFu, p, o));
        a = (p << 16) & 0x7FFF0000u;
        b = p & 0x7FFF0000u;
    } else {
#pragma unroll
        for (int o = 1; o < G; o <<= 1) {
            a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            b = max(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
        }
    }
}

// ---------------------------------------------------------------------------
// conversions (PTX cvt; RTNE, saturating to the largest finite value)
// ---------------------------------------------------------------------------

// Four FP32 values -> four FP8 codes in one word, a in the lowest byte.
template <int FMT> QD uint32_t cvt_fp8x4(float a, float b, float c, float d);
template <> QD uint32_t cvt_fp8x4<E4M3>(float a, float b, float c, float d)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}
template <> QD uint32_t cvt_fp8x4<E5M2>(float a, float b, float c, float d)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// Eight FP32 values -> eight E2M1 codes in one word, v0 in bits 3-0.
QD uint32_t cvt_fp4x8(float v0, float v1, float v2, float v3, float v4, float v5, float v6, float v7)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r) : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return r;
}

// One E4M3 code (saturating RTNE) of an FP32 value, and its exact value.
QD uint32_t e4m3_code(float f)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(f));
    return (uint32_t)h & 0xFFu;
}
QD float e4m3_value(uint32_t code)
{
    uint32_t h2;
    uint16_t c = (uint16_t)code;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    float f;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

// Two FP8 codes (low, high byte of a 16-bit value) -> two exact FP32 values.
template <int FMT> QD float2 fp8x2_to_f32(uint32_t two);
template <> QD float2 fp8x2_to_f32<E4M3>(uint32_t two)
{
    uint32_t h2;
    uint16_t c = (uint16_t)two;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}
template <> QD float2 fp8x2_to_f32<E5M2>(uint32_t two)
{
    uint32_t h2;
    uint16_t c = (uint16_t)two;
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(c));
    float lo, hi;
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}

// FP32 -> BF16 bits, round to nearest even.
QD uint32_t bf16_bits(float f)
{
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}

// a *= s0 and b *= s1: two IEEE round-to-nearest FP32 products in one
// packed instruction (the same results as two separate multiplies).
QD void mul2(float &a, float &b, float s0, float s1)
{
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%0, %1};\n\t"
        "mov.b64 y, {%2, %3};\n\t"
        "mul.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "+f"(a), "+f"(b) : "f"(s0), "f"(s1));
}

// Butterfly on two column pairs: (a, b) -> (a + b, a - b) for (a0, b0) and
// (a1, b1) together (one packed FP32x2 add and one sub, each rounded once).
QD void bfly2(float &a0, float &a1, float &b0, float &b1)
{
    asm("{\n\t.reg .b64 x, y, s, d;\n\t"
        "mov.b64 x, {%0, %1};\n\t"
        "mov.b64 y, {%2, %3};\n\t"
        "add.rn.f32x2 s, x, y;\n\t"
        "sub.rn.f32x2 d, x, y;\n\t"
        "mov.b64 {%0, %1}, s;\n\t"
        "mov.b64 {%2, %3}, d;\n\t}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// The VEC elements of a 16-byte row chunk times s, as FP8 codes (VEC/4 words,
// element 0 in the lowest byte).
template <int DT, int FMT> QD void chunk_fp8(const uint4 &v, float s, uint32_t *o)
{
    constexpr int VEC = In<DT>::VEC;
    float f[VEC];
#pragma unroll
    for (int j = 0; j < VEC; j++) f[j] = elem<DT>(v, j);
#pragma unroll
    for (int j = 0; j < VEC; j += 2) mul2(f[j], f[j + 1], s, s);
#pragma unroll
    for (int w = 0; w < VEC / 4; w++) o[w] = cvt_fp8x4<FMT>(f[4 * w], f[4 * w + 1], f[4 * w + 2], f[4 * w + 3]);
}

// ---------------------------------------------------------------------------
// scales
// ---------------------------------------------------------------------------

// alpha = fmax / a; a = 0 -> 1; an alpha that overflows -> FLT_MAX.
QD float alpha_from_amax(float fmax, float a)
{
    if (a == 0.0f) return 1.0f;
    float al = __fdiv_rn(fmax, a);
    if (al == __int_as_float(0x7F800000)) al = FLT_MAX;
    return al;
}

// E8M0 code for a block whose largest magnitude has FP32 bits b:
// clamp(floor(log2 b) - emax + 127, 0, 254), b = 0 -> 127.  For a normal b,
// floor(log2 b) + 127 is the exponent field E, so the code is E - emax; a
// subnormal b (E = 0) clamps to 0 either way, and inf / NaN (E = 255) give
// 255 - emax, the same as floor(log2) = 128.
template <int FMT> QD uint32_t mx_code(uint32_t b)
{
    if (b == 0) return 127u;
    int c = (int)(b >> 23) - Fp8<FMT>::EMAX;
    c = c < 0 ? 0 : (c > 254 ? 254 : c);
    return (uint32_t)c;
}

// 2^(127 - code) as an FP32 value (code in [0, 254]; 2^-127 is subnormal).
QD float mx_inv_scale(uint32_t code)
{
    int e = 127 - (int)code;
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11)
// ---------------------------------------------------------------------------

// Round multipliers and key increments (Weyl constants) of the paper.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// The ten round keys of a seed (round r: key + r * increments), formed once
// on the host and passed to a kernel by value, so that each round reads its
// key from the kernel's parameters instead of adding the increments.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};
inline __host__ __device__ PhiloxKeys philox_keys(uint64_t seed)
{
    PhiloxKeys K;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; r++) {
        K.k0[r] = a;
        K.k1[r] = b;
        a += kPhiloxW0;
        b += kPhiloxW1;
    }
    return K;
}

// Philox4x32-10 of counter c under the key whose round keys K holds: ten
// rounds of (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (32 x 32 -> 64-bit
// products), c = (hi1 ^ c1 ^ k0[r], lo1, hi0 ^ c3 ^ k1[r], lo0).
QD uint4 philox4x32_10_rk(uint4 c, const PhiloxKeys &K)
{
#pragma unroll
    for (int r = 0; r < 10; r++) {
        const uint32_t hi0 = __umulhi(kPhiloxM0, c.x), lo0 = kPhiloxM0 * c.x;
        const uint32_t hi1 = __umulhi(kPhiloxM1, c.z), lo1 = kPhiloxM1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ K.k0[r], lo1, hi0 ^ c.w ^ K.k1[r], lo0);
    }
    return c;
}

// The 128 random bits of Philox block g of a stream, with round keys.
template <uint32_t STREAM> QD uint4 sr_bits_rk(uint64_t g, const PhiloxKeys &K)
{
    return philox4x32_10_rk(make_uint4((uint32_t)g, (uint32_t)(g >> 32), STREAM, 0u), K);
}

// Stochastic rounding onto the E2M1 grid by the conversion with random bits
// (cvt.rs.satfinite.e2m1x4.f32).  For a = |y| < 6 between the grid
// neighbours lo and lo + ulp (ulp 0.5 below 2, 1 in [2, 4), 2 in [4, 6)),
// T = floor(((a - lo) / ulp) * 2^16), the code rounds up iff T + R >= 2^16
// for the element's 16-bit draw R; |y| >= 6 gives 6, NaN gives +6 as the
// round-to-nearest conversion does, and the code carries y's sign.  The 32
// random bits r of a group of four give two draws, U0 = bytes 0 and 2 of r
// (byte 2 high) and U1 = bytes 1 and 3 (byte 3 high): y0 takes U0, y1 U0
// bit-reversed, y2 U1 and y3 U1 bit-reversed (the instruction's assignment
// when the operands are passed as {y3, y2, y1, y0}, which also puts y0's
// code in bits 3-0).
QD uint32_t cvt_rs_fp4x4(float y0, float y1, float y2, float y3, uint32_t r)
{
    uint16_t d;
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;" : "=h"(d) : "f"(y3), "f"(y2), "f"(y1), "f"(y0), "r"(r));
    return d;
}
// Eight values (y0 in bits 3-0) with the random words r0 (y0..y3) and r1 (y4..y7).
QD uint32_t cvt_rs_fp4x8(float y0, float y1, float y2, float y3, float y4, float y5, float y6, float y7,
                         uint32_t r0, uint32_t r1)
{
    uint32_t c;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rs.satfinite.e2m1x4.f32 lo, {%4, %3, %2, %1}, %9;\n\t"
        "cvt.rs.satfinite.e2m1x4.f32 hi, {%8, %7, %6, %5}, %10;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(c) : "f"(y0), "f"(y1), "f"(y2), "f"(y3), "f"(y4), "f"(y5), "f"(y6), "f"(y7), "r"(r0), "r"(r1));
    return c;
}
QD uint32_t cvt_rs_fp4x8(const float (&y)[8], uint32_t r0, uint32_t r1)
{
    return cvt_rs_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7], r0, r1);
}


// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

QD uint32_t warp_max(uint32_t v) { return __reduce_max_sync(0xFFFFFFFFu, v); }

// Max over groups of G consecutive lanes (G a power of two <= 32).
template <int G> QD uint32_t group_max(uint32_t v)
{
#pragma unroll
    for (int o = 1; o < G; o <<= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start before the kernel ahead of it in the stream has
// finished (once every CTA of that kernel has signalled or exited); it must
// call griddep_wait() before it touches anything that kernel writes.  In a
// kernel launched normally griddep_wait() returns at once.
QD void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QD void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

QD void flag_nonfinite(int32_t *status, uint32_t amax_bits)
{
    if (status != nullptr && amax_bits >= 0x7F800000u) atomicOr(status, kStNonFinite);
}

// CTA-wide max of m (blockDim.x a multiple of 32, at most 1024 threads),
// then one atomicMax into *dst from a CTA that raises it; a non-finite
// result is reported in *status.
QD void cta_max_to(uint32_t m, uint32_t *dst, int32_t *status)
{
    __shared__ uint32_t red[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
        m = warp_max(m);
        if (lane == 0) {
            if (m > *reinterpret_cast<volatile uint32_t *>(dst)) atomicMax(dst, m);
            flag_nonfinite(status, m);
        }
    }
}
// Thread-local record of non-finite maxima, posted once (see post_nonfinite).
QD uint32_t nonfinite(uint32_t amax_bits) { return amax_bits >= 0x7F800000u ? 1u : 0u; }
QD void post_nonfinite(int32_t *status, uint32_t seen)
{
    if (seen && status != nullptr) atomicOr(status, kStNonFinite);
}

// 4x4 byte transpose: in r[i] byte j = element (row i, col j);
// out c[j] byte i = the same element.
QD void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                     uint32_t &c0, uint32_t &c1, uint32_t &c2, uint32_t &c3)
{
    uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r2, r3, 0x5140);
    uint32_t t2 = __byte_perm(r0, r1, 0x7362), t3 = __byte_perm(r2, r3, 0x7362);
    c0 = __byte_perm(t0, t1, 0x5410);
    c1 = __byte_perm(t0, t1, 0x7632);
    c2 = __byte_perm(t2, t3, 0x5410);
    c3 = __byte_perm(t2, t3, 0x7632);
}

}  // namespace qk
