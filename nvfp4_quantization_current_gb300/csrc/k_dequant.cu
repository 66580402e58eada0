// Dequantizers (a12): codes + scales -> FP32 or BF16, one streaming pass.
//
//   current scaling  x_hat = q * s            ("FP8 Current Scaling ...",
//                                               section "Current Scaling")
//   MXFP8            x_hat = q * 2^(code-127)  ("Mixed-precision training:
//                                               fp16 to fp8", section "MXFP8")
//   blockwise        x_hat = q * s_tile
//   NVFP4            x_hat = q * (sb * s_g), the block factor formed once
//
// Codes decode exactly (cvt to f16x2, then to FP32); the one FP32 product per
// element is rounded to nearest; BF16 output rounds that FP32 value to
// nearest even.
//
// Work unit of the FP8 kernels: 16 bytes of output per lane (8 elements for
// BF16 output, 4 for FP32), so that one warp store covers 512 contiguous
// bytes; NVFP4 units are 16-element block rows (k_dq_fp4).  A CTA of 256
// threads covers BX units x BY rows (BX = units per row rounded to a power
// of two, at most 256); each thread keeps kDqRows rows of loads in flight
// (4: more, shorter CTAs fill the waves of mid-size tensors better than 8).
// No index division happens per element: the 2-D grid (x: row groups, y:
// unit blocks of a row) gives the row and the unit of every thread.
#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

constexpr int kDqRows = 4;    // rows per thread in the block-scaled kernels
constexpr int kDqUnits = 8;   // units per thread in flight in the flat current-scaling kernel
constexpr int kDqThreads = 256;

// FP32 pairs -> BF16x2 (round to nearest even), lo in the low half.
QD uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Store EPU FP32 values as 16 bytes of output.
template <int OUT> QD void store_unit(void *y, int64_t e, const float *f)
{
    if (OUT == F32)
        stg16(static_cast<float *>(y) + e, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                                      __float_as_uint(f[2]), __float_as_uint(f[3])));
    else
        stg16(static_cast<uint16_t *>(y) + e, make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                         pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7])));
}

// 2^(code - 127); code 255 is NaN.
QD float e8m0_value(uint32_t code) { return code == 255u ? __int_as_float(0x7FC00000) : mx_inv_scale(254u - code); }

// ---------------------------------------------------------------------------
// current scaling: flat over the R*C codes
// ---------------------------------------------------------------------------
template <int FMT, int OUT>
__global__ void __launch_bounds__(kDqThreads) k_dq_cs(const uint8_t *__restrict__ q, const float *__restrict__ scale,
                                                      int64_t n, void *__restrict__ y)
{
    constexpr int EPU = OUT == F32 ? 4 : 8;
    const float s = *scale;
    const int64_t nu = n / EPU, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < nu; i0 += kDqUnits * stride) {
        uint2 a[kDqUnits];
#pragma unroll
        for (int j = 0; j < kDqUnits; j++) {
            const int64_t u = i0 + j * stride;
            if (u < nu) {
                if (EPU == 8) a[j] = *reinterpret_cast<const uint2 *>(q + u * 8);
                else a[j] = make_uint2(*reinterpret_cast<const uint32_t *>(q + u * 4), 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < kDqUnits; j++) {
            const int64_t u = i0 + j * stride;
            if (u >= nu) break;
            float f[8];
#pragma unroll
            for (int p = 0; p < EPU / 2; p++) {
                const uint32_t wd = p < 2 ? a[j].x : a[j].y;
                const float2 d = fp8x2_to_f32<FMT>((wd >> (16 * (p & 1))) & 0xFFFFu);
                f[2 * p] = __fmul_rn(d.x, s);
                f[2 * p + 1] = __fmul_rn(d.y, s);
            }
            store_unit<OUT>(y, u * EPU, f);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < n - nu * EPU) {
        const int64_t t = nu * EPU + threadIdx.x;
        const float v = __fmul_rn(fp8x2_to_f32<FMT>(q[t]).x, s);
        if (OUT == F32) static_cast<float *>(y)[t] = v;
        else static_cast<uint16_t *>(y)[t] = (uint16_t)bf16_bits(v);
    }
}

// ---------------------------------------------------------------------------
// FP8 block-scaled codes.  KIND 0: MX row, e [R, C/32]; 1: MX col, e [R/32, C];
// 2: blockwise 1x128, s [R, C/128]; 3: blockwise 128x128, s [R/128, C/128].
// ---------------------------------------------------------------------------
template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(kDqThreads) k_dq_blocks(const uint8_t *__restrict__ q, const void *__restrict__ sc,
                                                          int64_t R, int64_t C, int bx_log2, void *__restrict__ y)
{
    constexpr int EPU = OUT == F32 ? 4 : 8;
    constexpr int CB = EPU;   // code bytes per unit
    const int BX = 1 << bx_log2, BY = kDqThreads >> bx_log2;
    const int tx = threadIdx.x & (BX - 1), ty = threadIdx.x >> bx_log2;
    const int64_t upr = C / EPU;
    const int64_t u = (int64_t)blockIdx.y * BX + tx;
    if (u >= upr) return;
    const int64_t c = u * EPU;
    const int64_t grp = blockIdx.x;

    uint2 a[kDqRows];
    uint2 e8[kDqRows];   // MX columnwise: the unit's EPU scale codes
    float fac[kDqRows];
    // MX columnwise: with BY <= 8 a thread's kDqRows rows (BY apart, from a
    // multiple of kDqRows * BY) lie in one 32-row block and share the unit's
    // scale codes, loaded and decoded once.
    const bool one_blk = KIND == 1 && BY * kDqRows <= 32;
    float ef[EPU];
#pragma unroll
    for (int i = 0; i < kDqRows; i++) {
        const int64_t r = (grp * kDqRows + i) * BY + ty;
        if (r >= R) break;
        const uint8_t *qp = q + r * C + c;
        if (CB == 8) a[i] = *reinterpret_cast<const uint2 *>(qp);
        else a[i] = make_uint2(*reinterpret_cast<const uint32_t *>(qp), 0u);
        if (KIND == 0) fac[i] = e8m0_value(static_cast<const uint8_t *>(sc)[r * (C / 32) + c / 32]);
        if (KIND == 1 && (i == 0 || !one_blk)) {
            const uint8_t *ep = static_cast<const uint8_t *>(sc) + (r / 32) * C + c;
            e8[i] = EPU == 8 ? *reinterpret_cast<const uint2 *>(ep) : make_uint2(*reinterpret_cast<const uint32_t *>(ep), 0u);
        }
        if (KIND == 2) fac[i] = static_cast<const float *>(sc)[r * (C / 128) + c / 128];
        if (KIND == 3) fac[i] = static_cast<const float *>(sc)[(r / 128) * (C / 128) + c / 128];
    }
#pragma unroll
    for (int i = 0; i < kDqRows; i++) {
        const int64_t r = (grp * kDqRows + i) * BY + ty;
        if (r >= R) break;
        float f[8];
        if (KIND == 1 && (i == 0 || !one_blk)) {
#pragma unroll
            for (int p = 0; p < EPU; p++) ef[p] = e8m0_value(((p < 4 ? e8[i].x : e8[i].y) >> (8 * (p & 3))) & 0xFFu);
        }
#pragma unroll
        for (int p = 0; p < EPU / 2; p++) {
            const uint32_t wd = p < 2 ? a[i].x : a[i].y;
            const float2 d = fp8x2_to_f32<FMT>((wd >> (16 * (p & 1))) & 0xFFFFu);
            if (KIND == 1) {
                f[2 * p] = __fmul_rn(d.x, ef[2 * p]);
                f[2 * p + 1] = __fmul_rn(d.y, ef[2 * p + 1]);
            } else {
                f[2 * p] = __fmul_rn(d.x, fac[i]);
                f[2 * p + 1] = __fmul_rn(d.y, fac[i]);
            }
        }
        store_unit<OUT>(y, r * C + c, f);
    }
}

// ---------------------------------------------------------------------------
// NVFP4: a unit is one 16-element row segment of a block (8 code bytes, one
// block scale, so the factor sb * s_g is formed once per 16 outputs).  The
// E2M1 pairs decode to f16x2 and widen to FP32 by a mixed-precision add of
// -0 (exact; FMA pipe); the products are packed FP32 multiplies.
// BLK 0: 1x16, sb [R, C/16]; 1: 16x16, sb [R/16, C/16].
// ---------------------------------------------------------------------------
QD float f16_lo_f32(uint32_t h2)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.f16 %0, l, 0f80000000;\n\t}" : "=f"(r) : "r"(h2));
    return r;
}
QD float f16_hi_f32(uint32_t h2)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.f16 %0, h, 0f80000000;\n\t}" : "=f"(r) : "r"(h2));
    return r;
}
// The 8 E2M1 codes of a word (code j in bits 4j+3..4j) as FP32, scaled by fac.
QD void fp4x8_scaled(uint32_t w, float fac, float *f)
{
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
#pragma unroll
    for (int p = 0; p < 4; p++) {
        f[2 * p] = f16_lo_f32(h[p]);
        f[2 * p + 1] = f16_hi_f32(h[p]);
        mul2(f[2 * p], f[2 * p + 1], fac, fac);
    }
}

// 16 FP32 values as 32 bytes (BF16) or 64 bytes (FP32) of output at element
// e; W32: y is 32-byte aligned and each 32 bytes leave in one store (a
// lane's 16-byte halves would each fill only half of 32 sectors per warp
// store).
template <int OUT, bool W32> QD void store16(void *y, int64_t e, const float *f)
{
    if (OUT == F32) {
        float *d = static_cast<float *>(y) + e;
        const uint4 v0 = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
        const uint4 v1 = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]), __float_as_uint(f[7]));
        const uint4 v2 = make_uint4(__float_as_uint(f[8]), __float_as_uint(f[9]), __float_as_uint(f[10]), __float_as_uint(f[11]));
        const uint4 v3 = make_uint4(__float_as_uint(f[12]), __float_as_uint(f[13]), __float_as_uint(f[14]), __float_as_uint(f[15]));
        if (W32) {
            stg32(d, v0, v1);
            stg32(d + 8, v2, v3);
        } else {
            stg16(d, v0);
            stg16(d + 4, v1);
            stg16(d + 8, v2);
            stg16(d + 12, v3);
        }
    } else {
        uint16_t *d = static_cast<uint16_t *>(y) + e;
        const uint4 v0 = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        const uint4 v1 = make_uint4(pack_bf16x2(f[8], f[9]), pack_bf16x2(f[10], f[11]), pack_bf16x2(f[12], f[13]),
                                    pack_bf16x2(f[14], f[15]));
        if (W32) {
            stg32(d, v0, v1);
        } else {
            stg16(d, v0);
            stg16(d + 8, v1);
        }
    }
}

template <int BLK, int OUT, bool W32>
__global__ void __launch_bounds__(kDqThreads) k_dq_fp4(const uint8_t *__restrict__ q, const uint8_t *__restrict__ sb,
                                                       const float *__restrict__ s_global, int64_t R, int64_t C,
                                                       int bx_log2, void *__restrict__ y)
{
    const int BX = 1 << bx_log2, BY = kDqThreads >> bx_log2;
    const int tx = threadIdx.x & (BX - 1), ty = threadIdx.x >> bx_log2;
    const int64_t upr = C / 16;
    const int64_t u = (int64_t)blockIdx.y * BX + tx;
    if (u >= upr) return;
    const float sg = *s_global;
    const int64_t r0 = (int64_t)blockIdx.x * (kDqRows * BY) + ty;
    uint2 a[kDqRows];
    uint32_t code[kDqRows];
#pragma unroll
    for (int i = 0; i < kDqRows; i++) {
        const int64_t r = r0 + (int64_t)i * BY;
        if (r < R) {
            a[i] = *reinterpret_cast<const uint2 *>(q + r * (C / 2) + u * 8);
            code[i] = sb[(BLK == 0 ? r : r / 16) * upr + u];
        }
    }
#pragma unroll
    for (int i = 0; i < kDqRows; i++) {
        const int64_t r = r0 + (int64_t)i * BY;
        if (r >= R) break;
        const float fac = __fmul_rn(e4m3_value(code[i]), sg);
        float f[16];
        fp4x8_scaled(a[i].x, fac, f);
        fp4x8_scaled(a[i].y, fac, f + 8);
        store16<OUT, W32>(y, r * C + u * 16, f);
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

cudaError_t launch_dq_cs(const uint8_t *q, const float *s, int64_t R, int64_t C, int fmt, int out, void *y,
                         cudaStream_t st)
{
    const int64_t n = R * C;
    if (n == 0) return cudaSuccess;
    const int epu = out == F32 ? 4 : 8;
    int64_t blocks = (n / epu + (int64_t)kDqThreads * kDqUnits - 1) / ((int64_t)kDqThreads * kDqUnits);
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (fmt == E4M3) {
        if (out == F32) k_dq_cs<E4M3, F32><<<(unsigned)blocks, kDqThreads, 0, st>>>(q, s, n, y);
        else k_dq_cs<E4M3, BF16><<<(unsigned)blocks, kDqThreads, 0, st>>>(q, s, n, y);
    } else {
        if (out == F32) k_dq_cs<E5M2, F32><<<(unsigned)blocks, kDqThreads, 0, st>>>(q, s, n, y);
        else k_dq_cs<E5M2, BF16><<<(unsigned)blocks, kDqThreads, 0, st>>>(q, s, n, y);
    }
    return cudaGetLastError();
}

template <int KIND>
static cudaError_t dq_blocks_t(const uint8_t *q, const void *sc, int64_t R, int64_t C, int fmt, int out, void *y,
                               cudaStream_t st)
{
    if (R == 0 || C == 0) return cudaSuccess;
    const int epu = out == F32 ? 4 : 8;
    const int64_t upr = C / epu;
    int lg = 0;
    while ((1 << lg) < upr && lg < 8) lg++;
    const int BY = kDqThreads >> lg;
    const int64_t gu = (upr + (1 << lg) - 1) >> lg;                                   // unit blocks of a row
    const int64_t gr = (R + (int64_t)BY * kDqRows - 1) / ((int64_t)BY * kDqRows);   // row groups
    if (gu > 65535 || gr > 2147483647LL) return cudaErrorInvalidConfiguration;
    const dim3 gridxy((unsigned)gr, (unsigned)gu);
#define DQ_LAUNCH(F, O) k_dq_blocks<KIND, F, O><<<gridxy, kDqThreads, 0, st>>>(q, sc, R, C, lg, y)
    if (fmt == E4M3) {
        if (out == F32) DQ_LAUNCH(E4M3, F32);
        else DQ_LAUNCH(E4M3, BF16);
    } else {
        if (out == F32) DQ_LAUNCH(E5M2, F32);
        else DQ_LAUNCH(E5M2, BF16);
    }
#undef DQ_LAUNCH
    return cudaGetLastError();
}

cudaError_t launch_dq_mxfp8(const uint8_t *q, const uint8_t *e, int64_t R, int64_t C, int fmt, int dir, int out,
                            void *y, cudaStream_t st)
{
    return dir == 0 ? dq_blocks_t<0>(q, e, R, C, fmt, out, y, st) : dq_blocks_t<1>(q, e, R, C, fmt, out, y, st);
}

cudaError_t launch_dq_blockwise(const uint8_t *q, const float *s, int64_t R, int64_t C, int tile, int out, void *y,
                                cudaStream_t st)
{
    return tile == 0 ? dq_blocks_t<2>(q, s, R, C, E4M3, out, y, st) : dq_blocks_t<3>(q, s, R, C, E4M3, out, y, st);
}

cudaError_t launch_dq_nvfp4(const uint8_t *q, const uint8_t *sb, const float *s_g, int64_t R, int64_t C, int blk,
                            int out, void *y, cudaStream_t st)
{
    if (R == 0 || C == 0) return cudaSuccess;
    const int64_t upr = C / 16;   // units (16 elements) per row
    int lg = 0;
    while ((1 << lg) < upr && lg < 8) lg++;
    const int BY = kDqThreads >> lg;
    const int64_t gu = (upr + (1 << lg) - 1) >> lg;                                   // unit blocks of a row
    const int64_t gr = (R + (int64_t)BY * kDqRows - 1) / ((int64_t)BY * kDqRows);   // row groups
    if (gu > 65535 || gr > 2147483647LL) return cudaErrorInvalidConfiguration;
    const dim3 gridxy((unsigned)gr, (unsigned)gu);
    const bool w32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
#define DQ4(B, O)                                                                                \
    (w32 ? k_dq_fp4<B, O, true><<<gridxy, kDqThreads, 0, st>>>(q, sb, s_g, R, C, lg, y)          \
         : k_dq_fp4<B, O, false><<<gridxy, kDqThreads, 0, st>>>(q, sb, s_g, R, C, lg, y))
    if (blk == 0) {
        if (out == F32) DQ4(0, F32);
        else DQ4(0, BF16);
    } else {
        if (out == F32) DQ4(1, F32);
        else DQ4(1, BF16);
    }
#undef DQ4
    return cudaGetLastError();
}

}  // namespace qk
