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
// nearest even.  Block-scaled kernels use a 2-D grid: x over 16-element
// chunks of a row, y over groups of 4 rows (grid-stride), so no index
// division happens per element and each thread has 4 independent loads in
// flight.
#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

constexpr int kDqRows = 4;

// Store 16 FP32 values (FP32 or BF16 output) at element offset e of y.
template <int OUT> QD void store16(void *y, int64_t e, const float *f)
{
    if (OUT == F32) {
        float *p = static_cast<float *>(y) + e;
#pragma unroll
        for (int i = 0; i < 4; i++)
            stg16(p + 4 * i, make_uint4(__float_as_uint(f[4 * i]), __float_as_uint(f[4 * i + 1]),
                                        __float_as_uint(f[4 * i + 2]), __float_as_uint(f[4 * i + 3])));
    } else {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; i++) w[i] = bf16_bits(f[2 * i]) | (bf16_bits(f[2 * i + 1]) << 16);
        uint16_t *p = static_cast<uint16_t *>(y) + e;
        stg16(p, make_uint4(w[0], w[1], w[2], w[3]));
        stg16(p + 8, make_uint4(w[4], w[5], w[6], w[7]));
    }
}

// 16 FP8 codes (a 16-byte vector) -> 16 FP32 values times per-element factors.
template <int FMT> QD void decode16(const uint4 &q, const float *fac, float *f)
{
#pragma unroll
    for (int w = 0; w < 4; w++) {
        const uint32_t c = word(q, w);
        const float2 a = fp8x2_to_f32<FMT>(c & 0xFFFFu), b = fp8x2_to_f32<FMT>(c >> 16);
        f[4 * w] = __fmul_rn(a.x, fac[4 * w]);
        f[4 * w + 1] = __fmul_rn(a.y, fac[4 * w + 1]);
        f[4 * w + 2] = __fmul_rn(b.x, fac[4 * w + 2]);
        f[4 * w + 3] = __fmul_rn(b.y, fac[4 * w + 3]);
    }
}

// ---------------------------------------------------------------------------
// current scaling: flat over the R*C codes
// ---------------------------------------------------------------------------
template <int FMT, int OUT>
__global__ void __launch_bounds__(256) k_dq_cs(const uint8_t *__restrict__ q, const float *__restrict__ scale, int64_t n,
                                               void *__restrict__ y)
{
    const float s = *scale;
    float fac[16];
#pragma unroll
    for (int i = 0; i < 16; i++) fac[i] = s;
    const int64_t nc = n / 16, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nc; i += 2 * stride) {
        const int64_t i1 = i + stride;
        const uint4 a = ldg_stream(q + i * 16);
        uint4 b = make_uint4(0, 0, 0, 0);
        if (i1 < nc) b = ldg_stream(q + i1 * 16);
        float f[16];
        decode16<FMT>(a, fac, f);
        store16<OUT>(y, i * 16, f);
        if (i1 < nc) {
            decode16<FMT>(b, fac, f);
            store16<OUT>(y, i1 * 16, f);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < n - nc * 16) {
        const int64_t t = nc * 16 + threadIdx.x;
        const float v = __fmul_rn(fp8x2_to_f32<FMT>(q[t]).x, s);
        if (OUT == F32) static_cast<float *>(y)[t] = v;
        else static_cast<uint16_t *>(y)[t] = (uint16_t)bf16_bits(v);
    }
}

// ---------------------------------------------------------------------------
// block-scaled FP8: MXFP8 (row / col), blockwise (1x128 / 128x128)
// KIND 0: MX row, e [R, C/32]; 1: MX col, e [R/32, C]; 2: BW 1x128, s [R, C/128];
// 3: BW 128x128, s [R/128, C/128].
// ---------------------------------------------------------------------------
// 2^(code - 127); code 255 is NaN.
QD float e8m0_value(uint32_t code) { return code == 255u ? __int_as_float(0x7FC00000) : mx_inv_scale(254u - code); }

template <int KIND> QD void chunk_factors(const void *sc, int64_t R, int64_t C, int64_t r, int64_t c, float *fac)
{
    if (KIND == 0) {
        const float f = e8m0_value(static_cast<const uint8_t *>(sc)[r * (C / 32) + c / 32]);
#pragma unroll
        for (int i = 0; i < 16; i++) fac[i] = f;
    } else if (KIND == 1) {
        const uint4 e = ldg_stream(static_cast<const uint8_t *>(sc) + (r / 32) * C + c);
#pragma unroll
        for (int i = 0; i < 16; i++) fac[i] = e8m0_value((word(e, i >> 2) >> (8 * (i & 3))) & 0xFFu);
    } else if (KIND == 2) {
        const float f = static_cast<const float *>(sc)[r * (C / 128) + c / 128];
#pragma unroll
        for (int i = 0; i < 16; i++) fac[i] = f;
    } else {
        const float f = static_cast<const float *>(sc)[(r / 128) * (C / 128) + c / 128];
#pragma unroll
        for (int i = 0; i < 16; i++) fac[i] = f;
    }
}

template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(256) k_dq_fp8_blocks(const uint8_t *__restrict__ q, const void *__restrict__ sc,
                                                       int64_t R, int64_t C, void *__restrict__ y)
{
    const int64_t cpr = C / 16;
    const int64_t cc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (cc >= cpr) return;
    const int64_t c = cc * 16;
    for (int64_t r0 = (int64_t)blockIdx.y * kDqRows; r0 < R; r0 += (int64_t)gridDim.y * kDqRows) {
        uint4 a[kDqRows];
#pragma unroll
        for (int i = 0; i < kDqRows; i++)
            if (r0 + i < R) a[i] = ldg_stream(q + (r0 + i) * C + c);
#pragma unroll
        for (int i = 0; i < kDqRows; i++) {
            if (r0 + i >= R) break;
            float fac[16], f[16];
            chunk_factors<KIND>(sc, R, C, r0 + i, c, fac);
            decode16<FMT>(a[i], fac, f);
            store16<OUT>(y, (r0 + i) * C + c, f);
        }
    }
}

// ---------------------------------------------------------------------------
// NVFP4: 16 elements (8 packed bytes) per chunk, one block scale per chunk.
// ---------------------------------------------------------------------------
template <int BLK, int OUT>
__global__ void __launch_bounds__(256) k_dq_nvfp4(const uint8_t *__restrict__ q, const uint8_t *__restrict__ sb,
                                                  const float *__restrict__ s_global, int64_t R, int64_t C,
                                                  void *__restrict__ y)
{
    const int64_t cpr = C / 16;
    const int64_t cc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (cc >= cpr) return;
    const float sg = *s_global;
    for (int64_t r0 = (int64_t)blockIdx.y * kDqRows; r0 < R; r0 += (int64_t)gridDim.y * kDqRows) {
        uint2 a[kDqRows];
#pragma unroll
        for (int i = 0; i < kDqRows; i++)
            if (r0 + i < R) a[i] = *reinterpret_cast<const uint2 *>(q + (r0 + i) * (C / 2) + cc * 8);
#pragma unroll
        for (int i = 0; i < kDqRows; i++) {
            const int64_t r = r0 + i;
            if (r >= R) break;
            const uint8_t code = BLK == 0 ? sb[r * cpr + cc] : sb[(r / 16) * cpr + cc];
            const float fac = __fmul_rn(e4m3_value(code), sg);
            float f[16];
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const uint32_t byte = ((b < 4 ? a[i].x : a[i].y) >> (8 * (b & 3))) & 0xFFu;
                const float2 p = fp4x2_to_f32(byte);
                f[2 * b] = __fmul_rn(p.x, fac);
                f[2 * b + 1] = __fmul_rn(p.y, fac);
            }
            store16<OUT>(y, r * C + cc * 16, f);
        }
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

static dim3 grid2d(int64_t R, int64_t C)
{
    const int64_t gx = (C / 16 + 255) / 256;
    int64_t gy = (R + kDqRows - 1) / kDqRows;
    const int64_t want = (int64_t)sm_count() * 8 / (gx > 0 ? gx : 1) + 1;
    if (gy > want) gy = want;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    return dim3((unsigned)gx, (unsigned)gy);
}

cudaError_t launch_dq_cs(const uint8_t *q, const float *s, int64_t R, int64_t C, int fmt, int out, void *y,
                         cudaStream_t st)
{
    const int64_t n = R * C;
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n / 16 + 511) / 512;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (fmt == E4M3) {
        if (out == F32) k_dq_cs<E4M3, F32><<<(unsigned)blocks, 256, 0, st>>>(q, s, n, y);
        else k_dq_cs<E4M3, BF16><<<(unsigned)blocks, 256, 0, st>>>(q, s, n, y);
    } else {
        if (out == F32) k_dq_cs<E5M2, F32><<<(unsigned)blocks, 256, 0, st>>>(q, s, n, y);
        else k_dq_cs<E5M2, BF16><<<(unsigned)blocks, 256, 0, st>>>(q, s, n, y);
    }
    return cudaGetLastError();
}

template <int KIND>
static cudaError_t dq_fp8_t(const uint8_t *q, const void *sc, int64_t R, int64_t C, int fmt, int out, void *y,
                            cudaStream_t st)
{
    if (R == 0 || C == 0) return cudaSuccess;
    const dim3 g = grid2d(R, C);
    if (fmt == E4M3) {
        if (out == F32) k_dq_fp8_blocks<KIND, E4M3, F32><<<g, 256, 0, st>>>(q, sc, R, C, y);
        else k_dq_fp8_blocks<KIND, E4M3, BF16><<<g, 256, 0, st>>>(q, sc, R, C, y);
    } else {
        if (out == F32) k_dq_fp8_blocks<KIND, E5M2, F32><<<g, 256, 0, st>>>(q, sc, R, C, y);
        else k_dq_fp8_blocks<KIND, E5M2, BF16><<<g, 256, 0, st>>>(q, sc, R, C, y);
    }
    return cudaGetLastError();
}

cudaError_t launch_dq_mxfp8(const uint8_t *q, const uint8_t *e, int64_t R, int64_t C, int fmt, int dir, int out,
                            void *y, cudaStream_t st)
{
    return dir == 0 ? dq_fp8_t<0>(q, e, R, C, fmt, out, y, st) : dq_fp8_t<1>(q, e, R, C, fmt, out, y, st);
}

cudaError_t launch_dq_blockwise(const uint8_t *q, const float *s, int64_t R, int64_t C, int tile, int out, void *y,
                                cudaStream_t st)
{
    return tile == 0 ? dq_fp8_t<2>(q, s, R, C, E4M3, out, y, st) : dq_fp8_t<3>(q, s, R, C, E4M3, out, y, st);
}

cudaError_t launch_dq_nvfp4(const uint8_t *q, const uint8_t *sb, const float *s_g, int64_t R, int64_t C, int blk,
                            int out, void *y, cudaStream_t st)
{
    if (R == 0 || C == 0) return cudaSuccess;
    const dim3 g = grid2d(R, C);
    if (blk == 0) {
        if (out == F32) k_dq_nvfp4<0, F32><<<g, 256, 0, st>>>(q, sb, s_g, R, C, y);
        else k_dq_nvfp4<0, BF16><<<g, 256, 0, st>>>(q, sb, s_g, R, C, y);
    } else {
        if (out == F32) k_dq_nvfp4<1, F32><<<g, 256, 0, st>>>(q, sb, s_g, R, C, y);
        else k_dq_nvfp4<1, BF16><<<g, 256, 0, st>>>(q, sb, s_g, R, C, y);
    }
    return cudaGetLastError();
}

}  // namespace qk
