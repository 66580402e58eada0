// MXFP8 quantize, rowwise 1x32 and columnwise 32x1, in one pass (a4, a5).
//
// "Mixed-precision training: fp16 to fp8", section "MXFP8": every 32
// elements share one E8M0 scale (an FP32 exponent field), value = element x
// scale; section "MXFP8 recipe": rowwise and columnwise copies differ only in
// the quantization direction, neither is transposed in memory.
// Scale code = clamp(floor(log2 b) - emax + 127, 0, 254), emax = 8 (E4M3) or
// 15 (E5M2), b = 0 -> 127; q = RTNE-saturate(x * 2^(127 - code)).
//
// A CTA owns 128 rows x (32*VEC) columns.  Rowwise: the 1x32 block of a row
// spans 32/VEC lanes, reduced with two or three xor-shuffles.  Columnwise:
// each warp reduces its 16 rows per column in registers, the two warps of a
// 32-row block exchange their partial maxima through shared memory.  Both
// outputs are written in the [M, K] layout straight from registers.
#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads) k_mxfp8(const void *__restrict__ x, int64_t M, int64_t K,
                                                    uint8_t *__restrict__ q_row, uint8_t *__restrict__ e_row,
                                                    uint8_t *__restrict__ q_col, uint8_t *__restrict__ e_col,
                                                    int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, BYTES = In<DT>::BYTES, TC = 32 * VEC, CW = VEC / 4, LPB = 32 / VEC;
    __shared__ uint4 part[kWarps][32];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_k = (K + TC - 1) / TC;
    const int64_t tm = blockIdx.x / tiles_k, tk = blockIdx.x - tm * tiles_k;
    const int64_t m0 = tm * kTileRows + warp * kRowsPerWarp;
    const int64_t k0 = tk * TC + lane * VEC;
    const bool colok = k0 < K;

    uint4 v[kRowsPerWarp];
    const char *base = static_cast<const char *>(x) + (m0 * K + k0) * BYTES;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; r++)
        v[r] = (colok && m0 + r < M) ? ldg_stream(base + (int64_t)r * K * BYTES) : make_uint4(0, 0, 0, 0);

    if (q_row != nullptr) {
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) {
            const uint32_t b = group_max<LPB>(absmax_bits<DT>(v[r]));
            const uint32_t code = mx_code<FMT>(b);
            const float inv = mx_inv_scale(code);
            if (colok && m0 + r < M) {
                uint32_t o[CW];
#pragma unroll
                for (int w = 0; w < CW; w++)
                    o[w] = cvt_fp8x4<FMT>(__fmul_rn(elem<DT>(v[r], 4 * w), inv), __fmul_rn(elem<DT>(v[r], 4 * w + 1), inv),
                                          __fmul_rn(elem<DT>(v[r], 4 * w + 2), inv), __fmul_rn(elem<DT>(v[r], 4 * w + 3), inv));
                uint8_t *dst = q_row + (m0 + r) * K + k0;
                if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                else stg4(dst, o[0]);
                if (lane % LPB == 0) {
                    e_row[(m0 + r) * (K / 32) + k0 / 32] = (uint8_t)code;
                    flag_nonfinite(status, b);
                }
            }
        }
    }

    if (q_col != nullptr) {
        uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) {
            acc.x = colmax_word<DT>(acc.x, v[r].x);
            acc.y = colmax_word<DT>(acc.y, v[r].y);
            acc.z = colmax_word<DT>(acc.z, v[r].z);
            acc.w = colmax_word<DT>(acc.w, v[r].w);
        }
        part[warp][lane] = acc;
        __syncthreads();
        const uint4 o4 = part[warp ^ 1][lane];
        acc.x = colmax_word<DT>(acc.x, o4.x);
        acc.y = colmax_word<DT>(acc.y, o4.y);
        acc.z = colmax_word<DT>(acc.z, o4.z);
        acc.w = colmax_word<DT>(acc.w, o4.w);
        if (colok && m0 < M) {
            float inv[VEC];
            uint32_t codes[VEC];
#pragma unroll
            for (int j = 0; j < VEC; j++) {
                const uint32_t b = colmax_bits<DT>(acc, j);
                codes[j] = mx_code<FMT>(b);
                inv[j] = mx_inv_scale(codes[j]);
                if ((warp & 1) == 0) flag_nonfinite(status, b);
            }
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; r++) {
                uint32_t o[CW];
#pragma unroll
                for (int w = 0; w < CW; w++)
                    o[w] = cvt_fp8x4<FMT>(__fmul_rn(elem<DT>(v[r], 4 * w), inv[4 * w]),
                                          __fmul_rn(elem<DT>(v[r], 4 * w + 1), inv[4 * w + 1]),
                                          __fmul_rn(elem<DT>(v[r], 4 * w + 2), inv[4 * w + 2]),
                                          __fmul_rn(elem<DT>(v[r], 4 * w + 3), inv[4 * w + 3]));
                uint8_t *dst = q_col + (m0 + r) * K + k0;
                if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                else stg4(dst, o[0]);
            }
            if ((warp & 1) == 0) {
                uint32_t s[CW];
#pragma unroll
                for (int w = 0; w < CW; w++)
                    s[w] = codes[4 * w] | (codes[4 * w + 1] << 8) | (codes[4 * w + 2] << 16) | (codes[4 * w + 3] << 24);
                uint8_t *dst = e_col + (m0 / 32) * K + k0;
                if (CW == 2) stg8(dst, s[0], s[CW - 1]);
                else stg4(dst, s[0]);
            }
        }
    }
}

template <int DT, int FMT>
static cudaError_t mx_t(const void *x, int64_t M, int64_t K, uint8_t *q_row, uint8_t *e_row, uint8_t *q_col,
                        uint8_t *e_col, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    const int64_t tiles = ((M + kTileRows - 1) / kTileRows) * ((K + TC - 1) / TC);
    k_mxfp8<DT, FMT><<<(unsigned)tiles, kThreads, 0, st>>>(x, M, K, q_row, e_row, q_col, e_col, status);
    return cudaGetLastError();
}

cudaError_t launch_mxfp8(const void *x, int dt, int64_t M, int64_t K, int fmt, uint8_t *q_row, uint8_t *e_row,
                         uint8_t *q_col, uint8_t *e_col, int32_t *status, cudaStream_t st)
{
    if (dt == BF16)
        return fmt == E4M3 ? mx_t<BF16, E4M3>(x, M, K, q_row, e_row, q_col, e_col, status, st)
                           : mx_t<BF16, E5M2>(x, M, K, q_row, e_row, q_col, e_col, status, st);
    return fmt == E4M3 ? mx_t<F32, E4M3>(x, M, K, q_row, e_row, q_col, e_col, status, st)
                       : mx_t<F32, E5M2>(x, M, K, q_row, e_row, q_col, e_col, status, st);
}

}  // namespace qk
