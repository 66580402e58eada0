// DeepSeek-V3-like blockwise FP8 quantize (a6: 1x128, a7: 128x128).
//
// "Mixed-precision training: fp16 to fp8", recipe 4 "Blockwise scaling" and
// the "Blockwise scaling" flow: E4M3 only, activations / gradients on 1x128
// tiles, weights on 128x128 tiles, FP32 scales; the wgrad operand is
// X^T[k, m][1x128], i.e. 128x1 blocks along M written transposed; for the
// 2D tiles the transposed copy holds the same values.
// Per tile: b = max|x|, alpha = 448 / b (b = 0 -> 1, overflow -> FLT_MAX),
// s = 1 / alpha, q = RTNE-saturate(alpha * x).
//
// A CTA owns 128 rows x (32*VEC) columns, i.e. exactly one 128-row block in
// M and 2 (BF16) or 1 (FP32) 128-column blocks in K.  Column maxima over the
// 128 rows are combined across the 8 warps in shared memory; the columnwise
// codes (own per-column scales) are produced directly in column order and
// staged in shared memory for full 128-byte transposed row writes.
#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

template <int DT, int TILE>
__global__ void __launch_bounds__(kThreads) k_blockwise(const void *__restrict__ x, int64_t M, int64_t K,
                                                        uint8_t *__restrict__ q_row, float *__restrict__ s_row,
                                                        uint8_t *__restrict__ q_colT, float *__restrict__ s_colT,
                                                        int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, BYTES = In<DT>::BYTES, TC = 32 * VEC, CW = VEC / 4, LPB = 128 / VEC;
    constexpr int NT = TC / 128;   // 128-column blocks per CTA
    __shared__ __align__(16) uint8_t sT[TC * kTileRows];
    __shared__ uint32_t red[kWarps][TC];
    __shared__ float calpha[TC];

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

    if (TILE == 0) {
        // ---------------- 1x128 rowwise ----------------
        if (q_row != nullptr) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; r++) {
                const uint32_t b = group_max<LPB>(absmax_bits<DT>(v[r]));
                const float alpha = alpha_from_amax(448.0f, __uint_as_float(b));
                if (colok && m0 + r < M) {
                    uint32_t o[CW];
#pragma unroll
                    for (int w = 0; w < CW; w++)
                        o[w] = cvt_fp8x4<E4M3>(__fmul_rn(alpha, elem<DT>(v[r], 4 * w)), __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 1)),
                                               __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 2)), __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 3)));
                    uint8_t *dst = q_row + (m0 + r) * K + k0;
                    if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                    else stg4(dst, o[0]);
                    if (lane % LPB == 0) {
                        s_row[(m0 + r) * (K / 128) + k0 / 128] = __fdiv_rn(1.0f, alpha);
                        flag_nonfinite(status, b);
                    }
                }
            }
        }
        if (q_colT == nullptr) return;
        // ---------------- 128x1 columnwise, transposed ----------------
        {
            uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; r++) {
                acc.x = colmax_word<DT>(acc.x, v[r].x);
                acc.y = colmax_word<DT>(acc.y, v[r].y);
                acc.z = colmax_word<DT>(acc.z, v[r].z);
                acc.w = colmax_word<DT>(acc.w, v[r].w);
            }
#pragma unroll
            for (int j = 0; j < VEC; j++) red[warp][lane * VEC + j] = colmax_bits<DT>(acc, j);
        }
        __syncthreads();
        for (int col = threadIdx.x; col < TC; col += kThreads) {
            uint32_t b = 0;
#pragma unroll
            for (int w = 0; w < kWarps; w++) b = max(b, red[w][col]);
            const float alpha = alpha_from_amax(448.0f, __uint_as_float(b));
            calpha[col] = alpha;
            const int64_t kg = tk * TC + col;
            if (kg < K) {
                s_colT[kg * (M / 128) + tm] = __fdiv_rn(1.0f, alpha);
                flag_nonfinite(status, b);
            }
        }
        __syncthreads();
        if (colok) {
#pragma unroll
            for (int j = 0; j < VEC; j++) {
                const int col = lane * VEC + j;
                const float alpha = calpha[col];
                uint32_t c[4];
#pragma unroll
                for (int g = 0; g < 4; g++)
                    c[g] = cvt_fp8x4<E4M3>(__fmul_rn(alpha, elem<DT>(v[4 * g], j)), __fmul_rn(alpha, elem<DT>(v[4 * g + 1], j)),
                                           __fmul_rn(alpha, elem<DT>(v[4 * g + 2], j)), __fmul_rn(alpha, elem<DT>(v[4 * g + 3], j)));
                *reinterpret_cast<uint4 *>(sT + col * kTileRows + (warp ^ (lane & 7)) * 16) = make_uint4(c[0], c[1], c[2], c[3]);
            }
        }
    } else {
        // ---------------- 128x128: one scale per tile ----------------
        uint32_t b = 0;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) b = max(b, absmax_bits<DT>(v[r]));
        b = group_max<LPB>(b);
        __shared__ uint32_t tred[kWarps][NT];
        if (lane % LPB == 0) tred[warp][lane / LPB] = b;
        __syncthreads();
        b = 0;
#pragma unroll
        for (int w = 0; w < kWarps; w++) b = max(b, tred[w][lane / LPB]);
        const float alpha = alpha_from_amax(448.0f, __uint_as_float(b));
        if (colok && warp == 0 && lane % LPB == 0) {
            const float s = __fdiv_rn(1.0f, alpha);
            const int64_t kb = k0 / 128;
            if (s_row != nullptr) s_row[tm * (K / 128) + kb] = s;
            if (s_colT != nullptr) s_colT[kb * (M / 128) + tm] = s;
            flag_nonfinite(status, b);
        }
        if (colok) {
            uint32_t code[kRowsPerWarp][CW];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; r++)
#pragma unroll
                for (int w = 0; w < CW; w++)
                    code[r][w] = cvt_fp8x4<E4M3>(__fmul_rn(alpha, elem<DT>(v[r], 4 * w)), __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 1)),
                                                 __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 2)), __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 3)));
            if (q_row != nullptr) {
                uint8_t *dst = q_row + m0 * K + k0;
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; r++) {
                    if (CW == 2) stg8(dst + (int64_t)r * K, code[r][0], code[r][CW - 1]);
                    else stg4(dst + (int64_t)r * K, code[r][0]);
                }
            }
            if (q_colT != nullptr) {
#pragma unroll
                for (int w = 0; w < CW; w++) {
                    uint32_t c[4][4];
#pragma unroll
                    for (int g = 0; g < 4; g++)
                        transpose4x4(code[4 * g][w], code[4 * g + 1][w], code[4 * g + 2][w], code[4 * g + 3][w],
                                     c[0][g], c[1][g], c[2][g], c[3][g]);
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int col = lane * VEC + 4 * w + i;
                        *reinterpret_cast<uint4 *>(sT + col * kTileRows + (warp ^ (lane & 7)) * 16) =
                            make_uint4(c[i][0], c[i][1], c[i][2], c[i][3]);
                    }
                }
            }
        }
        if (q_colT == nullptr) return;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < TC * 8 / kThreads; it++) {
        const int idx = it * kThreads + threadIdx.x;
        const int col = idx >> 3, ch = idx & 7;
        const int64_t kg = tk * TC + col, mg = tm * kTileRows + ch * 16;
        if (kg < K && mg < M) {
            const int phys = ch ^ ((col / VEC) & 7);
            stg16(q_colT + kg * M + mg, *reinterpret_cast<const uint4 *>(sT + col * kTileRows + phys * 16));
        }
    }
}

template <int DT, int TILE>
static cudaError_t bw_t(const void *x, int64_t M, int64_t K, uint8_t *q_row, float *s_row, uint8_t *q_colT,
                        float *s_colT, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    const int64_t tiles = ((M + kTileRows - 1) / kTileRows) * ((K + TC - 1) / TC);
    k_blockwise<DT, TILE><<<(unsigned)tiles, kThreads, 0, st>>>(x, M, K, q_row, s_row, q_colT, s_colT, status);
    return cudaGetLastError();
}

cudaError_t launch_blockwise(const void *x, int dt, int64_t M, int64_t K, int tile, uint8_t *q_row, float *s_row,
                             uint8_t *q_colT, float *s_colT, int32_t *status, cudaStream_t st)
{
    if (dt == BF16)
        return tile == 0 ? bw_t<BF16, 0>(x, M, K, q_row, s_row, q_colT, s_colT, status, st)
                         : bw_t<BF16, 1>(x, M, K, q_row, s_row, q_colT, s_colT, status, st);
    return tile == 0 ? bw_t<F32, 0>(x, M, K, q_row, s_row, q_colT, s_colT, status, st)
                     : bw_t<F32, 1>(x, M, K, q_row, s_row, q_colT, s_colT, status, st);
}

}  // namespace qk
