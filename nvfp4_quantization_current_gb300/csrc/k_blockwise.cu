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
// On the tile engine: a 128 x TC tile holds exactly one 128-row block in M
// and TC/128 blocks in K.
//  row pass - thread (warp w, lane l): rows 8w..8w+7, 16 bytes each; a
//             1x128 block spans 128/VEC lanes (xor-shuffle max);
//  col pass - thread (word column t % 128, 32-row quarter t / 128) reads 32
//             words; 1x128 (128x1 blocks along M): quarter maxima meet in
//             shared memory; the codes of each column are produced in
//             column order and parked in the stage (now free) as
//             [column][128 rows] with swizzled 16-byte chunks;
//  copy-out - 8 threads per q_colT row write its 128 bytes.
// For 128x128 the tile maxima come from the row-pass registers (warp
// shuffles, then shared memory across the 16 warps).
#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

// alpha = 448 / b and s = 1 / alpha for a tile maximum b.  For BF16 inputs b
// has a 7-bit mantissa m, b = (1 + m/128) 2^e; while alpha and s stay normal,
// RN(448 / b) = RN(448 / (1 + m/128)) 2^-e and RN(1 / alpha) =
// RN(1 / RN(448 / (1 + m/128))) 2^e exactly (rounding commutes with scaling
// by a power of two), so both come from two 128-entry tables per CTA and an
// exponent shift.  Exponent fields below 10 (b < 2^-117, where s would be
// subnormal), inf / NaN and FP32 inputs take the divisions.
struct BwScaleTab {
    float a[128], s[128];
};

template <int DT> QD void bw_scales(uint32_t b, const BwScaleTab &tab, float &alpha, float &s)
{
    const uint32_t E = b >> 23;
    if (DT == BF16 && E >= 10u && E < 255u) {
        const uint32_t m = (b >> 16) & 0x7Fu;
        const int sh = ((int)E - 127) << 23;
        alpha = __uint_as_float((uint32_t)((int)__float_as_uint(tab.a[m]) - sh));
        s = __uint_as_float((uint32_t)((int)__float_as_uint(tab.s[m]) + sh));
    } else {
        alpha = alpha_from_amax(448.0f, __uint_as_float(b));
        s = __fdiv_rn(1.0f, alpha);
    }
}

template <int DT, int TILE>
__global__ void __launch_bounds__(kEngThreads, 1) k_blockwise(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                              uint8_t *__restrict__ q_row, float *__restrict__ s_row,
                                                              uint8_t *__restrict__ q_colT, float *__restrict__ s_colT,
                                                              int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, CW = VEC / 4, LPB = 128 / VEC, CPW = 4 / In<DT>::BYTES;
    constexpr int NT = TC / 128;   // 128-column blocks per tile
    __shared__ uint32_t red[4][TC];
    __shared__ uint32_t tred[kEngWarps][NT];
    __shared__ BwScaleTab tab;
    if (DT == BF16 && threadIdx.x < 128) {
        const float a = __fdiv_rn(448.0f, 1.0f + (float)threadIdx.x * (1.0f / 128.0f));
        tab.a[threadIdx.x] = a;
        tab.s[threadIdx.x] = __fdiv_rn(1.0f, a);
    }   // visible after the engine's first barrier

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, wc = t & 127, quarter = t >> 7;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;

    run_tiles(&tmap, tiles_m, tiles_k, TC, false, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        const int64_t k = kb + lane * VEC;
        float colalpha[CPW];
        uint32_t w[32];

        if constexpr (TILE == 0) {
            // ---------------- 1x128 rowwise ----------------
            if (q_row != nullptr) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int r = 8 * warp + j;
                    const uint4 v = lds16(st + r * kRowBytes + lane * 16);
                    const uint32_t b = group_max<LPB>(absmax_bits<DT>(v));
                    float alpha, sc;
                    bw_scales<DT>(b, tab, alpha, sc);
                    uint32_t o[CW];
                    chunk_fp8<DT, E4M3>(v, alpha, o);
                    if (mb + r < M && k < K) {
                        uint8_t *dst = q_row + (mb + r) * K + k;
                        if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                        else stg4(dst, o[0]);
                        if (lane % LPB == 0) {
                            s_row[(mb + r) * (K / 128) + k / 128] = sc;
                            flag_nonfinite(status, b);
                        }
                    }
                }
            }
            if (q_colT == nullptr) return;
            // ---------------- 128x1 columnwise ----------------
#pragma unroll
            for (int r = 0; r < 32; r++) w[r] = lds4(st + (32 * quarter + r) * kRowBytes + wc * 4);
            {
                uint32_t bm[CPW];
                column_absmax<DT, 32>(w, bm);
#pragma unroll
                for (int c = 0; c < CPW; c++) red[quarter][wc * CPW + c] = bm[c];
            }
            __syncthreads();   // partial maxima visible; every read of the stage is done
#pragma unroll
            for (int c = 0; c < CPW; c++) {
                const int col = wc * CPW + c;
                const uint32_t b = max(max(red[0][col], red[1][col]), max(red[2][col], red[3][col]));
                float sc;
                bw_scales<DT>(b, tab, colalpha[c], sc);
                if (quarter == 0 && kb + col < K) {
                    s_colT[(kb + col) * (M / 128) + tm] = sc;
                    flag_nonfinite(status, b);
                }
            }
        } else {
            // ---------------- 128x128: one scale per tile ----------------
            uint4 v[8];
            uint32_t b = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                v[j] = lds16(st + (8 * warp + j) * kRowBytes + lane * 16);
                b = max(b, absmax_bits<DT>(v[j]));
            }
            b = group_max<LPB>(b);
            if (lane % LPB == 0) tred[warp][lane / LPB] = b;
            if (q_colT != nullptr) {
#pragma unroll
                for (int r = 0; r < 16; r++) w[r] = lds4(st + (16 * quarter + r) * kRowBytes + wc * 4);
#pragma unroll
                for (int r = 0; r < 16; r++) w[16 + r] = lds4(st + (16 * (quarter + 4) + r) * kRowBytes + wc * 4);
            }
            __syncthreads();   // tile maxima visible; every read of the stage is done
            uint32_t bt = 0;
#pragma unroll
            for (int q = 0; q < kEngWarps; q++) bt = max(bt, tred[q][lane / LPB]);
            float alpha, sc;
            bw_scales<DT>(bt, tab, alpha, sc);
            if (warp == 0 && lane % LPB == 0 && k < K) {
                if (s_row != nullptr) s_row[tm * (K / 128) + k / 128] = sc;
                if (s_colT != nullptr) s_colT[(k / 128) * (M / 128) + tm] = sc;
                flag_nonfinite(status, bt);
            }
            if (q_row != nullptr && k < K) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    uint32_t o[CW];
                    chunk_fp8<DT, E4M3>(v[j], alpha, o);
                    uint8_t *dst = q_row + (mb + 8 * warp + j) * K + k;
                    if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                    else stg4(dst, o[0]);
                }
            }
            if (q_colT == nullptr) return;
#pragma unroll
            for (int c = 0; c < CPW; c++) {
                const int blk = (wc * CPW + c) / 128;
                uint32_t bb = 0;
#pragma unroll
                for (int q = 0; q < kEngWarps; q++) bb = max(bb, tred[q][blk]);
                float sc;
                bw_scales<DT>(bb, tab, colalpha[c], sc);
            }
        }
        // ---- columnwise codes, column order, into the stage as [column][128 rows]
        // (1x128: rows 32*quarter..+31 in w; 128x128: rows 16*quarter..+15 and 16*(quarter+4)..+15)
#pragma unroll
        for (int c = 0; c < CPW; c++) {
            const int col = wc * CPW + c;
            uint32_t o[8];
            column_fp8<DT, E4M3, 32>(w, c, colalpha[c], o);
            const int ch0 = TILE == 0 ? 2 * quarter : quarter, ch1 = TILE == 0 ? 2 * quarter + 1 : quarter + 4;
            uint8_t *base = st + col * 128;
            *reinterpret_cast<uint4 *>(base + ((ch0 ^ (wc & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(base + ((ch1 ^ (wc & 7)) * 16)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < TC * 8 / kEngThreads; it++) {
            const int idx = it * kEngThreads + t;
            const int col = idx >> 3, ch = idx & 7;
            const int64_t kg = kb + col, mg = mb + ch * 16;
            if (kg < K && mg < M)
                stg16(q_colT + kg * M + mg, lds16(st + col * 128 + ((ch ^ ((col / CPW) & 7)) * 16)));
        }
    });
}

template <int DT, int TILE>
static cudaError_t bw_t(const void *x, int64_t M, int64_t K, uint8_t *q_row, float *s_row, uint8_t *q_colT,
                        float *s_colT, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    alignas(64) CUtensorMap map;
    cudaError_t e = make_tile_map(&map, x, DT, M, K);
    if (e != cudaSuccess) return e;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(k_blockwise<DT, TILE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEngSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int64_t tiles = ((M + kTileRowsE - 1) / kTileRowsE) * ((K + TC - 1) / TC);
    const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
    k_blockwise<DT, TILE><<<grid, kEngThreads, kEngSmem, st>>>(map, M, K, q_row, s_row, q_colT, s_colT, status);
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
