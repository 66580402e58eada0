// MXFP8 quantize, rowwise 1x32 and columnwise 32x1, in one pass (a4, a5).
//
// "Mixed-precision training: fp16 to fp8", section "MXFP8": every 32
// elements share one E8M0 scale (an FP32 exponent field), value = element x
// scale; section "MXFP8 recipe": rowwise and columnwise copies differ only in
// the quantization direction, neither is transposed in memory.
// Scale code = clamp(floor(log2 b) - emax + 127, 0, 254), emax = 8 (E4M3) or
// 15 (E5M2), b = 0 -> 127; q = RTNE-saturate(x * 2^(127 - code)).
//
// On the tile engine (128 x TC tiles in shared memory):
//  row pass - thread (warp w, lane l) handles rows 8w..8w+7, 16 bytes each;
//             a 1x32 block spans 32/VEC lanes (xor-shuffle max); codes and
//             scales go to global memory straight from registers;
//  col pass - thread (word column t % 128, 32-row block t / 128) reads the
//             32 words of its block, reduces each of its CPW columns, writes
//             the E8M0 codes, and parks the element codes in the stage (now
//             free) as a row-major [128][TC] byte tile;
//  copy-out - 16-byte row segments of q_col.
#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

template <int DT, int FMT>
__global__ void __launch_bounds__(kEngThreads, 1) k_mxfp8(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                          uint8_t *__restrict__ q_row, uint8_t *__restrict__ e_row,
                                                          uint8_t *__restrict__ q_col, uint8_t *__restrict__ e_col,
                                                          int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, CW = VEC / 4, LPB = 32 / VEC, CPW = 4 / In<DT>::BYTES;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, wc = t & 127, band = t >> 7;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;

    run_tiles(&tmap, tiles_m, tiles_k, TC, false, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        if (q_row != nullptr) {
            const int64_t k = kb + lane * VEC;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int r = 8 * warp + j;
                const uint4 v = lds16(st + r * kRowBytes + lane * 16);
                const uint32_t b = group_max<LPB>(absmax_bits<DT>(v));
                const uint32_t code = mx_code<FMT>(b);
                const float inv = mx_inv_scale(code);
                uint32_t o[CW];
                chunk_fp8<DT, FMT>(v, inv, o);
                if (mb + r < M && k < K) {
                    uint8_t *dst = q_row + (mb + r) * K + k;
                    if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                    else stg4(dst, o[0]);
                    if (lane % LPB == 0) {
                        e_row[(mb + r) * (K / 32) + k / 32] = (uint8_t)code;
                        flag_nonfinite(status, b);
                    }
                }
            }
        }
        if (q_col == nullptr) return;
        // ---- 32x1 blocks: one block of CPW columns per thread
        uint32_t w[32];
#pragma unroll
        for (int r = 0; r < 32; r++) w[r] = lds4(st + (32 * band + r) * kRowBytes + wc * 4);
        float inv[CPW];
        uint32_t codes = 0, bm[CPW];
        column_absmax<DT, 32>(w, bm);
#pragma unroll
        for (int c = 0; c < CPW; c++) {
            const uint32_t b = bm[c];
            const uint32_t code = mx_code<FMT>(b);
            inv[c] = mx_inv_scale(code);
            codes |= code << (8 * c);
            if (kb + wc * CPW < K && mb + 32 * band < M) flag_nonfinite(status, b);
        }
        const int64_t kg = kb + wc * CPW;
        if (kg < K && mb + 32 * band < M) {
            uint8_t *dst = e_col + (tm * 4 + band) * K + kg;
            if (CPW == 2) *reinterpret_cast<uint16_t *>(dst) = (uint16_t)codes;
            else *dst = (uint8_t)codes;
        }
        __syncthreads();   // every read of the stage is done: reuse it as a [128][TC] code tile
#pragma unroll
        for (int r = 0; r < 32; r += 4) {
            if (CPW == 2) {
                // rows r..r+3 x 2 columns -> two words of (row r c0, row r c1, row r+1 c0, row r+1 c1)
                float f[8];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    f[2 * q] = word_elem<DT>(w[r + q], 0);
                    f[2 * q + 1] = word_elem<DT>(w[r + q], 1);
                    mul2(f[2 * q], f[2 * q + 1], inv[0], inv[CPW - 1]);
                }
                const uint32_t p0 = cvt_fp8x4<FMT>(f[0], f[1], f[2], f[3]);
                const uint32_t p1 = cvt_fp8x4<FMT>(f[4], f[5], f[6], f[7]);
                uint8_t *base = st + (32 * band + r) * TC + wc * 2;
                *reinterpret_cast<uint16_t *>(base) = (uint16_t)p0;
                *reinterpret_cast<uint16_t *>(base + TC) = (uint16_t)(p0 >> 16);
                *reinterpret_cast<uint16_t *>(base + 2 * TC) = (uint16_t)p1;
                *reinterpret_cast<uint16_t *>(base + 3 * TC) = (uint16_t)(p1 >> 16);
            } else {
                float f[4];
#pragma unroll
                for (int q = 0; q < 4; q++) f[q] = word_elem<DT>(w[r + q], 0);
                mul2(f[0], f[1], inv[0], inv[0]);
                mul2(f[2], f[3], inv[0], inv[0]);
                const uint32_t p = cvt_fp8x4<FMT>(f[0], f[1], f[2], f[3]);
                uint8_t *base = st + (32 * band + r) * TC + wc;
                base[0] = (uint8_t)p;
                base[TC] = (uint8_t)(p >> 8);
                base[2 * TC] = (uint8_t)(p >> 16);
                base[3 * TC] = (uint8_t)(p >> 24);
            }
        }
        __syncthreads();
        constexpr int SEGS = TC / 16;   // 16-byte segments per code row
#pragma unroll
        for (int it = 0; it < kTileRowsE * SEGS / kEngThreads; it++) {
            const int idx = it * kEngThreads + t;
            const int r = idx / SEGS, sg = idx % SEGS;
            const int64_t m = mb + r, k = kb + 16 * sg;
            if (m < M && k < K) stg16(q_col + m * K + k, lds16(st + r * TC + 16 * sg));
        }
    });
}

template <int DT, int FMT>
static cudaError_t mx_t(const void *x, int64_t M, int64_t K, uint8_t *q_row, uint8_t *e_row, uint8_t *q_col,
                        uint8_t *e_col, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    alignas(64) CUtensorMap map;
    cudaError_t e = make_tile_map(&map, x, DT, M, K);
    if (e != cudaSuccess) return e;
    static bool attr = false;
    if (!attr) {
        e = cudaFuncSetAttribute(k_mxfp8<DT, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEngSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int64_t tiles = ((M + kTileRowsE - 1) / kTileRowsE) * ((K + TC - 1) / TC);
    const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
    k_mxfp8<DT, FMT><<<grid, kEngThreads, kEngSmem, st>>>(map, M, K, q_row, e_row, q_col, e_col, status);
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
