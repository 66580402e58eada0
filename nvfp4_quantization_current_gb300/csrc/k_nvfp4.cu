// NVFP4 quantize (a8-a11): E2M1 codes, one E4M3 scale per 1x16 (or 16x16)
// block, one FP32 tensor scale; RTNE or stochastic rounding.
//
// "Mixed-precision training: fp16 to fp8", sections "NVFP4" (E2M1 values,
// two codes per byte, RTNE default, stochastic rounding option) and recipe 6
// (1x16 blocks, E4M3 block scale, extra FP32 global scale).  "From BF16 to
// FP8/FP4 ...", section 2.4: 16x16 2D scaling for weights, 1x16 for
// activations and gradients, stochastic rounding on gradients only; the FP4
// GEMM is TN-only, so a columnwise copy is stored transposed even for 2D
// weights ("Mixed-precision training ...", summary).
// Two-level scale: alpha_g = 2688 / amax, s_g = 1 / alpha_g; per block
// sb = E4M3((b * alpha_g) / 6) (b = 0 -> 1.0), enc = alpha_g / sb,
// q = E2M1(x * enc).
//
// The amax comes from the preceding amax pass (or the caller); this pass
// walks the tensor backwards for L2 reuse, like the current-scaling cast.
// CTA tile 128 x (32*VEC).  Rowwise 1x16 blocks span 16/VEC lanes; a
// columnwise 16x1 block is the 16 rows one thread holds, so its scale needs
// no communication; its codes are produced in column order and staged in
// shared memory for transposed writes.  For 16x16 tiles the transposed copy
// is the row codes turned around by an in-register nibble transpose.
#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

QD void nv_block_scale(uint32_t b, float alpha_g, uint32_t &sb, float &enc)
{
    if (b == 0) {
        sb = 0x38u;   // 1.0
        enc = alpha_g;
        return;
    }
    const float sbf = __fdiv_rn(__fmul_rn(__uint_as_float(b), alpha_g), 6.0f);
    sb = e4m3_code(sbf);
    const float sv = e4m3_value(sb);
    enc = (sv == 0.0f) ? 0.0f : __fdiv_rn(alpha_g, sv);
}

// 16 random bits for element e (0..7) of a Philox block.
QD uint32_t r16_of(const uint4 &R, int e) { return (word(R, e >> 1) >> (16 * (e & 1))) & 0xFFFFu; }

// In-place transpose of an 8x8 nibble matrix: a[i] nibble j -> a[j] nibble i.
QD void transpose8x8_nibbles(uint32_t *a)
{
#pragma unroll
    for (int i = 0; i < 4; i++) {   // 4x4 blocks
        uint32_t t = ((a[i] >> 16) ^ a[i + 4]) & 0x0000FFFFu;
        a[i + 4] ^= t;
        a[i] ^= t << 16;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 4)
#pragma unroll
        for (int j = 0; j < 2; j++) {   // 2x2 blocks
            uint32_t t = ((a[i + j] >> 8) ^ a[i + j + 2]) & 0x00FF00FFu;
            a[i + j + 2] ^= t;
            a[i + j] ^= t << 8;
        }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {   // single nibbles
        uint32_t t = ((a[i] >> 4) ^ a[i + 1]) & 0x0F0F0F0Fu;
        a[i + 1] ^= t;
        a[i] ^= t << 4;
    }
}

template <int DT, int BLK, int RND>
__global__ void __launch_bounds__(kThreads) k_nvfp4(const void *__restrict__ x, int64_t M, int64_t K,
                                                    const float *__restrict__ amax, uint64_t seed, uint64_t offset,
                                                    uint8_t *__restrict__ q_row, uint8_t *__restrict__ sb_row,
                                                    uint8_t *__restrict__ q_colT, uint8_t *__restrict__ sb_colT,
                                                    float *__restrict__ s_global, int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, BYTES = In<DT>::BYTES, TC = 32 * VEC, LPB = 16 / VEC;
    __shared__ __align__(16) uint8_t sT[TC * (kTileRows / 2)];
    __shared__ uint8_t sSB[kWarps * TC];

    const float A = *amax;
    const float alpha_g = alpha_from_amax(2688.0f, A);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *s_global = __fdiv_rn(1.0f, alpha_g);
        flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
    }
    const int64_t tiles_k = (K + TC - 1) / TC;
    if (M == 0 || tiles_k == 0) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)gridDim.x - 1 - blockIdx.x;   // backwards: L2-resident data first
    const int64_t tm = t / tiles_k, tk = t - tm * tiles_k;
    const int64_t m0 = tm * kTileRows + warp * kRowsPerWarp;
    const int64_t k0 = tk * TC + lane * VEC;
    const bool ok = (k0 < K) && (m0 < M);   // M % 16 == 0: a warp's rows are all valid or none

    uint4 v[kRowsPerWarp];
    const char *base = static_cast<const char *>(x) + (m0 * K + k0) * BYTES;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; r++) v[r] = ok ? ldg_stream(base + (int64_t)r * K * BYTES) : make_uint4(0, 0, 0, 0);

    uint32_t rowcode[kRowsPerWarp];   // VEC nibbles per row (BF16: 8 -> a word, FP32: 4 -> low half)

    if (BLK == 0) {
        // ---------------- 1x16 rowwise ----------------
        if (q_row != nullptr) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; r++) {
                const uint32_t b = group_max<LPB>(absmax_bits<DT>(v[r]));
                uint32_t sb;
                float enc;
                nv_block_scale(b, alpha_g, sb, enc);
                float y[8];
#pragma unroll
                for (int j = 0; j < 8; j++) y[j] = j < VEC ? __fmul_rn(elem<DT>(v[r], j < VEC ? j : 0), enc) : 0.0f;
                if (RND == 1) {
                    const int64_t i0 = (m0 + r) * K + k0;
                    const uint4 R = sr_bits(seed, offset + (uint64_t)(i0 >> 3), 0u);
                    const int e0 = (int)(i0 & 7);
#pragma unroll
                    for (int j = 0; j < VEC; j++) y[j] = sr_e2m1_value(y[j], r16_of(R, e0 + j));
                }
                rowcode[r] = cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
                if (ok) {
                    uint8_t *dst = q_row + (m0 + r) * (K / 2) + k0 / 2;
                    if (VEC == 8) stg4(dst, rowcode[r]);
                    else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)rowcode[r];
                    if (lane % LPB == 0) {
                        sb_row[(m0 + r) * (K / 16) + k0 / 16] = (uint8_t)sb;
                        flag_nonfinite(status, b);
                    }
                }
            }
        }
        if (q_colT == nullptr) return;
        // ---------------- 16x1 columnwise (in-thread blocks), transposed ----------------
        uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) {
            acc.x = colmax_word<DT>(acc.x, v[r].x);
            acc.y = colmax_word<DT>(acc.y, v[r].y);
            acc.z = colmax_word<DT>(acc.z, v[r].z);
            acc.w = colmax_word<DT>(acc.w, v[r].w);
        }
        if (ok) {
#pragma unroll
            for (int j = 0; j < VEC; j++) {
                const uint32_t b = colmax_bits<DT>(acc, j);
                uint32_t sb;
                float enc;
                nv_block_scale(b, alpha_g, sb, enc);
                float y[16];
#pragma unroll
                for (int r = 0; r < 16; r++) y[r] = __fmul_rn(elem<DT>(v[r], j), enc);
                if (RND == 1) {
                    const int64_t it0 = (k0 + j) * M + m0;   // multiple of 16
                    const uint4 R0 = sr_bits(seed, offset + (uint64_t)(it0 >> 3), 1u);
                    const uint4 R1 = sr_bits(seed, offset + (uint64_t)(it0 >> 3) + 1u, 1u);
#pragma unroll
                    for (int r = 0; r < 8; r++) {
                        y[r] = sr_e2m1_value(y[r], r16_of(R0, r));
                        y[r + 8] = sr_e2m1_value(y[r + 8], r16_of(R1, r));
                    }
                }
                const uint32_t lo = cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
                const uint32_t hi = cvt_fp4x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
                const int col = lane * VEC + j;
                *reinterpret_cast<uint2 *>(sT + col * (kTileRows / 2) + (warp ^ (lane & 7)) * 8) = make_uint2(lo, hi);
                sSB[warp * TC + col] = (uint8_t)sb;
                flag_nonfinite(status, b);
            }
        }
    } else {
        // ---------------- 16x16: one scale per tile ----------------
        uint32_t b = 0;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) b = max(b, absmax_bits<DT>(v[r]));
        b = group_max<LPB>(b);
        uint32_t sb;
        float enc;
        nv_block_scale(b, alpha_g, sb, enc);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) {
            float y[8];
#pragma unroll
            for (int j = 0; j < 8; j++) y[j] = j < VEC ? __fmul_rn(elem<DT>(v[r], j < VEC ? j : 0), enc) : 0.0f;
            if (RND == 1) {
                const int64_t i0 = (m0 + r) * K + k0;
                const uint4 R = sr_bits(seed, offset + (uint64_t)(i0 >> 3), 0u);
                const int e0 = (int)(i0 & 7);
#pragma unroll
                for (int j = 0; j < VEC; j++) y[j] = sr_e2m1_value(y[j], r16_of(R, e0 + j));
            }
            rowcode[r] = cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
        }
        if (ok) {
            if (q_row != nullptr) {
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; r++) {
                    uint8_t *dst = q_row + (m0 + r) * (K / 2) + k0 / 2;
                    if (VEC == 8) stg4(dst, rowcode[r]);
                    else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)rowcode[r];
                }
            }
            if (lane % LPB == 0) {
                if (sb_row != nullptr) sb_row[(m0 / 16) * (K / 16) + k0 / 16] = (uint8_t)sb;
                if (sb_colT != nullptr) sb_colT[(k0 / 16) * (M / 16) + m0 / 16] = (uint8_t)sb;
                flag_nonfinite(status, b);
            }
            if (q_colT != nullptr) {
                uint32_t lo[8], hi[8];
                if (VEC == 8) {
#pragma unroll
                    for (int r = 0; r < 8; r++) {
                        lo[r] = rowcode[r];
                        hi[r] = rowcode[r + 8];
                    }
                    transpose8x8_nibbles(lo);
                    transpose8x8_nibbles(hi);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; j++) {
                        uint32_t l = 0, h = 0;
#pragma unroll
                        for (int r = 0; r < 8; r++) {
                            l |= ((rowcode[r] >> (4 * j)) & 0xFu) << (4 * r);
                            h |= ((rowcode[r + 8] >> (4 * j)) & 0xFu) << (4 * r);
                        }
                        lo[j] = l;
                        hi[j] = h;
                    }
                }
#pragma unroll
                for (int j = 0; j < VEC; j++) {
                    const int col = lane * VEC + j;
                    *reinterpret_cast<uint2 *>(sT + col * (kTileRows / 2) + (warp ^ (lane & 7)) * 8) = make_uint2(lo[j], hi[j]);
                }
            }
        }
        if (q_colT == nullptr) return;
    }

    __syncthreads();
    // transposed codes: 8 lanes per q_colT row, one 8-byte chunk (16 rows of m) each
#pragma unroll
    for (int it = 0; it < TC * 8 / kThreads; it++) {
        const int idx = it * kThreads + threadIdx.x;
        const int col = idx >> 3, ch = idx & 7;
        const int64_t kg = tk * TC + col, mg = tm * kTileRows + ch * 16;
        if (kg < K && mg < M) {
            const int phys = ch ^ ((col / VEC) & 7);
            const uint2 val = *reinterpret_cast<const uint2 *>(sT + col * (kTileRows / 2) + phys * 8);
            stg8(q_colT + kg * (M / 2) + mg / 2, val.x, val.y);
        }
    }
    if (BLK == 0) {
        // columnwise block scales: 8 per column of the tile (one per warp)
        const int64_t rows_left = (M - tm * kTileRows) / 16;
        const int nb = rows_left < kWarps ? (int)rows_left : kWarps;
        for (int col = threadIdx.x; col < TC; col += kThreads) {
            const int64_t kg = tk * TC + col;
            if (kg >= K) continue;
            uint8_t *dst = sb_colT + kg * (M / 16) + tm * kWarps;
            if (nb == kWarps && (M % 128) == 0) {
                uint32_t w0 = 0, w1 = 0;
#pragma unroll
                for (int w = 0; w < 4; w++) {
                    w0 |= (uint32_t)sSB[w * TC + col] << (8 * w);
                    w1 |= (uint32_t)sSB[(w + 4) * TC + col] << (8 * w);
                }
                stg8(dst, w0, w1);
            } else {
                for (int w = 0; w < nb; w++) dst[w] = sSB[w * TC + col];
            }
        }
    }
}

template <int DT, int BLK, int RND>
static cudaError_t nv_t(const void *x, int64_t M, int64_t K, const float *amax, uint64_t seed, uint64_t offset,
                        uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT, float *s_global,
                        int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    int64_t tiles = ((M + kTileRows - 1) / kTileRows) * ((K + TC - 1) / TC);
    if (tiles < 1) tiles = 1;   // an empty tensor still gets its global scale
    k_nvfp4<DT, BLK, RND><<<(unsigned)tiles, kThreads, 0, st>>>(x, M, K, amax, seed, offset, q_row, sb_row, q_colT,
                                                                sb_colT, s_global, status);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4(const void *x, int dt, int64_t M, int64_t K, int blk, int rnd, uint64_t seed,
                         uint64_t offset, const float *amax, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT,
                         uint8_t *sb_colT, float *s_global, int32_t *status, cudaStream_t st)
{
#define NV_ARGS x, M, K, amax, seed, offset, q_row, sb_row, q_colT, sb_colT, s_global, status, st
    if (dt == BF16) {
        if (blk == 0) return rnd == 0 ? nv_t<BF16, 0, 0>(NV_ARGS) : nv_t<BF16, 0, 1>(NV_ARGS);
        return rnd == 0 ? nv_t<BF16, 1, 0>(NV_ARGS) : nv_t<BF16, 1, 1>(NV_ARGS);
    }
    if (blk == 0) return rnd == 0 ? nv_t<F32, 0, 0>(NV_ARGS) : nv_t<F32, 0, 1>(NV_ARGS);
    return rnd == 0 ? nv_t<F32, 1, 0>(NV_ARGS) : nv_t<F32, 1, 1>(NV_ARGS);
#undef NV_ARGS
}

}  // namespace qk
