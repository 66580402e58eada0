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
// On the tile engine (the amax comes from the preceding amax pass or the
// caller; tiles are walked backwards for L2 reuse), thread (warp w, lane l)
// holds rows 8w..8w+7 x one 16-byte column chunk in registers.
//  1x16 rowwise - a block spans 16/VEC lanes; stochastic rounding draws one
//                 Philox block (8 elements) per thread and row;
//  16x1 colwise - a block is the 8 rows of warps 2p and 2p+1: their column
//                 maxima meet in shared memory; each column's 8 values are
//                 encoded into one word of row nibbles (SR: one Philox block
//                 per column), parked in the consumed stage and written as
//                 q_colT rows;
//  16x16        - the block maximum spans 2 warps x 16/VEC lanes; the
//                 transposed copy is the row codes nibble-transposed.
#include <cstring>

#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

// With 1x16 blocks both per-CTA lookup tables of k_nvfp4 hold 16
// interleaved copies (entry e, copy j at word 16 e + j) and lane l reads copy
// l % 16, so lanes that look up different entries meet in one bank at most in
// pairs (with one copy up to four entries share a bank).  16x16 lookups are
// uniform across the lanes of a block and keep one copy.
template <int BLK> constexpr int kTabCopies = BLK == 0 ? 16 : 1;

// Block scale code sb = E4M3(RN(RN(b * alpha_g) / 6)) (b = 0 -> 0x38, 1.0).
// T1 points at this lane's copy of the mantissa table.
// For BF16 inputs b = (1 + m/128) 2^(E-127); writing alpha_g = a_m 2^ae with
// a_m in [1, 2), RN(RN(b alpha_g) / 6) = RN(RN((1 + m/128) a_m) / 6)
// 2^(E-127+ae) while the values stay normal (rounding commutes with
// power-of-two scaling), so it is a per-CTA 128-entry table plus an exponent
// shift; anything that would fall below 2^-126 encodes to E4M3 +0 either way,
// and anything at or above 2^128 saturates to 448 (0x7E) either way.
// FP32 inputs, subnormal or non-finite b, and an alpha_g that is 0 or NaN
// (a non-finite tensor amax; ae is then kNoTable) take the two operations.
constexpr int kNoTable = -100000;
template <int DT, int C = 1> QD uint32_t nv_sb_code(uint32_t b, float alpha_g, const uint32_t *T1, int ae)
{
    if (b == 0) return 0x38u;
    const uint32_t E = b >> 23;
    if (DT == BF16 && E != 0u && E != 255u && ae != kNoTable) {
        const uint32_t t = T1[((b >> 16) & 0x7Fu) * C];
        const int ne = (int)(t >> 23) + (int)E - 127 + ae;
        if (ne <= 0) return 0u;
        if (ne >= 255) return 0x7Eu;
        return e4m3_code(__uint_as_float((t & 0x807FFFFFu) | ((uint32_t)ne << 23)));
    }
    return e4m3_code(__fdiv_rn(__fmul_rn(__uint_as_float(b), alpha_g), 6.0f));
}

// The encode factor enc = alpha_g / f(sb) (0 when f(sb) = 0) depends only on
// the code: each CTA tabulates it for the 128 positive codes (entry 0x38 =
// alpha_g also serves b = 0).


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

// Codes of one row chunk (VEC elements, VEC/2 bytes) with scale factor enc;
// SR draws the Philox block of element index i0 (row-major, stream 0).
template <int DT, int RND>
QD uint32_t nv_row_codes(const uint4 &v, float enc, uint64_t seed, uint64_t offset, int64_t i0)
{
    constexpr int VEC = In<DT>::VEC;
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; j++) y[j] = j < VEC ? elem<DT>(v, j < VEC ? j : 0) : 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; j += 2) mul2(y[j], y[j + 1], enc, enc);
    if (RND == 1) {
        const uint4 R = sr_bits(seed, offset + (uint64_t)(i0 >> 3), 0u);
        const int e0 = (int)(i0 & 7);
#pragma unroll
        for (int j = 0; j < VEC; j += 2) {   // draws e0 + j, e0 + j + 1: one word (e0 is 0, or 4 for FP32 chunks)
            float r0, r1;
            r16_pair(VEC == 8 ? word(R, j >> 1) : (e0 ? word(R, 2 + (j >> 1)) : word(R, j >> 1)), r0, r1);
            y[j] = sr_e2m1_value(y[j], r0);
            y[j + 1] = sr_e2m1_value(y[j + 1], r1);
        }
    }
    return cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}

// Transposed FP4 codes of a tile: col[c] holds, for column c of this
// thread's chunk, the 8 codes of rows 8w..8w+7 (row 8w in bits 3-0).  They
// are parked at [column][64 bytes] in the consumed stage (4-byte slot w,
// XOR-swizzled by lane) and written as q_colT rows by copy_out_fp4T.
template <int VEC> QD void park_fp4T(uint8_t *stage, const uint32_t *col, int warp, int lane)
{
#pragma unroll
    for (int c = 0; c < VEC; c++)
        *reinterpret_cast<uint32_t *>(stage + (lane * VEC + c) * 64 + ((warp ^ (lane & 15)) * 4)) = col[c];
}

// With M % 32 == 0 the rows go out as 16-byte pieces (4 threads per 64-byte
// row): slots 4g..4g+3 sit in the aligned group 4g ^ (s & ~3), word k holding
// slot 4g + (k ^ (s & 3)).
template <int VEC>
QD void copy_out_fp4T(const uint8_t *stage, uint8_t *q_colT, int64_t M, int64_t K, int64_t mb, int64_t kb)
{
    constexpr int TC = 32 * VEC;
    if ((M & 31) == 0) {
#pragma unroll
        for (int it = 0; it < TC * 4 / kEngThreads; it++) {
            const int idx = it * kEngThreads + threadIdx.x;
            const int col = idx >> 2, g = idx & 3;   // rows 32g..32g+31 of the tile
            const int s = (col / VEC) & 15;
            const int64_t kg = kb + col, mg = mb + 32 * g;
            if (kg < K && mg < M) {
                uint4 w = *reinterpret_cast<const uint4 *>(stage + col * 64 + ((4 * g) ^ (s & ~3)) * 4);
                if (s & 1) w = make_uint4(w.y, w.x, w.w, w.z);
                if (s & 2) w = make_uint4(w.z, w.w, w.x, w.y);
                stg16(q_colT + kg * (M / 2) + mg / 2, w);
            }
        }
        return;
    }
#pragma unroll
    for (int it = 0; it < TC * 16 / kEngThreads; it++) {
        const int idx = it * kEngThreads + threadIdx.x;
        const int col = idx >> 4, sl = idx & 15;   // slot sl = rows 8sl..8sl+7 of the tile
        const int64_t kg = kb + col, mg = mb + 8 * sl;
        if (kg < K && mg < M)
            stg4(q_colT + kg * (M / 2) + mg / 2,
                 *reinterpret_cast<const uint32_t *>(stage + col * 64 + ((sl ^ ((col / VEC) & 15)) * 4)));
    }
}

// Columnwise block scales of a tile, sSB[g][col] for the 16-row group g of
// tile column col, written as sb_colT[kb + col][mb/16 + g].
template <int TC>
QD void copy_out_sbT(const uint8_t (*sSB)[TC], uint8_t *sb_colT, int64_t M, int64_t K, int64_t mb, int64_t kb)
{
    const int64_t left = (M - mb) / 16;
    const int nb = left < 8 ? (int)left : 8;
    for (int col = threadIdx.x; col < TC; col += kEngThreads) {
        const int64_t kg = kb + col;
        if (kg >= K) continue;
        uint8_t *dst = sb_colT + kg * (M / 16) + mb / 16;
        if (nb == 8 && (M % 128) == 0) {
            uint32_t w0 = 0, w1 = 0;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                w0 |= (uint32_t)sSB[q][col] << (8 * q);
                w1 |= (uint32_t)sSB[q + 4][col] << (8 * q);
            }
            stg8(dst, w0, w1);
        } else {
            for (int q = 0; q < nb; q++) dst[q] = sSB[q][col];
        }
    }
}

template <int DT, int BLK, int RND>
__global__ void __launch_bounds__(kEngThreads, 1) k_nvfp4(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                          const float *__restrict__ amax, uint64_t seed, uint64_t offset,
                                                          uint8_t *__restrict__ q_row, uint8_t *__restrict__ sb_row,
                                                          uint8_t *__restrict__ q_colT, uint8_t *__restrict__ sb_colT,
                                                          float *__restrict__ s_global, int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, LPB = 16 / VEC, TCP = kTabCopies<BLK>;
    __shared__ float enc_tab[128 * TCP];
    __shared__ uint32_t sb_tab[128 * TCP];   // BF16: RN(RN((1 + m/128) a_m) / 6) per mantissa m
    __shared__ uint4 part[kEngWarps][32];        // 1x16: per-warp column maxima over 8 rows
    __shared__ __align__(8) uint8_t sSB[8][TC];   // 1x16: columnwise block scales of a tile
    __shared__ uint32_t bred[kEngWarps][TC / 16];   // 16x16: half-block maxima

    griddep_wait();   // the amax pass ahead of this kernel is complete
    const float A = *amax;
    const float alpha_g = alpha_from_amax(2688.0f, A);
    const uint32_t ag = __float_as_uint(alpha_g);
    // alpha_g = 2688 / A is a normal float for every finite A > 0 (and 1 for
    // A = 0); a non-finite A gives 0 or NaN, which the table cannot scale
    const bool ag_normal = (ag >> 23) != 0u && (ag >> 23) != 255u;
    const int ae = ag_normal ? (int)(ag >> 23) - 127 : kNoTable;
    if (threadIdx.x < 128) {
        const float sv = e4m3_value(threadIdx.x);
        const float ev = sv == 0.0f ? 0.0f : __fdiv_rn(alpha_g, sv);
        const float a_m = __uint_as_float((ag & 0x807FFFFFu) | (127u << 23));
        const uint32_t tv = __float_as_uint(__fdiv_rn(__fmul_rn(1.0f + (float)threadIdx.x * (1.0f / 128.0f), a_m), 6.0f));
#pragma unroll
        for (int j = 0; j < TCP; j++) {
            enc_tab[threadIdx.x * TCP + j] = ev;
            sb_tab[threadIdx.x * TCP + j] = tv;
        }
    }   // visible after the engine's first barrier
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *s_global = __fdiv_rn(1.0f, alpha_g);
        flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
    }
    if (M == 0 || K == 0) return;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;
    const float *encT = enc_tab + (lane & (TCP - 1));   // this lane's copy: entry e at encT[e * TCP]
    const uint32_t *sbT = sb_tab + (lane & (TCP - 1));

    run_tiles(&tmap, tiles_m, tiles_k, TC, true, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        const int64_t k = kb + lane * VEC, m0 = mb + 8 * warp;
        const bool kok = k < K;
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = lds16(st + (8 * warp + j) * kRowBytes + lane * 16);
        uint32_t colw[8];   // transposed codes: column c -> 8 row nibbles

        if constexpr (BLK == 0) {
            if (q_colT != nullptr) {   // column maxima of this warp's 8 rows
                uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    acc.x = colmax_word<DT>(acc.x, v[j].x);
                    acc.y = colmax_word<DT>(acc.y, v[j].y);
                    acc.z = colmax_word<DT>(acc.z, v[j].z);
                    acc.w = colmax_word<DT>(acc.w, v[j].w);
                }
                part[warp][lane] = acc;
            }
            // ---------------- 1x16 rowwise ----------------
            uint32_t nf = 0;
            if (DT == BF16 && q_row != nullptr) {
                // A block is 2 lanes.  The 8 row maxima, two BF16 magnitudes per
                // word, are halved across the pair: this lane keeps rows
                // rb..rb+3 (rb = 4 * (lane & 1)), computes their block scales and
                // encode factors, and takes the partner's 4 factors by shuffle.
                const int nrows = !kok ? 0 : (m0 + 8 <= M ? 8 : (m0 < M ? (int)(M - m0) : 0));
                uint32_t P[4];
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const uint4 &a = v[2 * p], &b = v[2 * p + 1];
                    const uint32_t ma = hmax_abs2(hmax_abs2(a.x, a.y), hmax_abs2(a.z, a.w));
                    const uint32_t mb2 = hmax_abs2(hmax_abs2(b.x, b.y), hmax_abs2(b.z, b.w));
                    P[p] = hmax_abs2(__byte_perm(ma, mb2, 0x5410), __byte_perm(ma, mb2, 0x7632));   // row 2p low, 2p+1 high
                }
                const bool b0 = lane & 1;
                const int rb = b0 ? 4 : 0;
                uint32_t k0 = b0 ? P[2] : P[0], k1 = b0 ? P[3] : P[1];
                const uint32_t s0 = b0 ? P[0] : P[2], s1 = b0 ? P[1] : P[3];
                k0 = hmax_abs2(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, 1));
                k1 = hmax_abs2(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, 1));
                float own[4];
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    const uint32_t kw = h < 2 ? k0 : k1;
                    const uint32_t bits = ((h & 1) ? kw : (kw << 16)) & 0x7FFF0000u;   // row rb + h
                    const uint32_t sb = nv_sb_code<DT, TCP>(bits, alpha_g, sbT, ae);
                    own[h] = encT[(sb & 0x7Fu) * TCP];
                    if (rb + h < nrows) {
                        sb_row[(m0 + rb + h) * (K / 16) + k / 16] = (uint8_t)sb;
                        nf |= nonfinite(bits);
                    }
                }
                float encr[8];
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    const float other = __shfl_xor_sync(0xFFFFFFFFu, own[h], 1);
                    encr[h] = b0 ? other : own[h];
                    encr[4 + h] = b0 ? own[h] : other;
                }
                uint8_t *qr = q_row + m0 * (K / 2) + k / 2;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const uint32_t code = nv_row_codes<DT, RND>(v[j], encr[j], seed, offset, (m0 + j) * K + k);
                    if (j < nrows) stg4(qr + j * (K / 2), code);
                }
            } else if (q_row != nullptr) {
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    uint32_t bb[2] = {absmax_bits<DT>(v[j]), absmax_bits<DT>(v[j + 1])};
                    group_max2<DT, LPB>(bb[0], bb[1]);
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int64_t m = m0 + j + h;
                        const uint32_t sb = nv_sb_code<DT, TCP>(bb[h], alpha_g, sbT, ae);
                        const uint32_t code = nv_row_codes<DT, RND>(v[j + h], encT[(sb & 0x7Fu) * TCP], seed, offset, m * K + k);
                        const bool ok = m < M && kok;
                        if (ok) {
                            uint8_t *dst = q_row + m * (K / 2) + k / 2;
                            if (VEC == 8) stg4(dst, code);
                            else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)code;
                        }
                        if (ok && lane % LPB == 0) sb_row[m * (K / 16) + k / 16] = (uint8_t)sb;
                        nf |= ok ? nonfinite(bb[h]) : 0u;
                    }
                }
            }
            post_nonfinite(status, nf);
            if (q_colT == nullptr) return;
            __syncthreads();   // partial maxima posted; every read of the stage is done
            // ---------------- 16x1 columnwise: warps 2p, 2p+1 share a block ----------------
            uint4 cm = part[warp][lane];
            {
                const uint4 o4 = part[warp ^ 1][lane];
                cm.x = colmax_word<DT>(cm.x, o4.x);
                cm.y = colmax_word<DT>(cm.y, o4.y);
                cm.z = colmax_word<DT>(cm.z, o4.z);
                cm.w = colmax_word<DT>(cm.w, o4.w);
            }
            // each column's block scale, then its 8 rows with the block's factor:
            // one E2M1 word per column (row 8w in bits 3-0)
            uint32_t nfc = 0;
            // RTNE: this thread's VEC column scale codes, stored together below
            // (with SR the register they take costs more than the byte stores)
            uint32_t sbw[VEC / 4] = {};
#pragma unroll
            for (int c = 0; c < VEC; c++) {
                const uint32_t b = colmax_bits<DT>(cm, c);
                const uint32_t sb = nv_sb_code<DT, TCP>(b, alpha_g, sbT, ae);
                const float enc = encT[(sb & 0x7Fu) * TCP];
                if (RND == 0) sbw[c >> 2] |= sb << (8 * (c & 3));
                else if ((warp & 1) == 0) sSB[warp >> 1][lane * VEC + c] = (uint8_t)sb;
                nfc |= ((warp & 1) == 0 && kok && m0 < M) ? nonfinite(b) : 0u;
                float y[8];
#pragma unroll
                for (int j = 0; j < 8; j++) y[j] = elem<DT>(v[j], c);
#pragma unroll
                for (int j = 0; j < 8; j += 2) mul2(y[j], y[j + 1], enc, enc);
                if (RND == 1) {
                    // rows m0 .. m0 + 7 of column k + c, stream 1: Philox block (m0 / 8) * K + k + c
                    const uint4 R = sr_bits(seed, offset + (uint64_t)((m0 >> 3) * K + k + c), 1u);
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        float r0, r1;
                        r16_pair(word(R, j >> 1), r0, r1);
                        y[j] = sr_e2m1_value(y[j], r0);
                        y[j + 1] = sr_e2m1_value(y[j + 1], r1);
                    }
                }
                colw[c] = cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
            }
            if (RND == 0 && (warp & 1) == 0) {   // one store of VEC codes (bytes lane*VEC .. +VEC-1)
                if constexpr (VEC == 8) *reinterpret_cast<uint2 *>(&sSB[warp >> 1][lane * VEC]) = make_uint2(sbw[0], sbw[1]);
                else *reinterpret_cast<uint32_t *>(&sSB[warp >> 1][lane * VEC]) = sbw[0];
            }
            post_nonfinite(status, nfc);
        } else {
            // ---------------- 16x16: one scale per tile ----------------
            uint32_t b = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) b = max(b, absmax_bits<DT>(v[j]));
            b = group_max<LPB>(b);
            if (lane % LPB == 0) bred[warp][lane / LPB] = b;
            __syncthreads();   // half-block maxima posted; every read of the stage is done
            b = max(bred[warp & ~1][lane / LPB], bred[warp | 1][lane / LPB]);
            const uint32_t sb = nv_sb_code<DT, TCP>(b, alpha_g, sbT, ae);
            const float enc = encT[(sb & 0x7Fu) * TCP];
            const int64_t m16 = mb + 16 * (warp >> 1);
            if ((warp & 1) == 0 && lane % LPB == 0 && m16 < M && kok) {
                if (sb_row != nullptr) sb_row[(m16 / 16) * (K / 16) + k / 16] = (uint8_t)sb;
                if (sb_colT != nullptr) sb_colT[(k / 16) * (M / 16) + m16 / 16] = (uint8_t)sb;
                flag_nonfinite(status, b);
            }
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int64_t m = m0 + j;
                const uint32_t code = nv_row_codes<DT, RND>(v[j], enc, seed, offset, m * K + k);
                if (q_row != nullptr && m < M && kok) {
                    uint8_t *dst = q_row + m * (K / 2) + k / 2;
                    if (VEC == 8) stg4(dst, code);
                    else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)code;
                }
                colw[j] = code;
            }
            if (q_colT == nullptr) return;
            transpose8x8_nibbles(colw);
        }
        // ---- transposed codes: parked in the consumed stage, then q_colT rows
        park_fp4T<VEC>(st, colw, warp, lane);
        __syncthreads();
        copy_out_fp4T<VEC>(st, q_colT, M, K, mb, kb);
        if constexpr (BLK == 0) copy_out_sbT<TC>(sSB, sb_colT, M, K, mb, kb);
    });
}

template <int DT, int BLK, int RND>
static cudaError_t nv_t(const void *x, int64_t M, int64_t K, const float *amax, uint64_t seed, uint64_t offset,
                        uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT, float *s_global,
                        int32_t *status, cudaStream_t st, bool after_amax)
{
    constexpr int TC = 32 * In<DT>::VEC;
    alignas(64) CUtensorMap map;
    const bool empty = M == 0 || K == 0;
    if (!empty) {
        cudaError_t e = make_tile_map(&map, x, DT, M, K);
        if (e != cudaSuccess) return e;
    } else {
        memset(&map, 0, sizeof map);   // never dereferenced: the kernel returns before touching tiles
    }
    {
        const cudaError_t ea = engine_smem_ready<k_nvfp4<DT, BLK, RND>>();
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kTileRowsE - 1) / kTileRowsE) * ((K + TC - 1) / TC);
    int grid = (int)(tiles < sm_count() ? tiles : sm_count());
    if (grid < 1) grid = 1;   // an empty tensor still gets its global scale
    return launch_k(after_amax, k_nvfp4<DT, BLK, RND>, dim3(grid), dim3(kEngThreads), kEngSmem, st, map, M, K, amax,
                    seed, offset, q_row, sb_row, q_colT, sb_colT, s_global, status);
}

cudaError_t launch_nvfp4(const void *x, int dt, int64_t M, int64_t K, int blk, int rnd, uint64_t seed,
                         uint64_t offset, const float *amax, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT,
                         uint8_t *sb_colT, float *s_global, int32_t *status, cudaStream_t st, bool after_amax)
{
#define NV_ARGS x, M, K, amax, seed, offset, q_row, sb_row, q_colT, sb_colT, s_global, status, st, after_amax
    if (dt == BF16) {
        if (blk == 0) return rnd == 0 ? nv_t<BF16, 0, 0>(NV_ARGS) : nv_t<BF16, 0, 1>(NV_ARGS);
        return rnd == 0 ? nv_t<BF16, 1, 0>(NV_ARGS) : nv_t<BF16, 1, 1>(NV_ARGS);
    }
    if (blk == 0) return rnd == 0 ? nv_t<F32, 0, 0>(NV_ARGS) : nv_t<F32, 0, 1>(NV_ARGS);
    return rnd == 0 ? nv_t<F32, 1, 0>(NV_ARGS) : nv_t<F32, 1, 1>(NV_ARGS);
#undef NV_ARGS
}

// ---------------------------------------------------------------------------
// Random Hadamard transform + columnwise NVFP4 of the result ("From BF16 to
// FP8/FP4 ...", sections 2.4 and 5.6: RHT on the weight-gradient GEMM
// inputs, to spread block-level outliers before FP4 quantization).
// x' = (1/4) H D x on every 16-row group of every column (H the 16-point
// Sylvester Hadamard matrix, D the signs of a 16-bit mask): signs, then the
// butterfly with strides 1, 2, 4, 8 in FP32, then the exact factor 1/4.
// The 16x1 blocks of the columnwise copy are exactly these groups.
// Thread t of a tile owns group g = t / 64 and 8 bytes of each of its 16
// rows (CPT = 4 BF16 or 2 FP32 columns), so a block never leaves its thread;
// column pairs go through the butterfly as packed FP32x2 operations.
// PASS 0 reduces max|x'| (the tensor amax of the transformed copy) into
// *amax; PASS 1 encodes with the tensor scale from *amax, parks the codes in
// the consumed stage and writes q_colT rows (as k_nvfp4 does).
// ---------------------------------------------------------------------------
template <int DT, int RND, int PASS>
__global__ void __launch_bounds__(kEngThreads, 1) k_nvfp4_rht(const __grid_constant__ CUtensorMap tmap, int64_t M,
                                                              int64_t K, uint32_t sign_mask, float *amax, uint64_t seed,
                                                              uint64_t offset, uint8_t *__restrict__ q_colT,
                                                              uint8_t *__restrict__ sb_colT, float *__restrict__ s_global,
                                                              int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, CPT = VEC / 2;
    // PASS 0 writes no tensor scale: its s_global slot carries the optional
    // max|x| output (the untransformed tensor's amax, in the same read)
    float *const amax_x = PASS == 0 ? s_global : nullptr;
    __shared__ float enc_tab[128];
    __shared__ uint8_t sSB[8][TC];
    float alpha_g = 1.0f;
    if (PASS == 0) griddep_launch_dependents();   // the encode pass may be scheduled; it waits for the amax
    if (PASS == 1) {
        griddep_wait();   // the amax pass ahead of this one is complete
        const float A = *amax;
        alpha_g = alpha_from_amax(2688.0f, A);
        if (threadIdx.x < 128) {
            const float sv = e4m3_value(threadIdx.x);
            enc_tab[threadIdx.x] = sv == 0.0f ? 0.0f : __fdiv_rn(alpha_g, sv);
        }   // visible after the engine's first barrier
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            *s_global = __fdiv_rn(1.0f, alpha_g);
            flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
        }
    }
    if (M == 0 || K == 0) return;
    const int g = threadIdx.x >> 6, q = threadIdx.x & 63;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;
    uint32_t mx = 0;   // PASS 0: max |x'| bits of this thread (zero-filled rows and columns give 0)
    uint32_t mxx = 0;  // PASS 0 with amax_x: max |x| of this thread (the untransformed tensor), as k_amax takes
                       // it: BF16 packed two per word, FP32 as a float

    run_tiles(&tmap, tiles_m, tiles_k, TC, PASS == 1, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        uint2 raw[16];
#pragma unroll
        for (int r = 0; r < 16; r++) raw[r] = *reinterpret_cast<const uint2 *>(st + (16 * g + r) * kRowBytes + q * 8);
        if (PASS == 0 && amax_x != nullptr) {
#pragma unroll
            for (int r = 0; r < 16; r++) {
                if (DT == BF16)
                    mxx = hmax_abs2(mxx, hmax_abs2(raw[r].x, raw[r].y));
                else
                    mxx = __float_as_uint(fmax_abs(fmax_abs(__uint_as_float(mxx), __uint_as_float(raw[r].x)),
                                                   __uint_as_float(raw[r].y)));
            }
        }
        uint32_t code[CPT][2];   // per column: rows 16g..16g+7 and 16g+8..16g+15, first row in bits 3-0
#pragma unroll
        for (int p = 0; p < CPT / 2; p++) {   // column pair (2p, 2p+1) of the thread's CPT columns
            float a[16], b[16];
#pragma unroll
            for (int r = 0; r < 16; r++) {
                const uint32_t neg = ((sign_mask >> r) & 1u) << 31;
                if (DT == BF16) {
                    const uint32_t w = p == 0 ? raw[r].x : raw[r].y;
                    a[r] = __uint_as_float((w << 16) ^ neg);
                    b[r] = __uint_as_float((w & 0xFFFF0000u) ^ neg);
                } else {
                    a[r] = __uint_as_float(raw[r].x ^ neg);
                    b[r] = __uint_as_float(raw[r].y ^ neg);
                }
            }
#pragma unroll
            for (int h = 1; h < 16; h *= 2)
#pragma unroll
                for (int i = 0; i < 16; i++)
                    if ((i & h) == 0) bfly2(a[i], b[i], a[i + h], b[i + h]);
#pragma unroll
            for (int i = 0; i < 16; i++) mul2(a[i], b[i], 0.25f, 0.25f);
            if (PASS == 0) {
#pragma unroll
                for (int i = 0; i < 16; i++) mx = max(mx, __float_as_uint(fmax_abs(a[i], b[i])) & 0x7FFFFFFFu);
                continue;
            }
            // block scales and encode factors of the two columns
            float ma = 0.0f, mbx = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                ma = fmax_abs(ma, a[i]);
                mbx = fmax_abs(mbx, b[i]);
            }
            const uint32_t ba = __float_as_uint(ma) & 0x7FFFFFFFu, bb = __float_as_uint(mbx) & 0x7FFFFFFFu;
            const uint32_t sa = nv_sb_code<F32>(ba, alpha_g, nullptr, 0), sbb = nv_sb_code<F32>(bb, alpha_g, nullptr, 0);
            const float ea = enc_tab[sa & 0x7Fu], eb = enc_tab[sbb & 0x7Fu];
            const int c0 = q * CPT + 2 * p;   // tile column of a
            sSB[g][c0] = (uint8_t)sa;
            sSB[g][c0 + 1] = (uint8_t)sbb;
            const bool live = mb + 16 * g < M;
            post_nonfinite(status, live && (kb + c0 < K) ? nonfinite(ba) | nonfinite(bb) : 0u);
#pragma unroll
            for (int i = 0; i < 16; i++) mul2(a[i], b[i], ea, eb);
            if constexpr (RND == 1) {
                // rows m .. m + 15 of columns kb + c0, kb + c0 + 1, stream 1: Philox blocks
                // (m / 8 + hh) * K + column, two per column
                const int64_t m = mb + 16 * g;
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    const uint64_t gb = offset + (uint64_t)(((m >> 3) + hh) * K + kb + c0);
                    const uint4 Ra = sr_bits(seed, gb, 1u);
                    const uint4 Rb = sr_bits(seed, gb + 1, 1u);
                    float ra[8], rb[8];
                    r16_block(Ra, ra);
                    r16_block(Rb, rb);
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        a[8 * hh + j] = sr_e2m1_value(a[8 * hh + j], ra[j]);
                        b[8 * hh + j] = sr_e2m1_value(b[8 * hh + j], rb[j]);
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                code[2 * p][hh] = cvt_fp4x8(a[8 * hh], a[8 * hh + 1], a[8 * hh + 2], a[8 * hh + 3], a[8 * hh + 4],
                                            a[8 * hh + 5], a[8 * hh + 6], a[8 * hh + 7]);
                code[2 * p + 1][hh] = cvt_fp4x8(b[8 * hh], b[8 * hh + 1], b[8 * hh + 2], b[8 * hh + 3], b[8 * hh + 4],
                                                b[8 * hh + 5], b[8 * hh + 6], b[8 * hh + 7]);
            }
        }
        if (PASS == 0) return;
        __syncthreads();   // every read of the stage is done: park the codes in it
#pragma unroll
        for (int c = 0; c < CPT; c++) {
            const int col = q * CPT + c;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const int sl = 2 * g + hh;   // 8-row slot, as copy_out_fp4T reads it
                *reinterpret_cast<uint32_t *>(st + col * 64 + ((sl ^ ((col / VEC) & 15)) * 4)) = code[c][hh];
            }
        }
        __syncthreads();
        copy_out_fp4T<VEC>(st, q_colT, M, K, mb, kb);
        copy_out_sbT<TC>(sSB, sb_colT, M, K, mb, kb);
    });
    if (PASS == 0) {
        griddep_wait();   // the zeroing of the amax words ahead of this pass is complete
        cta_max_to(mx, reinterpret_cast<uint32_t *>(amax), status);
        if (amax_x != nullptr) {
            if (DT == BF16) mxx = (hmax_abs2(mxx, __byte_perm(mxx, 0u, 0x1032)) << 16) & 0x7FFF0000u;
            else mxx &= 0x7FFFFFFFu;
            __syncthreads();   // the CTA reduction's shared words are free again
            cta_max_to(mxx, reinterpret_cast<uint32_t *>(amax_x), status);
        }
    }
}

template <int DT, int RND, int PASS>
static cudaError_t rht_pass(bool pdl, const CUtensorMap &map, int64_t M, int64_t K, uint32_t mask, float *amax,
                            float *amax_x, uint64_t seed, uint64_t offset, uint8_t *q_colT, uint8_t *sb_colT,
                            float *s_global, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    {
        const cudaError_t ea = engine_smem_ready<k_nvfp4_rht<DT, RND, PASS>>();
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kTileRowsE - 1) / kTileRowsE) * ((K + TC - 1) / TC);
    int grid = (int)(tiles < sm_count() ? tiles : sm_count());
    if (grid < 1) grid = 1;   // an empty tensor still gets its global scale
    return launch_k(pdl, k_nvfp4_rht<DT, RND, PASS>, dim3(grid), dim3(kEngThreads), kEngSmem, st, map, M, K, mask, amax,
                    seed, offset, q_colT, sb_colT, PASS == 0 ? amax_x : s_global, status);
}

template <int DT, int RND>
static cudaError_t rht_t(const void *x, int64_t M, int64_t K, uint32_t mask, bool compute_amax, float *amax,
                         uint64_t seed, uint64_t offset, uint8_t *q_colT, uint8_t *sb_colT, float *s_global,
                         int32_t *status, cudaStream_t st)
{
    alignas(64) CUtensorMap map;
    const bool empty = M == 0 || K == 0;
    if (!empty) {
        cudaError_t e = make_tile_map(&map, x, DT, M, K);
        if (e != cudaSuccess) return e;
    } else {
        memset(&map, 0, sizeof map);   // never dereferenced: the kernels return before touching tiles
    }
    if (compute_amax) {
        cudaError_t e = launch_zero_word(amax, st);
        if (e != cudaSuccess) return e;
        e = rht_pass<DT, 0, 0>(true, map, M, K, mask, amax, nullptr, seed, offset, q_colT, sb_colT, s_global, status,
                               st);   // no rounding in the amax pass
        if (e != cudaSuccess) return e;
    }
    return rht_pass<DT, RND, 1>(compute_amax, map, M, K, mask, amax, nullptr, seed, offset, q_colT, sb_colT, s_global,
                                status, st);
}

cudaError_t launch_rht_amax(const void *x, int dt, int64_t M, int64_t K, uint32_t sign_mask, float *amax,
                            float *amax_x, int32_t *status, cudaStream_t st)
{
    alignas(64) CUtensorMap map;
    if (M == 0 || K == 0) return launch_zero_word(amax, st, amax_x);
    cudaError_t e = make_tile_map(&map, x, dt, M, K);
    if (e == cudaSuccess) e = launch_zero_word(amax, st, amax_x);
    if (e != cudaSuccess) return e;
    return dt == BF16 ? rht_pass<BF16, 0, 0>(true, map, M, K, sign_mask, amax, amax_x, 0, 0, nullptr, nullptr, nullptr,
                                            status, st)
                      : rht_pass<F32, 0, 0>(true, map, M, K, sign_mask, amax, amax_x, 0, 0, nullptr, nullptr, nullptr,
                                           status, st);
}

cudaError_t launch_nvfp4_rht_colT(const void *x, int dt, int64_t M, int64_t K, uint32_t sign_mask, int rnd,
                                  uint64_t seed, uint64_t offset, bool compute_amax, float *amax, uint8_t *q_colT,
                                  uint8_t *sb_colT, float *s_global, int32_t *status, cudaStream_t st)
{
#define RHT_ARGS x, M, K, sign_mask, compute_amax, amax, seed, offset, q_colT, sb_colT, s_global, status, st
    if (dt == BF16) return rnd == 0 ? rht_t<BF16, 0>(RHT_ARGS) : rht_t<BF16, 1>(RHT_ARGS);
    return rnd == 0 ? rht_t<F32, 0>(RHT_ARGS) : rht_t<F32, 1>(RHT_ARGS);
#undef RHT_ARGS
}

}  // namespace qk
