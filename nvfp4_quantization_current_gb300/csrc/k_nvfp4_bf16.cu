// NVFP4 quantize of BF16 tensors (a8-a11), 1x16 and 16x16 blocks, RTNE or
// stochastic rounding, on the tile engine.  This is q_nvfp4's path for BF16
// inputs; FP32 inputs take k_nvfp4 (k_nvfp4.cu).  The arithmetic is the same:
// "Mixed-precision training: fp16 to fp8", sections "NVFP4" and recipe 6,
// and "From BF16 to FP8/FP4 ...", section 2.4 (1x16 blocks for activations
// and gradients, 16x16 for weights, stochastic rounding on gradients):
//   alpha_g = 2688 / amax, s_g = 1 / alpha_g;
//   per block sb = E4M3(RN(RN(b * alpha_g) / 6)) (b = 0 -> 1.0),
//   enc = alpha_g / sb (0 if sb is 0), q = E2M1(x * enc).
//
// Two CTAs of 256 threads per SM, each with its own three 64 x 256 stages
// (32 KiB of BF16 each; TileCfg<64, 256>): one CTA's barriers and
// latency-bound phases overlap the other's work, which one 512-thread CTA
// with 128-row tiles could not (its 16 warps move through the same phases
// together).
// Thread layout.  The 8 warps of a CTA cover a 64 x 256 tile: warp w takes
// rows 16 (w / 2) .. + 15 and columns 128 (w % 2) .. + 127 of the tile; lane
// l takes 8 of those rows (8 (l / 16) .. + 7) of one 16-byte column chunk
// (columns 8 (l % 16) .. + 7).  Hence
//   a 1x16 row block    is the lane pair l, l ^ 1,
//   a 16x1 column block is the lane pair l, l ^ 16,
//   a 16x16 block       is the lanes l, l ^ 1, l ^ 16, l ^ 17:
// block maxima and block factors move by warp shuffles, and each block's
// scale is computed once (the two lanes of a pair split the pair's rows or
// columns between them and swap the factors).
// Row codes leave from registers (4 bytes per row and thread).  The
// columnwise codes of a thread (one word of 8 row nibbles per column) are
// parked in a buffer of their own behind the stages and leave as 16-byte
// pieces of q_colT rows, the column block scales through shared memory as
// 4-byte pieces of sb_colT rows.
//
// Stochastic rounding: Philox4x32-10 with round keys formed on the host;
// the rowwise copy draws one Philox block per row and thread (8 consecutive
// columns, stream 0), the columnwise copy one per column and thread (8
// consecutive rows, stream 1); each element is rounded with
// sr_e2m1_dither.
#include <cstring>

#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

using NvCfg = TileCfg<64, 256, 3>;
constexpr int kNvRows = NvCfg::kRows, kNvThreads = NvCfg::kThreads;
constexpr int kNvTabCopies = 4;                          // interleaved copies of each per-CTA table
constexpr int kNvParkBytes = 256 * (kNvRows / 2);        // parked columnwise codes of a tile: [256 columns][rows / 2]
constexpr int kNvSmem = NvCfg::kSmem + kNvParkBytes;     // dynamic shared memory of a CTA

// Block scale code of a block with maximum b (FP32 bits of a BF16 value):
// sb = E4M3(RN(RN(b * alpha_g) / 6)), b = 0 -> 0x38.
// nvb_sb_exact takes the two operations.  nvb_sb_fast, for a normal b and a
// normal alpha_g = a_m 2^ae (a_m in [1, 2)), writes b = (1 + m/128) 2^(E-127):
// the rounded quotient is RN(RN((1 + m/128) a_m) / 6) 2^(E-127+ae) while it
// stays a normal float (rounding commutes with power-of-two scaling), i.e. a
// per-CTA table over the 128 mantissas (T: this lane's copy) plus an exponent
// shift.  A quotient below 2^-126 encodes to E4M3 +0 either way and one at or
// above 2^128 saturates to 448 (0x7E) either way, so the exponent is clamped
// to [0, 254] instead of branching.  aem = ae - 127.
// nvb_sb_rare: b needs the two operations (a subnormal, inf or NaN maximum).
QD uint32_t nvb_sb_exact(uint32_t b, float alpha_g)
{
    return b == 0 ? 0x38u : e4m3_code(__fdiv_rn(__fmul_rn(__uint_as_float(b), alpha_g), 6.0f));
}
QD uint32_t nvb_sb_fast(uint32_t b, const uint32_t *T, int aem)
{
    const uint32_t t = T[((b >> 16) & 0x7Fu) * kNvTabCopies];
    int ne = (int)(t >> 23) + (int)(b >> 23) + aem;
    ne = min(max(ne, 0), 254);
    const uint32_t code = e4m3_code(__uint_as_float((t & 0x807FFFFFu) | ((uint32_t)ne << 23)));
    return b == 0 ? 0x38u : code;
}
QD bool nvb_sb_rare(uint32_t b) { return b != 0 && ((b >> 23) - 1u) >= 254u; }

// Block scale codes of N blocks with maxima b[]: the table path, and, when
// any lane of the warp holds a rare maximum or the CTA has no table (a
// non-finite amax), the two operations for those (one warp-uniform branch).
template <int N>
QD void nvb_sb_codes(const uint32_t (&b)[N], uint32_t (&sb)[N], float alpha_g, const uint32_t *T, int aem, bool tab)
{
    bool rare = !tab;
#pragma unroll
    for (int h = 0; h < N; h++) {
        sb[h] = nvb_sb_fast(b[h], T, aem);
        rare |= nvb_sb_rare(b[h]);
    }
    if (__any_sync(0xFFFFFFFFu, rare)) {
#pragma unroll
        for (int h = 0; h < N; h++)
            if (!tab || nvb_sb_rare(b[h])) sb[h] = nvb_sb_exact(b[h], alpha_g);
    }
}

// E2M1 codes of 8 values (y[0] in bits 3-0) after the products y *= enc;
// with stochastic rounding each element takes the dither of its 16 bits of
// the Philox block R (element j: word j / 2, low half for even j).
template <int RND> QD uint32_t nvb_codes8(float (&y)[8], float enc, const uint4 &R, uint32_t dm)
{
#pragma unroll
    for (int j = 0; j < 8; j += 2) mul2(y[j], y[j + 1], enc, enc);
    if (RND == 1) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const uint32_t w = word(R, j >> 1);
            y[j] = sr_e2m1_dither(y[j], sr_dither_lo(w, dm));
            y[j + 1] = sr_e2m1_dither(y[j + 1], sr_dither_hi(w, dm));
        }
    }
    return cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}

// The 8 BF16 values of a 16-byte chunk as FP32.
QD void bf16x8_to_f32(const uint4 &v, float (&y)[8])
{
#pragma unroll
    for (int j = 0; j < 8; j++) y[j] = elem<BF16>(v, j);
}

template <int BLK, int RND>
__global__ void __launch_bounds__(kNvThreads, 2)
    k_nvfp4_bf16(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K, const float *__restrict__ amax,
                 const __grid_constant__ PhiloxKeys keys, uint64_t offset, uint8_t *__restrict__ q_row,
                 uint8_t *__restrict__ sb_row, uint8_t *__restrict__ q_colT, uint8_t *__restrict__ sb_colT,
                 float *__restrict__ s_global, int32_t *status)
{
    constexpr int TC = 256;   // tile columns
    __shared__ float enc_tab[128 * kNvTabCopies];      // alpha_g / f(code), entry e copy j at e * copies + j
    __shared__ uint32_t sb_tab[128 * kNvTabCopies];    // RN(RN((1 + m/128) a_m) / 6) per mantissa m
    __shared__ __align__(8) uint8_t sSB[kNvRows / 16][TC];   // 1x16: column block scales [16-row group][tile column]
    extern __shared__ __align__(1024) uint8_t dsm[];
    uint8_t *const park = dsm + NvCfg::kSmem;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int wr = warp >> 1, wc = warp & 1, rp = lane >> 4, cc = lane & 15;
    const int tr = 16 * wr + 8 * rp;      // the thread's first row in a tile
    const int tcol = 128 * wc + 8 * cc;   // its first column in a tile
    const float *encT = enc_tab + (lane & (kNvTabCopies - 1));
    const uint32_t *sbT = sb_tab + (lane & (kNvTabCopies - 1));
    const int64_t tiles_m = (M + kNvRows - 1) / kNvRows, tiles_k = (K + TC - 1) / TC;
    float alpha_g = 1.0f;
    int aem = 0;        // exponent of alpha_g minus 127, for the mantissa table
    bool tab = true;    // alpha_g is a normal float, so the mantissa table applies

    // after the first tiles are requested: the tensor scale from the amax of
    // the pass ahead of this kernel, and the per-CTA tables
    auto pre = [&] {
        griddep_wait();
        const float A = *amax;
        alpha_g = alpha_from_amax(2688.0f, A);
        const uint32_t ag = __float_as_uint(alpha_g);
        // alpha_g is a normal float for every finite amax (1 for amax 0); a
        // non-finite amax gives 0 or NaN, which the mantissa table cannot scale
        tab = (ag >> 23) != 0u && (ag >> 23) != 255u;
        aem = (int)(ag >> 23) - 254;
        if (t < 128) {
            const float sv = e4m3_value(t);
            const float ev = sv == 0.0f ? 0.0f : __fdiv_rn(alpha_g, sv);
            const float a_m = __uint_as_float((ag & 0x807FFFFFu) | (127u << 23));
            const uint32_t tv = __float_as_uint(__fdiv_rn(__fmul_rn(1.0f + (float)t * (1.0f / 128.0f), a_m), 6.0f));
#pragma unroll
            for (int j = 0; j < kNvTabCopies; j++) {
                enc_tab[t * kNvTabCopies + j] = ev;
                sb_tab[t * kNvTabCopies + j] = tv;
            }
        }
        if (blockIdx.x == 0 && t == 0) {
            *s_global = __fdiv_rn(1.0f, alpha_g);
            flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
        }
        __syncthreads();   // tables visible to every thread
    };

    auto body = [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kNvRows, kb = tk * TC;
        const int64_t m0 = mb + tr, k = kb + tcol;
        // M and K are multiples of 16: a thread's 8 rows and 8 columns are all
        // inside the tensor or all outside
        const bool live = m0 < M && k < K;
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = lds16(st + (tr + j) * kRowBytes + 2 * tcol);
        uint32_t colw[8];   // columnwise codes: column c -> its 8 rows' nibbles, row tr in bits 3-0
        uint32_t nf = 0;    // a non-finite block maximum seen by this thread

        if constexpr (BLK == 0) {
            // ---------------- 1x16 rowwise ----------------
            if (q_row != nullptr) {
                // row maxima, two rows per word: P[p] = (row 2p, row 2p + 1)
                uint32_t P[4];
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const uint4 &a = v[2 * p], &b = v[2 * p + 1];
                    const uint32_t ma = hmax_abs2(hmax_abs2(a.x, a.y), hmax_abs2(a.z, a.w));
                    const uint32_t mb2 = hmax_abs2(hmax_abs2(b.x, b.y), hmax_abs2(b.z, b.w));
                    P[p] = hmax_abs2(__byte_perm(ma, mb2, 0x5410), __byte_perm(ma, mb2, 0x7632));
                }
                // the pair's lane with cc even takes the block maxima of rows 0-3,
                // its partner those of rows 4-7
                const bool odd = cc & 1;
                const int rb = odd ? 4 : 0;
                uint32_t k0 = odd ? P[2] : P[0], k1 = odd ? P[3] : P[1];
                const uint32_t s0 = odd ? P[0] : P[2], s1 = odd ? P[1] : P[3];
                k0 = hmax_abs2(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, 1));
                k1 = hmax_abs2(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, 1));
                uint32_t bits[4], sb[4];
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    const uint32_t kw = h < 2 ? k0 : k1;
                    bits[h] = ((h & 1) ? kw : (kw << 16)) & 0x7FFF0000u;
                }
                nvb_sb_codes<4>(bits, sb, alpha_g, sbT, aem, tab);
                float own[4];
                uint8_t *sbr = sb_row + (m0 + rb) * (K / 16) + (k >> 4);
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    own[h] = encT[(sb[h] & 0x7Fu) * kNvTabCopies];
                    if (live) {
                        sbr[h * (K / 16)] = (uint8_t)sb[h];
                        nf |= nonfinite(bits[h]);
                    }
                }
                float encr[8];
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    const float other = __shfl_xor_sync(0xFFFFFFFFu, own[h], 1);
                    encr[h] = odd ? other : own[h];
                    encr[4 + h] = odd ? own[h] : other;
                }
                uint8_t *qr = q_row + m0 * (K / 2) + (k >> 1);
                const uint64_t g0 = offset + (uint64_t)((m0 * K + k) >> 3);   // row m0's Philox block
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    float y[8];
                    bf16x8_to_f32(v[j], y);
                    uint4 R = make_uint4(0u, 0u, 0u, 0u);
                    if (RND == 1) R = sr_bits_rk<0>(g0 + (uint64_t)j * (uint64_t)(K >> 3), keys);
                    const uint32_t code = nvb_codes8<RND>(y, encr[j], R, RND == 1 ? sr_dither_mask(encr[j]) : 0u);
                    if (live) stg4(qr + j * (K / 2), code);
                }
            }
            if (q_colT != nullptr) {
                // ---------------- 16x1 columnwise ----------------
                // the chunk again from the stage (it stays valid for the whole tile:
                // the codes are parked elsewhere), so the row pass did not have to
                // keep it in registers
                if (q_row != nullptr) {
#pragma unroll
                    for (int j = 0; j < 8; j++) v[j] = lds16_again(st + (tr + j) * kRowBytes + 2 * tcol);
                }
                // column maxima of the 8 rows (two columns per word), then of the pair's 16
                uint4 acc = v[0];
#pragma unroll
                for (int j = 1; j < 8; j++) {
                    acc.x = hmax_abs2(acc.x, v[j].x);
                    acc.y = hmax_abs2(acc.y, v[j].y);
                    acc.z = hmax_abs2(acc.z, v[j].z);
                    acc.w = hmax_abs2(acc.w, v[j].w);
                }
                acc.x = hmax_abs2(acc.x, __shfl_xor_sync(0xFFFFFFFFu, acc.x, 16));
                acc.y = hmax_abs2(acc.y, __shfl_xor_sync(0xFFFFFFFFu, acc.y, 16));
                acc.z = hmax_abs2(acc.z, __shfl_xor_sync(0xFFFFFFFFu, acc.z, 16));
                acc.w = hmax_abs2(acc.w, __shfl_xor_sync(0xFFFFFFFFu, acc.w, 16));
                // the lane of the upper 8 rows takes columns 4-7, its partner columns 0-3
                const uint32_t wA = rp ? acc.z : acc.x, wB = rp ? acc.w : acc.y;
                uint32_t bits[4], sb[4];
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    const uint32_t w = h < 2 ? wA : wB;
                    bits[h] = ((h & 1) ? w : (w << 16)) & 0x7FFF0000u;
                }
                nvb_sb_codes<4>(bits, sb, alpha_g, sbT, aem, tab);
                float ownc[4];
                uint32_t sbw = 0;
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    ownc[h] = encT[(sb[h] & 0x7Fu) * kNvTabCopies];
                    sbw |= sb[h] << (8 * h);
                    nf |= live ? nonfinite(bits[h]) : 0u;
                }
                *reinterpret_cast<uint32_t *>(&sSB[wr][tcol + 4 * rp]) = sbw;
                float encc[8];
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    const float other = __shfl_xor_sync(0xFFFFFFFFu, ownc[h], 16);
                    encc[h] = rp ? other : ownc[h];
                    encc[4 + h] = rp ? ownc[h] : other;
                }
                // column (k + c) rows m0 .. m0 + 7 draw Philox block (m0 / 8) * K + k + c of stream 1
                const uint64_t gc = offset + (uint64_t)((m0 >> 3) * K + k);
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    float y[8];
#pragma unroll
                    for (int j = 0; j < 8; j++) y[j] = elem<BF16>(v[j], c);
                    uint4 R = make_uint4(0u, 0u, 0u, 0u);
                    if (RND == 1) R = sr_bits_rk<1>(gc + (uint64_t)c, keys);
                    colw[c] = nvb_codes8<RND>(y, encc[c], R, RND == 1 ? sr_dither_mask(encc[c]) : 0u);
                }
            }
        } else {
            // ---------------- 16x16: one scale per block of four lanes ----------------
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) m = hmax_abs2(m, hmax_abs2(hmax_abs2(v[j].x, v[j].y), hmax_abs2(v[j].z, v[j].w)));
            m = hmax_abs2(m, __byte_perm(m, 0u, 0x1032));
            uint32_t bb[1] = {(m << 16) & 0x7FFF0000u}, sbb[1];
            bb[0] = max(bb[0], __shfl_xor_sync(0xFFFFFFFFu, bb[0], 1));
            bb[0] = max(bb[0], __shfl_xor_sync(0xFFFFFFFFu, bb[0], 16));
            nvb_sb_codes<1>(bb, sbb, alpha_g, sbT, aem, tab);
            const uint32_t bits = bb[0], sb = sbb[0];
            const float enc = encT[(sb & 0x7Fu) * kNvTabCopies];
            const int64_t m16 = mb + 16 * wr;   // the block's first row
            if (live && (lane & 17) == 0) {
                if (sb_row != nullptr) sb_row[(m16 >> 4) * (K / 16) + (k >> 4)] = (uint8_t)sb;
                if (sb_colT != nullptr) sb_colT[(k >> 4) * (M / 16) + (m16 >> 4)] = (uint8_t)sb;
                nf |= nonfinite(bits);
            }
            uint8_t *qr = q_row + m0 * (K / 2) + (k >> 1);
            const uint64_t g0 = offset + (uint64_t)((m0 * K + k) >> 3);
            const uint32_t dm = RND == 1 ? sr_dither_mask(enc) : 0u;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                float y[8];
                bf16x8_to_f32(v[j], y);
                uint4 R = make_uint4(0u, 0u, 0u, 0u);
                if (RND == 1) R = sr_bits_rk<0>(g0 + (uint64_t)j * (uint64_t)(K >> 3), keys);
                colw[j] = nvb_codes8<RND>(y, enc, R, dm);
                if (q_row != nullptr && live) stg4(qr + j * (K / 2), colw[j]);
            }
            if (q_colT != nullptr) transpose8x8_nibbles(colw);   // now column c -> its 8 rows
        }
        post_nonfinite(status, nf);
        if (q_colT == nullptr) return;
        // ---- columnwise codes: parked as [column][rows / 2 bytes], 4-byte slot tr / 8
        // XOR-swizzled by the column chunk, then written as q_colT rows
#pragma unroll
        for (int c = 0; c < 8; c++)
            *reinterpret_cast<uint32_t *>(park + (tcol + c) * (kNvRows / 2) +
                                          ((((tr >> 3) ^ cc) & (kNvRows / 8 - 1)) * 4)) = colw[c];
        __syncthreads();
        copy_out_fp4T<8, kNvRows, kNvThreads>(park, q_colT, M, K, mb, kb);
        if constexpr (BLK == 0) copy_out_sbT<TC, kNvRows, kNvThreads>(sSB, sb_colT, M, K, mb, kb);
    };

    run_tiles<NvCfg>(&tmap, tiles_m, tiles_k, TC, true, status, pre, body);
}

template <int BLK, int RND>
static cudaError_t nvb_t(const void *x, int64_t M, int64_t K, const float *amax, uint64_t seed, uint64_t offset,
                         uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT, float *s_global,
                         int32_t *status, cudaStream_t st, bool after_amax)
{
    alignas(64) CUtensorMap map;
    if (M != 0 && K != 0) {
        cudaError_t e = make_tile_map(&map, x, BF16, M, K, kNvRows);
        if (e != cudaSuccess) return e;
    } else {
        memset(&map, 0, sizeof map);   // never dereferenced: an empty tensor has no tiles
    }
    {
        const cudaError_t ea = engine_smem_ready<k_nvfp4_bf16<BLK, RND>>(kNvSmem, true);
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kNvRows - 1) / kNvRows) * ((K + 255) / 256);
    const int64_t slots = 2 * (int64_t)sm_count();   // two CTAs per SM
    int grid = (int)(tiles < slots ? tiles : slots);
    if (grid < 1) grid = 1;   // an empty tensor still gets its global scale
    const PhiloxKeys keys = philox_keys(seed);
    return launch_k(after_amax, k_nvfp4_bf16<BLK, RND>, dim3(grid), dim3(kNvThreads), kNvSmem, st, map, M, K, amax,
                    keys, offset, q_row, sb_row, q_colT, sb_colT, s_global, status);
}

cudaError_t launch_nvfp4_bf16(const void *x, int64_t M, int64_t K, int blk, int rnd, uint64_t seed, uint64_t offset,
                              const float *amax, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT,
                              float *s_global, int32_t *status, cudaStream_t st, bool after_amax)
{
#define NVB_ARGS x, M, K, amax, seed, offset, q_row, sb_row, q_colT, sb_colT, s_global, status, st, after_amax
    if (blk == 0) return rnd == 0 ? nvb_t<0, 0>(NVB_ARGS) : nvb_t<0, 1>(NVB_ARGS);
    return rnd == 0 ? nvb_t<1, 0>(NVB_ARGS) : nvb_t<1, 1>(NVB_ARGS);
#undef NVB_ARGS
}

}  // namespace qk
