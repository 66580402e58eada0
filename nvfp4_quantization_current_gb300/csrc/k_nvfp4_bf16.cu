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
// (32 KiB of BF16 each; TileCfg<64, 256>).
//
// Block scales come from two per-CTA tables built once from alpha_g: a byte
// table of sb over the BF16 bit patterns of b in a 24-binade window (below
// it sb is 0, above it 0x7E; see nv_lut_base) and the 128 encode factors
// alpha_g / f(sb).  A block whose maximum is not finite, and every block of
// a CTA whose alpha_g is not a normal float (an amax of inf or NaN), takes
// the two operations instead.
//
// 1x16 (k_nvfp4_bf16_1x16): the warps of a CTA split the two copies.
//   Row warps: a thread quantizes whole 1x16 row blocks (two 16-byte loads
//   from the stage, one 8-byte store of codes, one scale byte), so no block
//   needs a shuffle.
//   Column warps: a thread takes a pair of adjacent columns over 16-row
//   groups of the tile (4-byte loads, 32 lanes on 32 consecutive words).
//   The tile's columnwise codes are collected in shared memory as the dense
//   256 x 32-byte box of q_colT that they fill, and one bulk tensor store
//   (TMA) writes it in whole sectors; scattered 16-byte stores from the
//   lanes cost the load/store pipe a sector operation each.  The scales go
//   out as one word (or bytes) of an sb_colT row per column.
//   With both copies requested warps 0-3 take the rows and 4-7 the columns;
//   with one copy all eight warps take it.
// 16x16 (k_nvfp4_bf16_2d): a thread holds 8 rows x 8 columns (lanes l, l ^ 1,
//   l ^ 16, l ^ 17 share a block), the codes are computed once rowwise and
//   the columnwise copy is their nibble transpose, parked behind the stages
//   and written as q_colT rows.
//
// Stochastic rounding: Philox4x32-10 with round keys formed on the host.
// The rowwise copy takes stream 0 block offset + (m K + k) / 16 for the 16
// consecutive columns k.. of row m, the columnwise copy stream 1 block
// offset + (m / 16) K + k for the 16 consecutive rows m.. of column k (k,
// m multiples of 16); word t of a block serves elements 4t .. 4t + 3, which
// the conversion with random bits rounds (cvt_rs_fp4x4).
#include <cstring>

#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

using NvCfg = TileCfg<64, 256, 3>;
constexpr int kNvRows = NvCfg::kRows, kNvThreads = NvCfg::kThreads, kNvTC = 256;
constexpr int kNvTabCopies = 4;                          // interleaved copies of the encode-factor table
constexpr int kNvParkBytes = 256 * (kNvRows / 2);        // 16x16: parked columnwise codes of a tile
constexpr int kLutBinades = 24, kLut = kLutBinades * 128;
// 1x16: tiles of kN1Rows rows, kN1Ctas CTAs of 256 threads per SM
constexpr int kN1Rows = 64, kN1Ctas = 2;
using N1Cfg = TileCfg<kN1Rows, 256, 3>;
constexpr int kN1BoxBytes = 256 * (kN1Rows / 2);        // columnwise codes of a tile: [256 columns][kN1Rows / 2]

// ---------------------------------------------------------------------------
// block scales
// ---------------------------------------------------------------------------

// sb of a block with maximum b (FP32 bits of |x|, a BF16 value): the two
// operations as written.
QD uint32_t nvb_sb_exact(uint32_t b, float alpha_g)
{
    return b == 0 ? 0x38u : e4m3_code(__fdiv_rn(__fmul_rn(__uint_as_float(b), alpha_g), 6.0f));
}

// First BF16 pattern of the table window for alpha_g with biased exponent
// ea (1..254).  The window covers maxima b with biased exponent E in
// [244 - ea, 268 - ea).  Below it b < 2^(117 - ea) and alpha_g < 2^(ea - 126),
// so b alpha_g < 2^-9 and RN(RN(b alpha_g) / 6) <= RN(2^-9 / 6) < 2^-10, half
// the smallest E4M3 subnormal: code 0.  At or above its top b >= 2^(141 - ea)
// and alpha_g >= 2^(ea - 127), so b alpha_g >= 2^14 and the quotient exceeds
// 448: code 0x7E (the same for b = inf).
QD int nv_lut_base(uint32_t alpha_bits) { return (244 - (int)(alpha_bits >> 23)) * 128; }

// Builds this CTA's tables (all threads; a CTA barrier follows before use).
QD void nv_build_tables(float alpha_g, bool tab, int lut_base, uint8_t *lut, float *enc_tab)
{
    const int t = threadIdx.x;
    if (t < 128) {
        const float sv = e4m3_value(t);
        const float ev = sv == 0.0f ? 0.0f : __fdiv_rn(alpha_g, sv);
#pragma unroll
        for (int j = 0; j < kNvTabCopies; j++) enc_tab[t * kNvTabCopies + j] = ev;
    }
    if (tab) {
        for (int i = t; i < kLut; i += blockDim.x) {
            const int bb = i + lut_base;
            lut[i] = (uint8_t)((bb >= 0 && bb <= 0x7FFF) ? nvb_sb_exact((uint32_t)bb << 16, alpha_g) : 0u);
        }
    }
}

// sb of N blocks with maxima b[] from the table; when any lane of the warp
// holds a non-finite maximum or the CTA has no table, the two operations for
// those (one warp-uniform branch).
template <int N>
QD void nv_sb_codes(const uint32_t (&b)[N], uint32_t (&sb)[N], float alpha_g, const uint8_t *lut, int lut_base,
                    bool tab)
{
    bool rare = !tab;
#pragma unroll
    for (int h = 0; h < N; h++) {
        const int idx = min(max((int)(b[h] >> 16) - lut_base, 0), kLut - 1);
        const uint32_t c = lut[idx];
        sb[h] = b[h] == 0 ? 0x38u : c;
        rare |= b[h] >= 0x7F800000u;
    }
    if (__any_sync(0xFFFFFFFFu, rare)) {
#pragma unroll
        for (int h = 0; h < N; h++)
            if (!tab || b[h] >= 0x7F800000u) sb[h] = nvb_sb_exact(b[h], alpha_g);
    }
}

QD float nv_enc(const float *enc_tab, uint32_t sb, int lane)
{
    return enc_tab[(sb & 0x7Fu) * kNvTabCopies + (lane & (kNvTabCopies - 1))];
}

// ---------------------------------------------------------------------------
// element arithmetic
// ---------------------------------------------------------------------------

// BF16 halves of a word as FP32, by the mixed-precision add x + (-0) (exact;
// it runs on the FMA pipe, which the rest of the kernel leaves less busy
// than the integer / logic pipe).
QD float bf16_lo_f32(uint32_t w)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, l, 0f80000000;\n\t}" : "=f"(r) : "r"(w));
    return r;
}
QD float bf16_hi_f32(uint32_t w)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, h, 0f80000000;\n\t}" : "=f"(r) : "r"(w));
    return r;
}
QD void bf16x8_to_f32(const uint4 &v, float (&y)[8])
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
        y[2 * j] = bf16_lo_f32(word(v, j));
        y[2 * j + 1] = bf16_hi_f32(word(v, j));
    }
}

// E2M1 codes of 8 values (y[0] in bits 3-0) after the products y *= enc;
// with stochastic rounding y[0..3] take the random word r0 and y[4..7] r1.
template <int RND> QD uint32_t nvb_codes8(float (&y)[8], float enc, uint32_t r0, uint32_t r1)
{
#pragma unroll
    for (int j = 0; j < 8; j += 2) mul2(y[j], y[j + 1], enc, enc);
    if (RND == 1) return cvt_rs_fp4x8(y, r0, r1);
    return cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}

// FP32 bits of the larger magnitude of the two BF16 halves of a packed
// |max| word.
QD uint32_t halves_max_bits(uint32_t m)
{
    const uint32_t mm = hmax_abs2(m, __byte_perm(m, 0u, 0x1032));
    return (mm << 16) & 0x7FFF0000u;
}

// ---------------------------------------------------------------------------
// 1x16
// ---------------------------------------------------------------------------

// MODE 0: both copies (warps 0-3 rows, 4-7 columns); 1: rowwise only;
// 2: columnwise only (all warps).
// RHT (with MODE 0): the NVFP4 recipe's two copies in one pass.  The row
// warps quantize x with the tensor scale from *amax; the column warps
// quantize the random Hadamard transform x' = (1/4) H D x of every 16-row
// group of every column (D the signs of sign_mask) with the tensor scale from
// *amax_c, in the order of k_nvfp4_rht: signs on the FP32 bits, the butterfly
// with strides 1, 2, 4, 8, the exact factor 1/4, and the block scale by the
// two operations (x' is not a BF16 value, so the byte table does not apply).
template <int MODE, int RND, bool RHT = false>
__global__ void __launch_bounds__(kNvThreads, kN1Ctas)
    k_nvfp4_bf16_1x16(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K, const float *__restrict__ amax,
                      const __grid_constant__ PhiloxKeys keys, uint64_t offset, uint8_t *__restrict__ q_row,
                      uint8_t *__restrict__ sb_row, uint8_t *__restrict__ q_colT, uint8_t *__restrict__ sb_colT,
                      float *__restrict__ s_global, int32_t *status, const __grid_constant__ CUtensorMap cmap,
                      int col_tma, uint32_t sign_mask, const float *__restrict__ amax_c, float *__restrict__ s_global_c)
{
    static_assert(!RHT || MODE == 0, "the transformed column copy runs beside the row copy");
    constexpr int NR = MODE == 0 ? 128 : MODE == 1 ? 256 : 0;   // row threads (threads 0 .. NR - 1)
    constexpr int NC = kNvThreads - NR;                          // column threads (the rest)
    __shared__ float enc_tab[128 * kNvTabCopies];
    __shared__ float enc_tab_c[RHT ? 128 * kNvTabCopies : 1];   // RHT: alpha_c / f(code) for the column copy
    __shared__ uint8_t lut[kLut];
    extern __shared__ __align__(1024) uint8_t dsm[];
    uint8_t *const park = dsm + N1Cfg::kSmem;   // columnwise codes of a tile: [256 columns][kN1Rows / 2 bytes]

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t tiles_m = (M + kN1Rows - 1) / kN1Rows, tiles_k = (K + kNvTC - 1) / kNvTC;
    float alpha_g = 1.0f;
    float alpha_c = 1.0f;   // RHT: the column copy's tensor scale
    int lut_base = 0;
    bool tab = true;   // alpha_g is a normal float, so the byte table applies

    // after the first tiles are requested: the tensor scale from the amax of
    // the pass ahead of this kernel, and the per-CTA tables
    auto pre = [&] {
        griddep_wait();
        const float A = *amax;
        alpha_g = alpha_from_amax(2688.0f, A);
        const uint32_t ag = __float_as_uint(alpha_g);
        // alpha_g is a normal float for every finite amax (1 for amax 0); a
        // non-finite amax gives 0 or NaN
        tab = (ag >> 23) != 0u && (ag >> 23) != 255u;
        lut_base = nv_lut_base(ag);
        nv_build_tables(alpha_g, tab, lut_base, lut, enc_tab);
        if (blockIdx.x == 0 && t == 0) {
            *s_global = __fdiv_rn(1.0f, alpha_g);
            flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
        }
        if constexpr (RHT) {
            const float Ac = *amax_c;
            alpha_c = alpha_from_amax(2688.0f, Ac);
            if (t < 128) {
                const float sv = e4m3_value(t);
                const float ev = sv == 0.0f ? 0.0f : __fdiv_rn(alpha_c, sv);
#pragma unroll
                for (int j = 0; j < kNvTabCopies; j++) enc_tab_c[t * kNvTabCopies + j] = ev;
            }
            if (blockIdx.x == 0 && t == 0) {
                *s_global_c = __fdiv_rn(1.0f, alpha_c);
                flag_nonfinite(status, __float_as_uint(Ac) & 0x7FFFFFFFu);
            }
        }
        __syncthreads();   // tables visible to every thread
    };

    auto row_part = [&](const uint8_t *st, int64_t mb, int64_t kb, uint32_t &nf) {
        if constexpr (NR > 0) {
            constexpr int RPW = kN1Rows / (NR / 32);          // rows per row warp
            constexpr int BPT = kN1Rows * (kNvTC / 16) / NR;   // blocks per row thread
            // block b of row r: the lane's 16-byte loads go to chunks 2b + s and
            // 2b + 1 - s with s = bit 2 of b, so that the 8 lanes of each load
            // phase hit 8 different 16-byte bank groups
            const int b = lane & 15, s = (b >> 2) & 1;
            const int64_t k0 = kb + 16 * b;
            const int r0 = warp * RPW + (lane >> 4);   // the thread's first row in the tile; it steps by 2
            // rows of this thread still inside the tensor (M is a multiple of 16: tiles past the
            // bottom edge keep whole 16-row groups)
            const int64_t left = M - (mb + r0);
            const int live_rows = k0 < K ? (int)(left < 2 * BPT ? (left > 0 ? left : 0) : 2 * BPT) : 0;
            // row m0 = mb + r0 and its successors every 2 rows: output pointers and the Philox
            // block of the 1x16 block (words 0-1: its first 8 elements, 2-3: the last 8), each
            // advanced by a fixed stride per row pair
            uint8_t *qr = q_row + (mb + r0) * (K / 2) + (k0 >> 1);
            uint8_t *sr = sb_row + (mb + r0) * (K / 16) + (k0 >> 4);
            uint64_t ga = offset + (uint64_t)(((mb + r0) * K + k0) >> 4);
            const int64_t qstep = K, sstep = K / 8;   // two rows of codes / scales
            const uint64_t gstep = (uint64_t)(K >> 3);   // two rows of Philox blocks
            // fully unrolled, except with stochastic rounding beside the column role, where eight
            // copies of the Philox-heavy body next to the column code stall on instruction fetch
            // (ncu: 35.5 -> 44.8 us at 8192 x 4096)
            constexpr int kUnroll = (RND == 1 && NC > 0) ? 2 : BPT;
#pragma unroll kUnroll
            for (int i = 0; i < BPT; i++) {
                const uint8_t *src = st + (r0 + 2 * i) * kRowBytes + 32 * b;
                const uint4 va = lds16(src + 16 * s), vz = lds16(src + 16 - 16 * s);
                const uint32_t mx = hmax_abs2(hmax_abs2(hmax_abs2(va.x, va.y), hmax_abs2(va.z, va.w)),
                                              hmax_abs2(hmax_abs2(vz.x, vz.y), hmax_abs2(vz.z, vz.w)));
                uint32_t bits[1] = {halves_max_bits(mx)}, sb[1];
                nv_sb_codes<1>(bits, sb, alpha_g, lut, lut_base, tab);
                const float enc = nv_enc(enc_tab, sb[0], lane);
                uint4 R = make_uint4(0u, 0u, 0u, 0u);
                if (RND == 1) R = sr_bits_rk<0>(ga, keys);
                // va holds elements 8s .. 8s + 7 of the block, vz the other half
                const uint32_t ra0 = s ? R.z : R.x, ra1 = s ? R.w : R.y, rz0 = s ? R.x : R.z, rz1 = s ? R.y : R.w;
                float y[8];
                bf16x8_to_f32(va, y);
                const uint32_t ca = nvb_codes8<RND>(y, enc, ra0, ra1);
                bf16x8_to_f32(vz, y);
                const uint32_t cz = nvb_codes8<RND>(y, enc, rz0, rz1);
                if (2 * i < live_rows) {
                    stg8(qr, s ? cz : ca, s ? ca : cz);
                    *sr = (uint8_t)sb[0];
                    nf |= nonfinite(bits[0]);
                }
                qr += qstep;
                sr += sstep;
                ga += gstep;
            }
        }
    };

    auto col_part = [&](const uint8_t *st, int64_t mb, int64_t kb, uint32_t &nf) {
        if constexpr (NC > 0) {
            constexpr int GPT = (kN1Rows / 16) * (kNvTC / 2) / NC;   // 16-row groups per column thread
            const int c = t - NR;
            const int p = c & (kNvTC / 2 - 1);
            const int g0 = (c / (kNvTC / 2)) * GPT;
            const int64_t k = kb + 2 * p;
            uint32_t code[2][2 * GPT];   // [column][2 group + half]: 8 rows' nibbles, first row in bits 3-0
            uint32_t sbw[2] = {0u, 0u};  // [column]: scale of group g0 + gi at byte gi
#pragma unroll
            for (int gi = 0; gi < GPT; gi++) {
                const int g = g0 + gi;
                const uint8_t *src = st + (16 * g) * kRowBytes + 4 * p;
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; j++) w[j] = *reinterpret_cast<const uint32_t *>(src + j * kRowBytes);
                if constexpr (RHT) {
                const int64_t m16 = mb + 16 * g;
                const bool live = m16 < M && k < K;
                // columns 2p (a) and 2p + 1 (b) of the group's 16 rows: signs,
                // butterfly, 1/4
                float a[16], bv[16];
#pragma unroll
                for (int r = 0; r < 16; r++) {
                    const uint32_t neg = ((sign_mask >> r) & 1u) << 31;
                    a[r] = __uint_as_float((w[r] << 16) ^ neg);
                    bv[r] = __uint_as_float((w[r] & 0xFFFF0000u) ^ neg);
                }
#pragma unroll
                for (int hs = 1; hs < 16; hs *= 2)
#pragma unroll
                    for (int r = 0; r < 16; r++)
                        if ((r & hs) == 0) bfly2(a[r], bv[r], a[r + hs], bv[r + hs]);
#pragma unroll
                for (int r = 0; r < 16; r++) mul2(a[r], bv[r], 0.25f, 0.25f);
                float ma = 0.0f, mbx = 0.0f;
#pragma unroll
                for (int r = 0; r < 16; r++) {
                    ma = fmax_abs(ma, a[r]);
                    mbx = fmax_abs(mbx, bv[r]);
                }
                const uint32_t ba = __float_as_uint(ma) & 0x7FFFFFFFu, bb = __float_as_uint(mbx) & 0x7FFFFFFFu;
                const uint32_t sa = nvb_sb_exact(ba, alpha_c), sbb = nvb_sb_exact(bb, alpha_c);
                const float ea = nv_enc(enc_tab_c, sa, lane), eb = nv_enc(enc_tab_c, sbb, lane);
#pragma unroll
                for (int r = 0; r < 16; r++) mul2(a[r], bv[r], ea, eb);
                // rows m16 .. m16 + 15 of columns k, k + 1, stream 1: Philox blocks
                // (m16 / 16) K + column, words 0-1 for rows 0-7 and 2-3 for rows 8-15
                uint4 Ra = make_uint4(0u, 0u, 0u, 0u), Rb = Ra;
                if constexpr (RND == 1) {
                    const uint64_t gb = offset + (uint64_t)((m16 >> 4) * K + k);
                    Ra = sr_bits_rk<1>(gb, keys);
                    Rb = sr_bits_rk<1>(gb + 1, keys);
                }
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    const float *pa = a + 8 * hh, *pb = bv + 8 * hh;
                    if constexpr (RND == 1) {
                        code[0][2 * gi + hh] = cvt_rs_fp4x8(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], pa[6], pa[7],
                                                            hh ? Ra.z : Ra.x, hh ? Ra.w : Ra.y);
                        code[1][2 * gi + hh] = cvt_rs_fp4x8(pb[0], pb[1], pb[2], pb[3], pb[4], pb[5], pb[6], pb[7],
                                                            hh ? Rb.z : Rb.x, hh ? Rb.w : Rb.y);
                    } else {
                        code[0][2 * gi + hh] = cvt_fp4x8(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], pa[6], pa[7]);
                        code[1][2 * gi + hh] = cvt_fp4x8(pb[0], pb[1], pb[2], pb[3], pb[4], pb[5], pb[6], pb[7]);
                    }
                }
                sbw[0] |= sa << (8 * gi);
                sbw[1] |= sbb << (8 * gi);
                nf |= live ? nonfinite(ba) | nonfinite(bb) : 0u;
                } else {
                uint32_t m8[8];
#pragma unroll
                for (int j = 0; j < 8; j++) m8[j] = hmax_abs2(w[j], w[j + 8]);
#pragma unroll
                for (int j = 0; j < 4; j++) m8[j] = hmax_abs2(m8[j], m8[j + 4]);
                const uint32_t mx = hmax_abs2(hmax_abs2(m8[0], m8[2]), hmax_abs2(m8[1], m8[3]));
                uint32_t bits[2] = {(mx << 16) & 0x7FFF0000u, mx & 0x7FFF0000u}, sb[2];
                nv_sb_codes<2>(bits, sb, alpha_g, lut, lut_base, tab);
                const int64_t m16 = mb + 16 * g;
                const bool live = m16 < M && k < K;
#pragma unroll
                for (int h = 0; h < 2; h++) {   // h = 0: column 2p (low halves), 1: column 2p + 1
                    const float enc = nv_enc(enc_tab, sb[h], lane);
                    // the column's 16 rows, stream 1: Philox block (m16 / 16) K + column
                    uint4 R = make_uint4(0u, 0u, 0u, 0u);
                    if (RND == 1) R = sr_bits_rk<1>(offset + (uint64_t)((m16 >> 4) * K + k + h), keys);
#pragma unroll
                    for (int half = 0; half < 2; half++) {   // rows 8 half .. 8 half + 7 of the group
                        float y[8];
#pragma unroll
                        for (int j = 0; j < 8; j++) y[j] = h ? bf16_hi_f32(w[8 * half + j]) : bf16_lo_f32(w[8 * half + j]);
                        code[h][2 * gi + half] = nvb_codes8<RND>(y, enc, half ? R.z : R.x, half ? R.w : R.y);
                    }
                    sbw[h] |= sb[h] << (8 * gi);
                    nf |= live ? nonfinite(bits[h]) : 0u;
                }
                }
            }
            if (col_tma) {
                // the tile's columnwise codes as a dense [256 columns][kN1Rows / 2
                // bytes] box, which one bulk tensor store writes (the parts past
                // the tensor's edges are not written)
                if (c == 0) bulk_wait_read_all();   // the previous tile's store has read the box
                named_barrier(1, NC);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    uint8_t *dst = park + (2 * p + h) * (kN1Rows / 2) + 8 * g0;
                    if constexpr (GPT == 1) {
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(code[h][0], code[h][1]);
                    } else {
#pragma unroll
                        for (int q = 0; q < GPT / 2; q++)
                            *reinterpret_cast<uint4 *>(dst + 16 * q) =
                                make_uint4(code[h][4 * q], code[h][4 * q + 1], code[h][4 * q + 2], code[h][4 * q + 3]);
                    }
                }
                fence_proxy_async();   // generic-proxy writes of the box before the async-proxy read
                named_barrier(1, NC);
                if (c == 0) {
                    tma_store_tile(&cmap, park, (int)(mb / 2), (int)kb);
                    bulk_commit();
                }
            }
            if (k < K) {
                const int64_t mg = mb + 16 * g0;   // first row of this thread's groups
                const int64_t left = (M - mg) / 16;
                const int ng = left < GPT ? (int)(left > 0 ? left : 0) : GPT;   // groups inside the tensor
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    uint8_t *qc = q_colT + (k + h) * (M / 2) + mg / 2;
                    uint8_t *sc = sb_colT + (k + h) * (M / 16) + mg / 16;
                    if (col_tma) {
                        // codes leave with the bulk store
                    } else if (GPT >= 2 && ng == GPT && (M & 31) == 0) {
#pragma unroll
                        for (int q = 0; q < GPT / 2; q++)
                            stg16(qc + 16 * q, make_uint4(code[h][4 * q], code[h][4 * q + 1], code[h][4 * q + 2],
                                                          code[h][4 * q + 3]));
                    } else {
#pragma unroll
                        for (int gi = 0; gi < GPT; gi++)
                            if (gi < ng) stg8(qc + 8 * gi, code[h][2 * gi], code[h][2 * gi + 1]);
                    }
                    if (GPT == 4 && ng == 4 && (M & 63) == 0) {
                        stg4(sc, sbw[h]);
                    } else if (GPT == 2 && ng == 2 && (M & 31) == 0) {
                        *reinterpret_cast<uint16_t *>(sc) = (uint16_t)sbw[h];
                    } else {
#pragma unroll
                        for (int gi = 0; gi < GPT; gi++)
                            if (gi < ng) sc[gi] = (uint8_t)(sbw[h] >> (8 * gi));
                    }
                }
            }
        }
    };

    auto body = [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kN1Rows, kb = tk * kNvTC;
        uint32_t nf = 0;   // a non-finite block maximum seen by this thread
        if (t < NR) row_part(st, mb, kb, nf);
        else col_part(st, mb, kb, nf);
        post_nonfinite(status, nf);
    };

    run_tiles<N1Cfg>(&tmap, tiles_m, tiles_k, kNvTC, true, status, pre, body);
    if (NC > 0 && col_tma && t == NR) bulk_wait_all();   // the last box is written before the CTA ends
}

// ---------------------------------------------------------------------------
// 16x16
// ---------------------------------------------------------------------------

// Thread layout: the 8 warps of a CTA cover a 64 x 256 tile: warp w takes
// rows 16 (w / 2) .. + 15 and columns 128 (w % 2) .. + 127 of the tile; lane
// l takes 8 of those rows (8 (l / 16) .. + 7) of one 16-byte column chunk
// (columns 8 (l % 16) .. + 7), so a 16x16 block is the lanes l, l ^ 1, l ^ 16,
// l ^ 17.  The columnwise codes of a thread (one word of 8 row nibbles per
// column) are parked in a buffer of their own behind the stages and leave as
// 16-byte pieces of q_colT rows.
template <int RND>
__global__ void __launch_bounds__(kNvThreads, 2)
    k_nvfp4_bf16_2d(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K, const float *__restrict__ amax,
                    const __grid_constant__ PhiloxKeys keys, uint64_t offset, uint8_t *__restrict__ q_row,
                    uint8_t *__restrict__ sb_row, uint8_t *__restrict__ q_colT, uint8_t *__restrict__ sb_colT,
                    float *__restrict__ s_global, int32_t *status)
{
    __shared__ float enc_tab[128 * kNvTabCopies];
    __shared__ uint8_t lut[kLut];
    extern __shared__ __align__(1024) uint8_t dsm[];
    uint8_t *const park = dsm + NvCfg::kSmem;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int wr = warp >> 1, wc = warp & 1, rp = lane >> 4, cc = lane & 15;
    const int tr = 16 * wr + 8 * rp;      // the thread's first row in a tile
    const int tcol = 128 * wc + 8 * cc;   // its first column in a tile
    const int64_t tiles_m = (M + kNvRows - 1) / kNvRows, tiles_k = (K + kNvTC - 1) / kNvTC;
    float alpha_g = 1.0f;
    int lut_base = 0;
    bool tab = true;

    auto pre = [&] {
        griddep_wait();
        const float A = *amax;
        alpha_g = alpha_from_amax(2688.0f, A);
        const uint32_t ag = __float_as_uint(alpha_g);
        tab = (ag >> 23) != 0u && (ag >> 23) != 255u;
        lut_base = nv_lut_base(ag);
        nv_build_tables(alpha_g, tab, lut_base, lut, enc_tab);
        if (blockIdx.x == 0 && t == 0) {
            *s_global = __fdiv_rn(1.0f, alpha_g);
            flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
        }
        __syncthreads();
    };

    auto body = [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kNvRows, kb = tk * kNvTC;
        const int64_t m0 = mb + tr, k = kb + tcol;
        // M and K are multiples of 16: a thread's 8 rows and 8 columns are all
        // inside the tensor or all outside
        const bool live = m0 < M && k < K;
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = lds16(st + (tr + j) * kRowBytes + 2 * tcol);
        uint32_t colw[8];   // the 8 rows' codes, then (transposed) the 8 columns'
        uint32_t nf = 0;
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) m = hmax_abs2(m, hmax_abs2(hmax_abs2(v[j].x, v[j].y), hmax_abs2(v[j].z, v[j].w)));
        uint32_t bb[1] = {halves_max_bits(m)}, sbb[1];
        bb[0] = max(bb[0], __shfl_xor_sync(0xFFFFFFFFu, bb[0], 1));
        bb[0] = max(bb[0], __shfl_xor_sync(0xFFFFFFFFu, bb[0], 16));
        nv_sb_codes<1>(bb, sbb, alpha_g, lut, lut_base, tab);
        const uint32_t bits = bb[0], sb = sbb[0];
        const float enc = nv_enc(enc_tab, sb, lane);
        const int64_t m16 = mb + 16 * wr;   // the block's first row
        if (live && (lane & 17) == 0) {
            if (sb_row != nullptr) sb_row[(m16 >> 4) * (K / 16) + (k >> 4)] = (uint8_t)sb;
            if (sb_colT != nullptr) sb_colT[(k >> 4) * (M / 16) + (m16 >> 4)] = (uint8_t)sb;
            nf |= nonfinite(bits);
        }
        uint8_t *qr = q_row + m0 * (K / 2) + (k >> 1);
        // row m0 + j: Philox block of its 16 columns k & ~15 ..; this thread's 8
        // columns are that block's first half (words 0-1) or second (2-3)
        const uint64_t g0 = offset + (uint64_t)((m0 * K + k) >> 4);
        const bool hi8 = (k & 8) != 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float y[8];
            bf16x8_to_f32(v[j], y);
            uint4 R = make_uint4(0u, 0u, 0u, 0u);
            if (RND == 1) R = sr_bits_rk<0>(g0 + (uint64_t)j * (uint64_t)(K >> 4), keys);
            colw[j] = nvb_codes8<RND>(y, enc, hi8 ? R.z : R.x, hi8 ? R.w : R.y);
            if (q_row != nullptr && live) stg4(qr + j * (K / 2), colw[j]);
        }
        post_nonfinite(status, nf);
        if (q_colT == nullptr) return;
        transpose8x8_nibbles(colw);   // now column c -> its 8 rows
        // parked as [column][rows / 2 bytes], 4-byte slot tr / 8 XOR-swizzled
        // by the column chunk, then written as q_colT rows
#pragma unroll
        for (int c = 0; c < 8; c++)
            *reinterpret_cast<uint32_t *>(park + (tcol + c) * (kNvRows / 2) +
                                          ((((tr >> 3) ^ cc) & (kNvRows / 8 - 1)) * 4)) = colw[c];
        __syncthreads();
        copy_out_fp4T<8, kNvRows, kNvThreads>(park, q_colT, M, K, mb, kb);
    };

    run_tiles<NvCfg>(&tmap, tiles_m, tiles_k, kNvTC, true, status, pre, body);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

// 1x16: the input's tensor map, and, when the columnwise copy is requested
// and its rows (M / 2 bytes) are a multiple of 16 bytes, a store map over
// q_colT for the bulk tensor stores of the column warps.
template <auto Kernel>
static cudaError_t nvb_launch_1x16(const void *x, int64_t M, int64_t K, const float *amax, uint64_t seed,
                                   uint64_t offset, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT,
                                   float *s_global, int32_t *status, cudaStream_t st, bool after_amax,
                                   uint32_t sign_mask = 0, const float *amax_c = nullptr, float *s_global_c = nullptr)
{
    constexpr int smem = N1Cfg::kSmem + kN1BoxBytes;
    alignas(64) CUtensorMap map, cmap;
    memset(&map, 0, sizeof map);
    memset(&cmap, 0, sizeof cmap);
    int col_tma = 0;
    if (M != 0 && K != 0) {
        cudaError_t e = make_tile_map(&map, x, BF16, M, K, kN1Rows);
        if (e != cudaSuccess) return e;
        if (q_colT != nullptr && (M % 32) == 0) {
            e = make_store_map_u8(&cmap, q_colT, M / 2, K, kN1Rows / 2, kNvTC);
            if (e != cudaSuccess) return e;
            col_tma = 1;
        }
    }
    {
        const cudaError_t ea = engine_smem_ready<Kernel>(smem, true);
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kN1Rows - 1) / kN1Rows) * ((K + kNvTC - 1) / kNvTC);
    const int64_t slots = kN1Ctas * (int64_t)sm_count();   // kN1Ctas CTAs per SM
    int grid = (int)(tiles < slots ? tiles : slots);
    if (grid < 1) grid = 1;   // an empty tensor still gets its global scale
    const PhiloxKeys keys = philox_keys(seed);
    return launch_k(after_amax, Kernel, dim3(grid), dim3(kNvThreads), smem, st, map, M, K, amax, keys, offset, q_row,
                    sb_row, q_colT, sb_colT, s_global, status, cmap, col_tma, sign_mask, amax_c, s_global_c);
}

template <auto Kernel>
static cudaError_t nvb_launch(int smem, const void *x, int64_t M, int64_t K, const float *amax, uint64_t seed,
                              uint64_t offset, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT,
                              float *s_global, int32_t *status, cudaStream_t st, bool after_amax)
{
    alignas(64) CUtensorMap map;
    if (M != 0 && K != 0) {
        cudaError_t e = make_tile_map(&map, x, BF16, M, K, kNvRows);
        if (e != cudaSuccess) return e;
    } else {
        memset(&map, 0, sizeof map);   // never dereferenced: an empty tensor has no tiles
    }
    {
        const cudaError_t ea = engine_smem_ready<Kernel>(smem, true);
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kNvRows - 1) / kNvRows) * ((K + kNvTC - 1) / kNvTC);
    const int64_t slots = 2 * (int64_t)sm_count();   // two CTAs per SM
    int grid = (int)(tiles < slots ? tiles : slots);
    if (grid < 1) grid = 1;   // an empty tensor still gets its global scale
    const PhiloxKeys keys = philox_keys(seed);
    return launch_k(after_amax, Kernel, dim3(grid), dim3(kNvThreads), smem, st, map, M, K, amax, keys, offset, q_row,
                    sb_row, q_colT, sb_colT, s_global, status);
}

cudaError_t launch_nvfp4_bf16(const void *x, int64_t M, int64_t K, int blk, int rnd, uint64_t seed, uint64_t offset,
                              const float *amax, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT,
                              float *s_global, int32_t *status, cudaStream_t st, bool after_amax)
{
#define NVB_ARGS x, M, K, amax, seed, offset, q_row, sb_row, q_colT, sb_colT, s_global, status, st, after_amax
    if (blk == 1) {
        constexpr int smem = NvCfg::kSmem + kNvParkBytes;
        return rnd == 0 ? nvb_launch<k_nvfp4_bf16_2d<0>>(smem, NVB_ARGS) : nvb_launch<k_nvfp4_bf16_2d<1>>(smem, NVB_ARGS);
    }
    if (q_row != nullptr && q_colT != nullptr)
        return rnd == 0 ? nvb_launch_1x16<k_nvfp4_bf16_1x16<0, 0>>(NVB_ARGS)
                        : nvb_launch_1x16<k_nvfp4_bf16_1x16<0, 1>>(NVB_ARGS);
    if (q_colT == nullptr)   // rowwise only (also an empty tensor with no outputs)
        return rnd == 0 ? nvb_launch_1x16<k_nvfp4_bf16_1x16<1, 0>>(NVB_ARGS)
                        : nvb_launch_1x16<k_nvfp4_bf16_1x16<1, 1>>(NVB_ARGS);
    return rnd == 0 ? nvb_launch_1x16<k_nvfp4_bf16_1x16<2, 0>>(NVB_ARGS)
                    : nvb_launch_1x16<k_nvfp4_bf16_1x16<2, 1>>(NVB_ARGS);
#undef NVB_ARGS
}

// The NVFP4 recipe's two copies of a BF16 tensor in one pass (the rowwise
// 1x16 copy of x with the tensor scale from amax_row, the columnwise copy of
// its random Hadamard transform with the one from amax_col), behind the pass
// that reduced both maxima (after_amax) or with maxima given.
cudaError_t launch_nvfp4_bf16_recipe(const void *x, int64_t M, int64_t K, uint32_t sign_mask, int rnd, uint64_t seed,
                                     uint64_t offset, const float *amax_row, uint8_t *q_row, uint8_t *sb_row,
                                     float *s_global_row, const float *amax_col, uint8_t *q_colT, uint8_t *sb_colT,
                                     float *s_global_col, int32_t *status, cudaStream_t st, bool after_amax)
{
#define NVR_ARGS x, M, K, amax_row, seed, offset, q_row, sb_row, q_colT, sb_colT, s_global_row, status, st, after_amax, \
                 sign_mask, amax_col, s_global_col
    return rnd == 0 ? nvb_launch_1x16<k_nvfp4_bf16_1x16<0, 0, true>>(NVR_ARGS)
                    : nvb_launch_1x16<k_nvfp4_bf16_1x16<0, 1, true>>(NVR_ARGS);
#undef NVR_ARGS
}

}  // namespace qk
