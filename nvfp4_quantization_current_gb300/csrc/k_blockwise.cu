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
// and TC/128 blocks in K; thread (warp w, lane l) holds rows 8w..8w+7 x one
// 16-byte column chunk in registers.
//  1x128 rowwise  - a block spans 128/VEC lanes (xor-shuffle max);
//  128x1 colwise  - per-warp column maxima of the registers meet in shared
//                   memory, one thread per column reduces them to the
//                   column's alpha and s; the column-scaled codes of the same
//                   registers are byte-transposed, parked in the consumed
//                   stage and written as full 128-byte q_colT rows;
//  128x128        - the tile maximum comes from warp shuffles and one
//                   shared-memory reduction across the 16 warps; the
//                   transposed copy is the same codes byte-transposed.
//
// With P2 the tiles are held as MXFP8 ("Mixed-precision training ...",
// "Blockwise scaling": on Blackwell the recipe is emulated with MXFP8, a 1x128
// tile being 4 MXFP8 blocks that share one scale): the tile scale is b / 448
// rounded up to a power of two, stored as its E8M0 code once per 32 elements
// (e_row [M, K/32], e_colT [K, M/32]), and alpha = 2^(127 - code).
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

// E8M0 code of the power-of-two tile scale: the smallest 2^n with
// b <= 448 * 2^n, code = 127 + n clamped to [0, 254].  For b = (1 + f)
// 2^(E - 127) and 448 = 1.75 * 2^8 that is E - 8, plus one when the mantissa
// field exceeds that of 1.75 (0x600000); b = 0 -> 127 (scale 1); inf / NaN
// (E = 255) -> 247, the MXFP8 code of that exponent field.
QD uint32_t bw_p2_code(uint32_t b)
{
    if (b == 0u) return 127u;
    const int E = (int)(b >> 23);
    if (E == 255) return 247u;
    const int c = E - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return (uint32_t)(c < 0 ? 0 : (c > 254 ? 254 : c));
}

// alpha (and the FP32 s, or the E8M0 code with P2) of a tile maximum b.
template <int DT, bool P2> QD void bw_tile_scale(uint32_t b, const BwScaleTab &tab, float &alpha, float &s, uint32_t &code)
{
    if constexpr (P2) {
        code = bw_p2_code(b);
        alpha = mx_inv_scale(code);
        s = 0.0f;
    } else {
        bw_scales<DT>(b, tab, alpha, s);
        code = 0u;
    }
}

template <int DT, int TILE, bool P2>
__global__ void __launch_bounds__(kEngThreads, 1) k_blockwise(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                              uint8_t *__restrict__ q_row, void *__restrict__ sc_row,
                                                              uint8_t *__restrict__ q_colT, void *__restrict__ sc_colT,
                                                              int32_t *status)
{
    // scales: FP32 [M, K/128] / [K, M/128] (2D: [M/128, K/128] / [K/128, M/128]),
    // or with P2 E8M0 codes [M, K/32] / [K, M/32], one 4-byte word per 128 elements
    float *const s_row = static_cast<float *>(sc_row), *const s_colT = static_cast<float *>(sc_colT);
    uint8_t *const e_row = static_cast<uint8_t *>(sc_row), *const e_colT = static_cast<uint8_t *>(sc_colT);
    constexpr uint32_t kRep4 = 0x01010101u;
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, CW = VEC / 4, LPB = 128 / VEC;
    constexpr int NT = TC / 128;   // 128-column blocks per tile
    __shared__ uint4 part[kEngWarps][32];      // 1x128: per-warp column maxima (packed like the input)
    __shared__ __align__(16) float calpha[TC];   // 1x128: column alphas of the tile
    __shared__ uint32_t tred[kEngWarps][NT];   // 128x128: per-warp tile maxima
    __shared__ BwScaleTab tab;
    if (DT == BF16 && !P2 && threadIdx.x < 128) {
        const float a = __fdiv_rn(448.0f, 1.0f + (float)threadIdx.x * (1.0f / 128.0f));
        tab.a[threadIdx.x] = a;
        tab.s[threadIdx.x] = __fdiv_rn(1.0f, a);
    }   // visible after the engine's first barrier

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;

    run_tiles(&tmap, tiles_m, tiles_k, TC, false, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        const int64_t k = kb + lane * VEC, m0 = mb + 8 * warp;
        const bool kok = k < K;
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = lds16(st + (8 * warp + j) * kRowBytes + lane * 16);
        uint32_t code[8][CW];
        uint32_t cc2 = 0;   // 128x128 with P2: this lane's block code
        // 128x128 with P2: the code once per 32 elements, one 4-byte word per
        // thread: threads 0 .. 128*NT-1 take a row and block of e_row, threads
        // 256 .. 256+TC-1 a column of e_colT.  Lane h*LPB of every warp holds
        // block h's code (the branches are warp-uniform).  Issued after the
        // tile's codes are out.
        auto put_p2_codes = [&]() {
            if (t < 128 * NT) {
                const int r = t / NT, h = t % NT;
                const uint32_t ch = __shfl_sync(0xFFFFFFFFu, cc2, h * LPB);
                if (e_row != nullptr && kb + 128 * h < K)
                    stg4(e_row + (mb + r) * (K / 32) + (kb / 128 + h) * 4, ch * kRep4);
            } else if (t >= 256 && t < 256 + TC) {
                const int c = t - 256;
                const uint32_t ch = __shfl_sync(0xFFFFFFFFu, cc2, (c / 128) * LPB);
                if (e_colT != nullptr && kb + c < K) stg4(e_colT + (kb + c) * (M / 32) + tm * 4, ch * kRep4);
            }
        };

        if constexpr (TILE == 0) {
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
            // ---------------- 1x128 rowwise ----------------
            uint32_t nf = 0;
            if (DT == BF16 && q_row != nullptr) {
                // A block is one row of 16 lanes.  The 8 row maxima, two BF16
                // magnitudes per word, are reduced over the 16 lanes by a halving
                // exchange (5 shuffles); afterwards lane L of the group holds the
                // maximum of row (L >> 1) & 7, computes that row's alpha and s once,
                // and the alphas go back to every lane by index shuffles.
                const int nrows = !kok ? 0 : (m0 + 8 <= M ? 8 : (m0 < M ? (int)(M - m0) : 0));
                uint32_t P[4];
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const uint4 &a = v[2 * p], &b = v[2 * p + 1];
                    const uint32_t ma = hmax_abs2(hmax_abs2(a.x, a.y), hmax_abs2(a.z, a.w));
                    const uint32_t mb = hmax_abs2(hmax_abs2(b.x, b.y), hmax_abs2(b.z, b.w));
                    P[p] = hmax_abs2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));   // row 2p low, 2p+1 high
                }
                const int L = lane & 15;
                const bool b3 = L & 8, b2 = L & 4, b1 = L & 2;
                uint32_t k0 = b3 ? P[2] : P[0], k1 = b3 ? P[3] : P[1];          // keep rows 4*b3 .. 4*b3+3
                const uint32_t s0 = b3 ? P[0] : P[2], s1 = b3 ? P[1] : P[3];
                k0 = hmax_abs2(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, 8));
                k1 = hmax_abs2(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, 8));
                uint32_t kw = b2 ? k1 : k0;                                        // rows 4*b3+2*b2, +1
                kw = hmax_abs2(kw, __shfl_xor_sync(0xFFFFFFFFu, b2 ? k0 : k1, 4));
                kw = hmax_abs2(kw, __shfl_xor_sync(0xFFFFFFFFu, kw, 2));
                kw = hmax_abs2(kw, __shfl_xor_sync(0xFFFFFFFFu, kw, 1));
                const int r = (L >> 1) & 7;
                const uint32_t bm = (b1 ? kw : (kw << 16)) & 0x7FFF0000u;         // FP32 bits of row r's block max
                float alpha_r, s_r;
                uint32_t c_r;
                bw_tile_scale<DT, P2>(bm, tab, alpha_r, s_r, c_r);
                if ((L & 1) == 0 && r < nrows) {
                    if (P2) stg4(e_row + (m0 + r) * (K / 32) + (k / 128) * 4, c_r * kRep4);
                    else s_row[(m0 + r) * (K / 128) + k / 128] = s_r;
                    nf |= nonfinite(bm);
                }
                uint8_t *qr = q_row + m0 * K + k;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float alpha = __shfl_sync(0xFFFFFFFFu, alpha_r, (lane & 16) + 2 * j);
                    uint32_t o[CW];
                    chunk_fp8<DT, E4M3>(v[j], alpha, o);
                    if (j < nrows) {
                        if (CW == 2) stg8(qr + j * K, o[0], o[CW - 1]);
                        else stg4(qr + j * K, o[0]);
                    }
                }
            } else if (q_row != nullptr) {
                // rows of this thread that exist (all 8 except in the last tile row)
                const int nrows = !kok ? 0 : (m0 + 8 <= M ? 8 : (m0 < M ? (int)(M - m0) : 0));
                uint8_t *qr = q_row + m0 * K + k;
                const bool sl = lane % LPB == 0;
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    uint32_t bb[2] = {absmax_bits<DT>(v[j]), absmax_bits<DT>(v[j + 1])};
                    group_max2<DT, LPB>(bb[0], bb[1]);
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        float alpha, sc;
                        uint32_t cc;
                        bw_tile_scale<DT, P2>(bb[h], tab, alpha, sc, cc);
                        uint32_t o[CW];
                        chunk_fp8<DT, E4M3>(v[j + h], alpha, o);
                        if (j + h < nrows) {
                            uint8_t *dst = qr + (j + h) * K;
                            if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                            else stg4(dst, o[0]);
                            if (sl && P2) stg4(e_row + (m0 + j + h) * (K / 32) + (k / 128) * 4, cc * kRep4);
                            if (sl && !P2) s_row[(m0 + j + h) * (K / 128) + k / 128] = sc;
                            nf |= nonfinite(bb[h]);
                        }
                    }
                }
            }
            post_nonfinite(status, nf);
            if (q_colT == nullptr) return;
            __syncthreads();   // partial column maxima posted
            // ---------------- 128x1 columnwise ----------------
            if constexpr (DT == BF16) {
                // four threads per BF16 column pair (one 32-bit word of the
                // partials), each reducing 4 of the 16 warp partials; two shuffles
                // combine them and two of the four take one column each
                const int wp = t >> 2, sub = t & 3;          // 128 column pairs
                const int q = wp >> 2, wi = wp & 3;          // lane q of the partials, word wi
                const uint32_t *pw = reinterpret_cast<const uint32_t *>(&part[0][0]) + q * 4 + wi;
                uint32_t b2 = 0;
#pragma unroll
                for (int w = sub; w < kEngWarps; w += 4) b2 = hmax_abs2(b2, pw[w * 32 * 4]);
                b2 = hmax_abs2(b2, __shfl_xor_sync(0xFFFFFFFFu, b2, 1));
                b2 = hmax_abs2(b2, __shfl_xor_sync(0xFFFFFFFFu, b2, 2));
                if (sub < 2) {
                    const int col = 2 * wp + sub;             // low half: even column
                    const uint32_t b = (sub ? b2 : (b2 << 16)) & 0x7FFF0000u;
                    float alpha, sc;
                    uint32_t cc;
                    bw_tile_scale<DT, P2>(b, tab, alpha, sc, cc);
                    calpha[col] = alpha;
                    if (kb + col < K) {
                        if (P2) stg4(e_colT + (kb + col) * (M / 32) + tm * 4, cc * kRep4);
                        else s_colT[(kb + col) * (M / 128) + tm] = sc;
                        flag_nonfinite(status, b);
                    }
                }
            } else {
                constexpr int TPC = 2 * kEngThreads / TC >= 2 ? 2 : 1;   // threads per column (TC <= 256)
                const int col = t / TPC, half = t % TPC;
                if (col < TC) {
                    const int q = col / VEC, c = col % VEC;   // lane q of the partials holds this column
                    uint32_t b = 0;
#pragma unroll
                    for (int w = half; w < kEngWarps; w += TPC) b = max(b, colmax_bits<DT>(part[w][q], c));
                    if (TPC == 2) b = max(b, __shfl_xor_sync(0xFFFFFFFFu, b, 1));
                    if (half == 0) {
                        float alpha, sc;
                        uint32_t cc;
                        bw_tile_scale<DT, P2>(b, tab, alpha, sc, cc);
                        calpha[col] = alpha;
                        if (kb + col < K) {
                            if (P2) stg4(e_colT + (kb + col) * (M / 32) + tm * 4, cc * kRep4);
                            else s_colT[(kb + col) * (M / 128) + tm] = sc;
                            flag_nonfinite(status, b);
                        }
                    }
                }
            }
            __syncthreads();   // column alphas visible; every read of the stage is done
            float ca[VEC];
#pragma unroll
            for (int c = 0; c < VEC; c += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&calpha[lane * VEC + c]);
                ca[c] = a4.x;
                ca[c + 1] = a4.y;
                ca[c + 2] = a4.z;
                ca[c + 3] = a4.w;
            }
#pragma unroll
            for (int j = 0; j < 8; j++) {
                float f[VEC];
#pragma unroll
                for (int c = 0; c < VEC; c++) f[c] = elem<DT>(v[j], c);
#pragma unroll
                for (int c = 0; c < VEC; c += 2) mul2(f[c], f[c + 1], ca[c], ca[c + 1]);
#pragma unroll
                for (int q = 0; q < CW; q++) code[j][q] = cvt_fp8x4<E4M3>(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
            }
        } else {
            // ---------------- 128x128: one scale per tile ----------------
            uint32_t b = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) b = max(b, absmax_bits<DT>(v[j]));
            b = group_max<LPB>(b);
            if (lane % LPB == 0) tred[warp][lane / LPB] = b;
            __syncthreads();   // tile maxima posted; every read of the stage is done
            uint32_t bt;
            if constexpr (NT * kEngWarps == 32) {
                // lane l fetches warp (l % 16)'s maximum of block l / 16 (the block
                // of its own columns); 4 shuffles reduce over the 16 warps
                bt = tred[lane & 15][lane >> 4];
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) bt = max(bt, __shfl_xor_sync(0xFFFFFFFFu, bt, o));
            } else {
                bt = 0;
#pragma unroll
                for (int q = 0; q < kEngWarps; q++) bt = max(bt, tred[q][lane / LPB]);
            }
            float alpha, sc;
            uint32_t cc;
            bw_tile_scale<DT, P2>(bt, tab, alpha, sc, cc);
            if (!P2 && warp == 0 && lane % LPB == 0 && kok) {
                if (s_row != nullptr) s_row[tm * (K / 128) + k / 128] = sc;
                if (s_colT != nullptr) s_colT[(k / 128) * (M / 128) + tm] = sc;
            }
            cc2 = cc;
            if (warp == 0 && lane % LPB == 0 && kok) flag_nonfinite(status, bt);
#pragma unroll
            for (int j = 0; j < 8; j++) chunk_fp8<DT, E4M3>(v[j], alpha, code[j]);
            if (q_row != nullptr && kok) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    uint8_t *dst = q_row + (m0 + j) * K + k;
                    if (CW == 2) stg8(dst, code[j][0], code[j][CW - 1]);
                    else stg4(dst, code[j][0]);
                }
            }
            if (q_colT == nullptr) {
                if constexpr (P2) put_p2_codes();
                return;
            }
        }
        // ---- transposed codes: parked in the consumed stage, then full 128-byte rows
        park_fp8T<VEC>(st, code, warp, lane);
        __syncthreads();
        copy_out_fp8T<VEC>(st, q_colT, M, K, mb, kb);
        if constexpr (TILE == 1 && P2) put_p2_codes();
    });
}

template <int DT, int TILE, bool P2>
static cudaError_t bw_t(const void *x, int64_t M, int64_t K, uint8_t *q_row, void *s_row, uint8_t *q_colT,
                        void *s_colT, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    alignas(64) CUtensorMap map;
    cudaError_t e = make_tile_map(&map, x, DT, M, K);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t ea = engine_smem_ready<k_blockwise<DT, TILE, P2>>();
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kTileRowsE - 1) / kTileRowsE) * ((K + TC - 1) / TC);
    const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
    k_blockwise<DT, TILE, P2><<<grid, kEngThreads, kEngSmem, st>>>(map, M, K, q_row, s_row, q_colT, s_colT, status);
    return cudaGetLastError();
}

cudaError_t launch_blockwise(const void *x, int dt, int64_t M, int64_t K, int tile, uint8_t *q_row, float *s_row,
                             uint8_t *q_colT, float *s_colT, int32_t *status, cudaStream_t st)
{
    if (dt == BF16)
        return tile == 0 ? bw_t<BF16, 0, false>(x, M, K, q_row, s_row, q_colT, s_colT, status, st)
                         : bw_t<BF16, 1, false>(x, M, K, q_row, s_row, q_colT, s_colT, status, st);
    return tile == 0 ? bw_t<F32, 0, false>(x, M, K, q_row, s_row, q_colT, s_colT, status, st)
                     : bw_t<F32, 1, false>(x, M, K, q_row, s_row, q_colT, s_colT, status, st);
}

cudaError_t launch_blockwise_mx(const void *x, int dt, int64_t M, int64_t K, int tile, uint8_t *q_row,
                                uint8_t *e_row, uint8_t *q_colT, uint8_t *e_colT, int32_t *status, cudaStream_t st)
{
    if (dt == BF16)
        return tile == 0 ? bw_t<BF16, 0, true>(x, M, K, q_row, e_row, q_colT, e_colT, status, st)
                         : bw_t<BF16, 1, true>(x, M, K, q_row, e_row, q_colT, e_colT, status, st);
    return tile == 0 ? bw_t<F32, 0, true>(x, M, K, q_row, e_row, q_colT, e_colT, status, st)
                     : bw_t<F32, 1, true>(x, M, K, q_row, e_row, q_colT, e_colT, status, st);
}

}  // namespace qk
