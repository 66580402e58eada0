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
//  1x16 rowwise - a block spans 16/VEC lanes; stochastic rounding takes the
//                 words of the block's Philox block (16 elements) that cover
//                 the thread's chunk;
//  16x1 colwise - a block is the 8 rows of warps 2p and 2p+1: their column
//                 maxima meet in shared memory; each column's 8 values are
//                 encoded into one word of row nibbles (SR: half of the
//                 column block's Philox block), parked in the consumed stage
//                 and written as q_colT rows;
//  16x16        - the block maximum spans 2 warps x 16/VEC lanes; the
//                 transposed copy is the row codes nibble-transposed.
#include <cstring>

#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

// With 1x16 blocks the per-CTA encode table of k_nvfp4 holds 16
// interleaved copies (entry e, copy j at word 16 e + j) and lane l reads copy
// l % 16, so lanes that look up different entries meet in one bank at most in
// pairs (with one copy up to four entries share a bank).  16x16 lookups are
// uniform across the lanes of a block and keep one copy.
template <int BLK> constexpr int kTabCopies = BLK == 0 ? 16 : 1;

// Block scale code sb = E4M3(RN(RN(b * alpha_g) / 6)) (b = 0 -> 0x38, 1.0) of
// an FP32 block maximum with bits b.
QD uint32_t nv_sb_code(uint32_t b, float alpha_g)
{
    if (b == 0) return 0x38u;
    return e4m3_code(__fdiv_rn(__fmul_rn(__uint_as_float(b), alpha_g), 6.0f));
}

// The encode factor enc = alpha_g / f(sb) (0 when f(sb) = 0) depends only on
// the code: each CTA tabulates it for the 128 positive codes (entry 0x38 =
// alpha_g also serves b = 0).

// Codes of one row chunk (VEC elements, VEC/2 bytes) with scale factor enc;
// SR: the chunk's elements i0 .. (row-major, stream 0) are word (i0 % 16) / 4
// onward of Philox block offset + i0 / 16.
template <int DT, int RND>
QD uint32_t nv_row_codes(const uint4 &v, float enc, const PhiloxKeys &keys, uint64_t offset, int64_t i0)
{
    constexpr int VEC = In<DT>::VEC;
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; j++) y[j] = j < VEC ? elem<DT>(v, j < VEC ? j : 0) : 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; j += 2) mul2(y[j], y[j + 1], enc, enc);
    if (RND == 1) {
        const uint4 R = sr_bits_rk<0>(offset + (uint64_t)(i0 >> 4), keys);
        const int t = (int)((i0 >> 2) & 3);
        if (VEC == 4) return cvt_rs_fp4x4(y[0], y[1], y[2], y[3], word(R, t));
        return cvt_rs_fp4x8(y, word(R, t), word(R, t + 1));
    }
    return cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
}

// FP32 inputs (BF16 inputs take k_nvfp4_bf16).
template <int DT, int BLK, int RND>
__global__ void __launch_bounds__(kEngThreads, 1) k_nvfp4(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                          const float *__restrict__ amax,
                                                          const __grid_constant__ PhiloxKeys keys, uint64_t offset,
                                                          uint8_t *__restrict__ q_row, uint8_t *__restrict__ sb_row,
                                                          uint8_t *__restrict__ q_colT, uint8_t *__restrict__ sb_colT,
                                                          float *__restrict__ s_global, int32_t *status)
{
    static_assert(DT == F32, "BF16 inputs take k_nvfp4_bf16");
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, LPB = 16 / VEC, TCP = kTabCopies<BLK>;
    __shared__ float enc_tab[128 * TCP];
    __shared__ uint4 part[kEngWarps][32];        // 1x16: per-warp column maxima over 8 rows
    __shared__ __align__(8) uint8_t sSB[8][TC];   // 1x16: columnwise block scales of a tile
    __shared__ uint32_t bred[kEngWarps][TC / 16];   // 16x16: half-block maxima

    griddep_wait();   // the amax pass ahead of this kernel is complete
    const float A = *amax;
    const float alpha_g = alpha_from_amax(2688.0f, A);
    if (threadIdx.x < 128) {
        const float sv = e4m3_value(threadIdx.x);
        const float ev = sv == 0.0f ? 0.0f : __fdiv_rn(alpha_g, sv);
#pragma unroll
        for (int j = 0; j < TCP; j++) enc_tab[threadIdx.x * TCP + j] = ev;
    }   // visible after the engine's first barrier
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *s_global = __fdiv_rn(1.0f, alpha_g);
        flag_nonfinite(status, __float_as_uint(A) & 0x7FFFFFFFu);
    }
    if (M == 0 || K == 0) return;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;
    const float *encT = enc_tab + (lane & (TCP - 1));   // this lane's copy: entry e at encT[e * TCP]

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
            if (q_row != nullptr) {
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    uint32_t bb[2] = {absmax_bits<DT>(v[j]), absmax_bits<DT>(v[j + 1])};
                    group_max2<DT, LPB>(bb[0], bb[1]);
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int64_t m = m0 + j + h;
                        const uint32_t sb = nv_sb_code(bb[h], alpha_g);
                        const uint32_t code = nv_row_codes<DT, RND>(v[j + h], encT[(sb & 0x7Fu) * TCP], keys, offset, m * K + k);
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
                const uint32_t sb = nv_sb_code(b, alpha_g);
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
                    // rows m0 .. m0 + 7 of column k + c, stream 1: half (m0 % 16) / 8 of
                    // Philox block (m0 / 16) * K + k + c (words 0-1 or 2-3)
                    const uint4 R = sr_bits_rk<1>(offset + (uint64_t)((m0 >> 4) * K + k + c), keys);
                    const bool hi8 = (m0 & 8) != 0;
                    colw[c] = cvt_rs_fp4x8(y, hi8 ? R.z : R.x, hi8 ? R.w : R.y);
                } else {
                    colw[c] = cvt_fp4x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
                }
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
            const uint32_t sb = nv_sb_code(b, alpha_g);
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
                const uint32_t code = nv_row_codes<DT, RND>(v[j], enc, keys, offset, m * K + k);
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
    const PhiloxKeys keys = philox_keys(seed);
    return launch_k(after_amax, k_nvfp4<DT, BLK, RND>, dim3(grid), dim3(kEngThreads), kEngSmem, st, map, M, K, amax,
                    keys, offset, q_row, sb_row, q_colT, sb_colT, s_global, status);
}

cudaError_t launch_nvfp4(const void *x, int dt, int64_t M, int64_t K, int blk, int rnd, uint64_t seed,
                         uint64_t offset, const float *amax, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT,
                         uint8_t *sb_colT, float *s_global, int32_t *status, cudaStream_t st, bool after_amax)
{
#define NV_ARGS x, M, K, amax, seed, offset, q_row, sb_row, q_colT, sb_colT, s_global, status, st, after_amax
    if (dt == BF16)
        return launch_nvfp4_bf16(x, M, K, blk, rnd, seed, offset, amax, q_row, sb_row, q_colT, sb_colT, s_global,
                                 status, st, after_amax);
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
                                                              int64_t K, uint32_t sign_mask, float *amax,
                                                              const __grid_constant__ PhiloxKeys keys,
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
            const uint32_t sa = nv_sb_code(ba, alpha_g), sbb = nv_sb_code(bb, alpha_g);
            const float ea = enc_tab[sa & 0x7Fu], eb = enc_tab[sbb & 0x7Fu];
            const int c0 = q * CPT + 2 * p;   // tile column of a
            sSB[g][c0] = (uint8_t)sa;
            sSB[g][c0 + 1] = (uint8_t)sbb;
            const bool live = mb + 16 * g < M;
            post_nonfinite(status, live && (kb + c0 < K) ? nonfinite(ba) | nonfinite(bb) : 0u);
#pragma unroll
            for (int i = 0; i < 16; i++) mul2(a[i], b[i], ea, eb);
            // rows m .. m + 15 of columns kb + c0, kb + c0 + 1, stream 1: Philox blocks
            // (m / 16) * K + column, words 0-1 for rows 0-7 and 2-3 for rows 8-15
            uint4 Ra = make_uint4(0u, 0u, 0u, 0u), Rb = Ra;
            if constexpr (RND == 1) {
                const uint64_t gb = offset + (uint64_t)(((mb + 16 * g) >> 4) * K + kb + c0);
                Ra = sr_bits_rk<1>(gb, keys);
                Rb = sr_bits_rk<1>(gb + 1, keys);
            }
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const float *pa = a + 8 * hh, *pb = b + 8 * hh;
                if constexpr (RND == 1) {
                    code[2 * p][hh] = cvt_rs_fp4x8(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], pa[6], pa[7],
                                                   hh ? Ra.z : Ra.x, hh ? Ra.w : Ra.y);
                    code[2 * p + 1][hh] = cvt_rs_fp4x8(pb[0], pb[1], pb[2], pb[3], pb[4], pb[5], pb[6], pb[7],
                                                       hh ? Rb.z : Rb.x, hh ? Rb.w : Rb.y);
                } else {
                    code[2 * p][hh] = cvt_fp4x8(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], pa[6], pa[7]);
                    code[2 * p + 1][hh] = cvt_fp4x8(pb[0], pb[1], pb[2], pb[3], pb[4], pb[5], pb[6], pb[7]);
                }
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
    const PhiloxKeys keys = philox_keys(seed);
    return launch_k(pdl, k_nvfp4_rht<DT, RND, PASS>, dim3(grid), dim3(kEngThreads), kEngSmem, st, map, M, K, mask, amax,
                    keys, offset, q_colT, sb_colT, PASS == 0 ? amax_x : s_global, status);
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
