// MXFP8 quantize, rowwise 1x32 and columnwise 32x1, in one pass (a4, a5).
//
// "Mixed-precision training: fp16 to fp8", section "MXFP8": every 32
// elements share one E8M0 scale (an FP32 exponent field), value = element x
// scale; section "MXFP8 recipe": rowwise and columnwise copies differ only in
// the quantization direction, neither is transposed in memory.
// Scale code = clamp(floor(log2 b) - emax + 127, 0, 254), emax = 8 (E4M3) or
// 15 (E5M2), b = 0 -> 127; q = RTNE-saturate(x * 2^(127 - code)).
//
// On the tile engine with two 256-thread CTAs per SM (64 x TC tiles in
// shared memory, TileCfg<64, 256>; one CTA's barrier and latency-bound phases
// overlap the other's work): thread (warp w, lane l) holds rows 8w..8w+7 x
// one 16-byte column chunk in registers.
//  row pass - a 1x32 block spans 32/VEC lanes (xor-shuffle max);
//  col pass - each warp reduces its 8 rows per column in registers; the four
//             warps of a 32-row block meet in shared memory (one barrier);
//             the column-scaled codes of the same registers are stored in the
//             [M, K] layout.
// Both outputs leave straight from registers, 256 contiguous bytes per warp
// and row.
#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

using MxCfg = TileCfg<64, 256, 3>;

template <int DT, int FMT>
__global__ void __launch_bounds__(MxCfg::kThreads, 2) k_mxfp8(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                              uint8_t *__restrict__ q_row, uint8_t *__restrict__ e_row,
                                                              uint8_t *__restrict__ q_col, uint8_t *__restrict__ e_col,
                                                              int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, CW = VEC / 4, LPB = 32 / VEC;
    __shared__ uint4 part[MxCfg::kThreads / 32][32];   // per-warp column maxima over 8 rows (packed like the input)
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t tiles_m = (M + MxCfg::kRows - 1) / MxCfg::kRows, tiles_k = (K + TC - 1) / TC;

    run_tiles<MxCfg>(&tmap, tiles_m, tiles_k, TC, false, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * MxCfg::kRows, kb = tk * TC;
        const int64_t k = kb + lane * VEC, m0 = mb + 8 * warp;
        const bool kok = k < K;
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = lds16(st + (8 * warp + j) * kRowBytes + lane * 16);

        if (q_col != nullptr) {   // column maxima of this warp's 8 rows, before the row pass
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
        uint32_t nf = 0;   // non-finite block maxima seen by this thread
        if (DT == BF16 && q_row != nullptr) {
            // A block is 4 lanes.  The 8 row maxima, two BF16 magnitudes per
            // word, are halved across the group twice (3 shuffles): lane L keeps
            // rows 4*(L>>1 & 1) + 2*(L & 1) and the next, computes their codes
            // once, and the inverse scales go back by index shuffles.
            const int nrows = !kok ? 0 : (m0 + 8 <= M ? 8 : (m0 < M ? (int)(M - m0) : 0));
            uint32_t P[4];
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const uint4 &a = v[2 * p], &b = v[2 * p + 1];
                const uint32_t ma = hmax_abs2(hmax_abs2(a.x, a.y), hmax_abs2(a.z, a.w));
                const uint32_t mb = hmax_abs2(hmax_abs2(b.x, b.y), hmax_abs2(b.z, b.w));
                P[p] = hmax_abs2(__byte_perm(ma, mb, 0x5410), __byte_perm(ma, mb, 0x7632));   // row 2p low, 2p+1 high
            }
            const bool b1 = lane & 2, b0 = lane & 1;
            uint32_t k0 = b1 ? P[2] : P[0], k1 = b1 ? P[3] : P[1];          // rows 4*b1 .. 4*b1+3
            const uint32_t s0 = b1 ? P[0] : P[2], s1 = b1 ? P[1] : P[3];
            k0 = hmax_abs2(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, 2));
            k1 = hmax_abs2(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, 2));
            uint32_t kw = b0 ? k1 : k0;                                        // rows 4*b1+2*b0, +1
            kw = hmax_abs2(kw, __shfl_xor_sync(0xFFFFFFFFu, b0 ? k0 : k1, 1));
            const int r = 4 * (b1 ? 1 : 0) + 2 * (b0 ? 1 : 0);
            const uint32_t blo = (kw << 16) & 0x7FFF0000u, bhi = kw & 0x7FFF0000u;   // rows r, r + 1
            const uint32_t clo = mx_code<FMT>(blo), chi = mx_code<FMT>(bhi);
            const float ilo = mx_inv_scale(clo), ihi = mx_inv_scale(chi);
            if (r < nrows) {
                e_row[(m0 + r) * (K / 32) + k / 32] = (uint8_t)clo;
                nf |= nonfinite(blo);
            }
            if (r + 1 < nrows) {
                e_row[(m0 + r + 1) * (K / 32) + k / 32] = (uint8_t)chi;
                nf |= nonfinite(bhi);
            }
            uint8_t *qr = q_row + m0 * K + k;
            const int gb = lane & ~3;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                // row j lives in lane gb + 2*(j >> 2) + ((j >> 1) & 1), low half for even j
                const float inv = __shfl_sync(0xFFFFFFFFu, (j & 1) ? ihi : ilo, gb + 2 * (j >> 2) + ((j >> 1) & 1));
                uint32_t o[CW];
                chunk_fp8<DT, FMT>(v[j], inv, o);
                if (j < nrows) stg8(qr + j * K, o[0], o[CW - 1]);
            }
        } else if (q_row != nullptr) {
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t bb[2] = {absmax_bits<DT>(v[j]), absmax_bits<DT>(v[j + 1])};
                group_max2<DT, LPB>(bb[0], bb[1]);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const uint32_t code = mx_code<FMT>(bb[h]);
                    uint32_t o[CW];
                    chunk_fp8<DT, FMT>(v[j + h], mx_inv_scale(code), o);
                    const bool ok = m0 + j + h < M && kok;
                    if (ok) {
                        uint8_t *dst = q_row + (m0 + j + h) * K + k;
                        if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                        else stg4(dst, o[0]);
                    }
                    if (ok && lane % LPB == 0) e_row[(m0 + j + h) * (K / 32) + k / 32] = (uint8_t)code;
                    nf |= ok ? nonfinite(bb[h]) : 0u;
                }
            }
        }
        if (q_col == nullptr) {
            post_nonfinite(status, nf);
            return;
        }
        __syncthreads();   // the four warps of each 32-row block have posted their maxima
        // ---- 32x1 blocks: the block of this warp is rows 32*(warp/4) .. +31
        const int w0 = warp & ~3;
        uint4 cm = part[w0][lane];
#pragma unroll
        for (int q = 1; q < 4; q++) {
            const uint4 o4 = part[w0 + q][lane];
            cm.x = colmax_word<DT>(cm.x, o4.x);
            cm.y = colmax_word<DT>(cm.y, o4.y);
            cm.z = colmax_word<DT>(cm.z, o4.z);
            cm.w = colmax_word<DT>(cm.w, o4.w);
        }
        float inv[VEC];
        uint32_t codes[VEC];
#pragma unroll
        for (int c = 0; c < VEC; c++) {
            const uint32_t b = colmax_bits<DT>(cm, c);
            codes[c] = mx_code<FMT>(b);
            inv[c] = mx_inv_scale(codes[c]);
            nf |= ((warp & 3) == 0 && kok && m0 < M) ? nonfinite(b) : 0u;
        }
        post_nonfinite(status, nf);
        if ((warp & 3) == 0 && kok && m0 < M) {
            uint32_t sw[CW];
#pragma unroll
            for (int q = 0; q < CW; q++)
                sw[q] = codes[4 * q] | (codes[4 * q + 1] << 8) | (codes[4 * q + 2] << 16) | (codes[4 * q + 3] << 24);
            uint8_t *dst = e_col + (m0 / 32) * K + k;
            if (CW == 2) stg8(dst, sw[0], sw[CW - 1]);
            else stg4(dst, sw[0]);
        }
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float f[VEC];
#pragma unroll
            for (int c = 0; c < VEC; c++) f[c] = elem<DT>(v[j], c);
#pragma unroll
            for (int c = 0; c < VEC; c += 2) mul2(f[c], f[c + 1], inv[c], inv[c + 1]);
            uint32_t o[CW];
#pragma unroll
            for (int q = 0; q < CW; q++) o[q] = cvt_fp8x4<FMT>(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
            if (m0 + j < M && kok) {
                uint8_t *dst = q_col + (m0 + j) * K + k;
                if (CW == 2) stg8(dst, o[0], o[CW - 1]);
                else stg4(dst, o[0]);
            }
        }
    });
}

// ---------------------------------------------------------------------------
// Rowwise MXFP8 codes -> columnwise MXFP8 codes ("Mixed-precision training:
// fp16 to fp8", section "FP8 communication", EP: only the rowwise copy
// travels; a dequantize and re-quantize in the other direction makes the
// columnwise copy).  x_hat = code * 2^(e_row - 127) (one exact FP32
// product), then 32x1 blocks of x_hat as in k_mxfp8.  On the tile engine over
// the code matrix (two 256-thread CTAs per SM, TileCfg<64, 256>): a stage is
// 64 rows x 512 codes, thread (warp w, lane l) covers rows 8w..8w+7 x codes
// 16l..16l+15; x_hat is formed twice from the
// stage (once for the column maxima, which meet across the 4 warps of a
// 32-row block in shared memory, once for the codes) instead of being held
// in registers.
// ---------------------------------------------------------------------------
template <int FMT> QD void dq16(const uint4 &c, float f, float *x)
{
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const uint32_t wd = word(c, q);
        const float2 a = fp8x2_to_f32<FMT>(wd & 0xFFFFu), b = fp8x2_to_f32<FMT>(wd >> 16);
        x[4 * q] = a.x;
        x[4 * q + 1] = a.y;
        x[4 * q + 2] = b.x;
        x[4 * q + 3] = b.y;
    }
#pragma unroll
    for (int i = 0; i < 16; i += 2) mul2(x[i], x[i + 1], f, f);
}

template <int FMT>
__global__ void __launch_bounds__(MxCfg::kThreads, 2) k_mxfp8_requant(const __grid_constant__ CUtensorMap tmap, int64_t M,
                                                                      int64_t K, const uint8_t *__restrict__ e_row,
                                                                      uint8_t *__restrict__ q_col, uint8_t *__restrict__ e_col,
                                                                      int32_t *status)
{
    constexpr int TC = 512;   // codes per tile row
    constexpr int kTileRowsE = MxCfg::kRows;
    __shared__ uint32_t part[MxCfg::kThreads / 32][16][32];   // per warp, column, lane: |x_hat| maxima over 8 rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;

    // The row scales of this thread's 8 rows are loaded one tile ahead (the
    // CTA's next tile is t + gridDim.x), so that their latency hides behind a
    // whole tile instead of stalling the start of each one.
    uint32_t epre[8];
    auto load_e = [&](int64_t t) {
        const int64_t tm = t / tiles_k, tk = t - tm * tiles_k;
        const int64_t k = tk * TC + lane * 16, m0 = tm * kTileRowsE + 8 * warp;
        const bool ok = t < tiles_m * tiles_k && k < K;
#pragma unroll
        for (int j = 0; j < 8; j++) epre[j] = (ok && m0 + j < M) ? e_row[(m0 + j) * (K / 32) + k / 32] : 0u;
    };
    load_e(blockIdx.x);

    // the tensor map counts 2-byte elements: a tile is 256 of them per row
    run_tiles<MxCfg>(&tmap, tiles_m, tiles_k, TC / 2, false, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        const int64_t k = kb + lane * 16, m0 = mb + 8 * warp;
        const bool kok = k < K;
        const uint8_t *srow = st + (8 * warp) * kRowBytes + lane * 16;
        float fr[8];   // 2^(e_row - 127) of each row's 1x32 block (code 255 -> NaN)
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint32_t er = epre[j];
            fr[j] = er == 255u ? __uint_as_float(0x7FC00000u) : er == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(er << 23);
        }
        load_e(tm * tiles_k + tk + gridDim.x);
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; i++) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float x[16];
            dq16<FMT>(lds16(srow + j * kRowBytes), fr[j], x);
#pragma unroll
            for (int i = 0; i < 16; i++) acc[i] = fmax_abs(acc[i], x[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; i++) part[warp][i][lane] = __float_as_uint(acc[i]) & 0x7FFFFFFFu;
        // the four warps of this 32-row block have posted their maxima (named
        // barrier 1..4 per block; the engine's CTA barrier after each tile
        // orders the reads here before the next tile's writes).  Warp wq of
        // the block reduces columns 4wq..4wq+3 of each lane's 16, writes their
        // scale codes and leaves their factors 2^(127 - code) in its own
        // slots of those columns (read by no other warp before the second
        // barrier); then every warp reads the 16 factors.
        asm volatile("bar.sync %0, 128;" ::"r"(1 + (warp >> 2)) : "memory");
        const int w0 = warp & ~3, wq = warp & 3;
        const int64_t mblk = mb + 32 * (warp >> 2);
        uint32_t cw = 0, nf = 0;
        float invq[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int i = 4 * wq + j;
            const uint32_t b = max(max(part[w0][i][lane], part[w0 + 1][i][lane]), max(part[w0 + 2][i][lane], part[w0 + 3][i][lane]));
            const uint32_t c = mx_code<FMT>(b);
            cw |= c << (8 * j);
            invq[j] = mx_inv_scale(c);
            nf |= nonfinite(b);
        }
#pragma unroll
        for (int j = 0; j < 4; j++) part[warp][4 * wq + j][lane] = __float_as_uint(invq[j]);
        if (kok && mblk < M) {
            stg4(e_col + (mblk / 32) * K + k + 4 * wq, cw);
            post_nonfinite(status, nf);
        }
        asm volatile("bar.sync %0, 128;" ::"r"(1 + (warp >> 2)) : "memory");
        float inv[16];
#pragma unroll
        for (int i = 0; i < 16; i++) inv[i] = __uint_as_float(part[w0 + (i >> 2)][i][lane]);
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float x[16];
            dq16<FMT>(lds16(srow + j * kRowBytes), fr[j], x);
#pragma unroll
            for (int i = 0; i < 16; i += 2) mul2(x[i], x[i + 1], inv[i], inv[i + 1]);
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; q++) o[q] = cvt_fp8x4<FMT>(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            if (m0 + j < M && kok) stg16(q_col + (m0 + j) * K + k, make_uint4(o[0], o[1], o[2], o[3]));
        }
    });
}

template <int FMT>
static cudaError_t mx_requant_t(const uint8_t *q_row, const uint8_t *e_row, int64_t M, int64_t K, uint8_t *q_col,
                                uint8_t *e_col, int32_t *status, cudaStream_t st)
{
    alignas(64) CUtensorMap map;
    cudaError_t e = make_tile_map(&map, q_row, U8, M, K, MxCfg::kRows);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t ea = engine_smem_ready<k_mxfp8_requant<FMT>>(MxCfg::kSmem, true);
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + MxCfg::kRows - 1) / MxCfg::kRows) * ((K + 511) / 512);
    const int64_t slots = 2 * (int64_t)sm_count();   // two CTAs per SM
    const int grid = (int)(tiles < slots ? tiles : slots);
    k_mxfp8_requant<FMT><<<grid, MxCfg::kThreads, MxCfg::kSmem, st>>>(map, M, K, e_row, q_col, e_col, status);
    return cudaGetLastError();
}

cudaError_t launch_mxfp8_requant_col(const uint8_t *q_row, const uint8_t *e_row, int64_t M, int64_t K, int fmt,
                                     uint8_t *q_col, uint8_t *e_col, int32_t *status, cudaStream_t st)
{
    return fmt == E4M3 ? mx_requant_t<E4M3>(q_row, e_row, M, K, q_col, e_col, status, st)
                       : mx_requant_t<E5M2>(q_row, e_row, M, K, q_col, e_col, status, st);
}

template <int DT, int FMT>
static cudaError_t mx_t(const void *x, int64_t M, int64_t K, uint8_t *q_row, uint8_t *e_row, uint8_t *q_col,
                        uint8_t *e_col, int32_t *status, cudaStream_t st)
{
    constexpr int TC = 32 * In<DT>::VEC;
    alignas(64) CUtensorMap map;
    cudaError_t e = make_tile_map(&map, x, DT, M, K, MxCfg::kRows);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t ea = engine_smem_ready<k_mxfp8<DT, FMT>>(MxCfg::kSmem, true);
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + MxCfg::kRows - 1) / MxCfg::kRows) * ((K + TC - 1) / TC);
    const int64_t slots = 2 * (int64_t)sm_count();   // two CTAs per SM
    const int grid = (int)(tiles < slots ? tiles : slots);
    k_mxfp8<DT, FMT><<<grid, MxCfg::kThreads, MxCfg::kSmem, st>>>(map, M, K, q_row, e_row, q_col, e_col, status);
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
