/*
 * q.h -- C ABI of the GB300 (sm_103a) tensor quantizers.
 *
 * The operations turn a BF16 or FP32 tensor into low-precision codes plus
 * scales, and back, for FP8 / FP4 mixed-precision training.  Sources (cited
 * by tag in each entry):
 *   [MP] "Mixed-precision training: fp16 to fp8"
 *        (garden.houmin.site/infra/mixed-precision-fp8)
 *   [CS] "FP8 Current Scaling: quantization, scaling and precision bounds"
 *        (notes.kuangjux.top/Foundations/08_Quantization/fp8-current-scaling)
 *   [LP] "From BF16 to FP8/FP4: low-precision and mixed-precision LLM
 *        pretraining" (r00kie-liu.github.io/2026/07/23/
 *        low-precision-mixed-precision-pretraining)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors are row-major and contiguous.  x is [M, K]: M rows (tokens or
 * output features), K contiguous columns.  "Rowwise" quantizes blocks that
 * run along K; "columnwise" quantizes blocks that run along M.  Columnwise
 * outputs of current scaling, blockwise and NVFP4 are stored transposed,
 * [K, M] (the operand of the wgrad GEMM X^T, [MP] "Per-tensor Current
 * Scaling" and "Blockwise scaling" flows); the MXFP8 columnwise output stays
 * in the [M, K] layout ([MP] "MXFP8 recipe").
 *
 * Ownership: every pointer is caller-owned DEVICE memory (except where a
 * parameter says otherwise); the library never allocates, never frees and
 * keeps no per-call state.  Each call enqueues its kernels on `stream`
 * (NULL = the legacy default stream) and returns without synchronizing.
 * Outputs must not overlap the inputs or each other.  Calls share no device
 * state, so calls on different streams (or devices) may run concurrently;
 * the caller orders a call after the producer of its inputs.
 *
 * Alignment: x, y and every code buffer must be 16-byte aligned; FP32 scale
 * buffers 4-byte aligned.  The byte-scale buffers of columnwise copies
 * (e8m0_col of q_mxfp8 and q_mxfp8_requant_col, sb_colT of the NVFP4 calls,
 * e8m0 of dq_mxfp8 with Q_COL) are written or read in 8- or 16-byte pieces
 * and must be 16-byte aligned; the E8M0 buffers of q_blockwise_mx 4-byte
 * aligned; other byte-scale buffers (e8m0_row, sb_row, sb of dq_nvfp4) have
 * no alignment rule.  A violation returns Q_ERR_ALIGN before any launch.
 *
 * Errors: argument problems are detected on the host, before any launch,
 * and returned as a q_status (nothing is enqueued).  A failed launch returns
 * Q_ERR_CUDA.  q_last_error() gives a message for the calling thread's last
 * failure.  Conditions found on the device (non-finite input) are ORed into
 * the optional device word *status (may be NULL); the caller zeroes it.
 *
 * Empty tensors (M == 0 or K == 0) are valid: amax is 0, scales are 1, no
 * code is written and the code / block-scale buffers may be NULL.
 */
#ifndef Q_H_
#define Q_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t). */
typedef struct CUstream_st *q_stream_t;

typedef enum {
    Q_OK = 0,
    Q_ERR_ARG = 1,     /* NULL where a buffer is required, bad enum, nothing requested */
    Q_ERR_SHAPE = 2,   /* negative size, M*K >= 2^62, or a dimension not a multiple of the block */
    Q_ERR_ALIGN = 3,   /* a pointer violates the alignment rule above */
    Q_ERR_DTYPE = 4,   /* unsupported input / output dtype */
    Q_ERR_CUDA = 5     /* a CUDA launch failed; see q_last_error() */
} q_status;

typedef enum { Q_BF16 = 0, Q_F32 = 1 } q_dtype;
typedef enum { Q_E4M3 = 0, Q_E5M2 = 1 } q_fp8;
typedef enum { Q_T1x128 = 0, Q_T128x128 = 1 } q_tile;
typedef enum { Q_B1x16 = 0, Q_B16x16 = 1 } q_nvblk;
typedef enum { Q_RN = 0, Q_SR = 1 } q_round;
typedef enum { Q_ROW = 0, Q_COL = 1 } q_dir;
/* Whether the per-tensor amax is computed by the call (Q_AMAX_COMPUTE, the
 * value is written to *amax) or given by the caller in *amax on the device
 * (Q_AMAX_GIVEN), e.g. after a MAX all-reduce over the shards of a tensor
 * ([CS] "Cost and multi-GPU use": compute amax, synchronize amax, then
 * scale + cast). */
typedef enum { Q_AMAX_COMPUTE = 0, Q_AMAX_GIVEN = 1 } q_amax_mode;
/* How delayed scaling reduces its amax window: the largest entry, or the
 * latest one. */
typedef enum { Q_HIST_MAX = 0, Q_HIST_MOST_RECENT = 1 } q_hist_algo;

/* Bits ORed into *status by the kernels. */
#define Q_ST_NONFINITE 1   /* an amax (tensor or block) was inf or NaN */
#define Q_ST_TIMEOUT 2     /* a kernel gave up waiting for its input tiles (outputs incomplete) */

/* Thread-local message describing this thread's last failed call ("" if none). */
const char *q_last_error(void);

/* Version of this ABI (incremented on incompatible change).  2: the
 * stochastic-rounding draws of the columnwise NVFP4 copies are numbered by
 * the element's position in x (see q_nvfp4), so results differ from 1.
 * 3: q_nvfp4_recipe takes a q_amax_mode.  4: NVFP4 stochastic rounding is
 * the conversion with random bits (16 draws per Philox block), so results
 * differ from 3. */
int q_abi_version(void);

/*
 * a1: tensor amax.  *amax = max_i |x_i| over the n elements of x
 * ([CS] "Current Scaling": a = max_i |x_i|; [MP] recipe 3 step 1).
 * x: n elements of dtype `in`.  amax: one float.  Any n >= 0.
 */
q_status q_amax(const void *x, q_dtype in, int64_t n, float *amax, int32_t *status,
                q_stream_t stream);

/*
 * a1-a3: per-tensor current scaling ([CS] "Current Scaling"; [MP] recipe 3,
 * "Per-tensor Current Scaling" flow).
 *   amax  = max|x| (or given), alpha = Fmax / amax (Fmax 448 for E4M3,
 *   57344 for E5M2), s = 1 / alpha, q = saturate(RTNE(alpha * x)).
 *   amax = 0 gives alpha = s = 1; an alpha that overflows is FLT_MAX.
 * Reads x twice when the amax is computed (once for the amax, once for the
 * cast); the cast pass walks the tensor backwards so that the part still in
 * L2 from the first pass is read first.
 *   q_row  [M, K] codes or NULL;  q_colT [K, M] codes (the same codes,
 *   transposed) or NULL; at least one is required.
 *   amax   one float: written (Q_AMAX_COMPUTE) or read (Q_AMAX_GIVEN).
 *   scale  one float: s.
 * Shapes: any M, K >= 0 for q_row alone; q_colT needs M % 16 == 0 and
 * K % 16 == 0.
 */
q_status q_current_scaling(const void *x, q_dtype in, int64_t M, int64_t K, q_fp8 fmt,
                           uint8_t *q_row, uint8_t *q_colT,
                           float *amax, q_amax_mode amax_mode, float *scale,
                           int32_t *status, q_stream_t stream);

/*
 * Per-tensor delayed scaling ([MP] "Per-tensor delayed scaling"; window
 * settings as quoted on [LP] section 4.3: length 1024, reduction max).  Step
 * t quantizes x with a scale predicted from the amaxes of earlier steps and
 * records its own amax in the same read of x; q_delayed_scale_update then
 * derives the scale of step t+1 from the window.  Per step:
 *   q_delayed_scaling(x, ..., ds, &hist[t % N], scale_t, ...);
 *   q_delayed_scale_update(hist, N, t % N, algo, fmt, ds, ...);
 * ds is the device pair [alpha, s] (initially [1, 1], which is also what an
 * all-zero window gives).  The caller owns hist[N] (FP32, zero-initialized)
 * and ds, and keeps t.
 *
 * q_delayed_scaling: q = saturate(RTNE(alpha * x)) with alpha = ds[0];
 *   q_row / q_colT as in q_current_scaling (same shape rules);
 *   amax_out  one float, written: max|x| (this step's window entry);
 *   scale     one float, written: ds[1], the s that decodes these codes.
 * An empty tensor writes amax_out = 0 and scale = ds[1].  A non-finite x or
 * alpha is reported in *status.
 */
q_status q_delayed_scaling(const void *x, q_dtype in, int64_t M, int64_t K, q_fp8 fmt,
                           uint8_t *q_row, uint8_t *q_colT, const float *ds, float *amax_out, float *scale,
                           int32_t *status, q_stream_t stream);

/*
 * q_delayed_scale_update: ds = [alpha, s] from the window hist[0..N) (N >= 1,
 * slot pos < N holds the latest amax).  Q_HIST_MAX: A = the largest |entry|;
 * Q_HIST_MOST_RECENT: A = |hist[pos]|.  alpha = Fmax / A (A = 0 gives 1; an
 * alpha that overflows is FLT_MAX), s = 1 / alpha.  One CTA; reads N floats.
 */
q_status q_delayed_scale_update(const float *hist, int64_t N, int64_t pos, q_hist_algo algo, q_fp8 fmt,
                                float *ds, q_stream_t stream);

/*
 * a4/a5: MXFP8 ([MP] "MXFP8" and recipe 5): 32 elements share one E8M0
 * scale (an FP32 exponent field, 2^(code-127)).  Per block with
 * b = max|x|: code = clamp(floor(log2 b) - emax + 127, 0, 254), emax = 8 for
 * E4M3 and 15 for E5M2 (b = 0 gives 127); q = saturate(RTNE(x * 2^(127-code))).
 *   q_row    [M, K] codes, 1x32 blocks along K;  e8m0_row [M, K/32]
 *   q_col    [M, K] codes, 32x1 blocks along M;  e8m0_col [M/32, K]
 * Either direction may be NULL (both buffers of it), not both.
 * Shapes: K % 32 == 0; with q_col also M % 32 == 0.
 */
q_status q_mxfp8(const void *x, q_dtype in, int64_t M, int64_t K, q_fp8 fmt,
                 uint8_t *q_row, uint8_t *e8m0_row, uint8_t *q_col, uint8_t *e8m0_col,
                 int32_t *status, q_stream_t stream);

/*
 * MXFP8 rowwise codes -> columnwise codes ([MP] "FP8 communication", EP:
 * only the rowwise FP8 copy crosses the expert-parallel all-to-all, and a
 * de-quantize + re-quantize kernel in the other direction gives the
 * columnwise copy for the backward pass).  x_hat = q_row * 2^(e_row - 127)
 * in FP32, then q_col / e8m0_col of x_hat exactly as q_mxfp8 computes them
 * (32x1 blocks along M).  Power-of-two block scales make the result close
 * to direct columnwise quantization of the original tensor (equal wherever
 * the rowwise codes lost no bits that the columnwise codes keep).
 *   q_row [M, K] codes, e8m0_row [M, K/32] (as written by q_mxfp8);
 *   q_col [M, K] codes, e8m0_col [M/32, K] (written).  fmt is the format of
 *   both.  e8m0 code 255 (NaN) decodes to NaN and is reported in *status.
 * Shapes: M % 32 == 0, K % 32 == 0.  Reads the codes once (TMA tiles).
 */
q_status q_mxfp8_requant_col(const uint8_t *q_row, const uint8_t *e8m0_row, int64_t M, int64_t K, q_fp8 fmt,
                             uint8_t *q_col, uint8_t *e8m0_col, int32_t *status, q_stream_t stream);

/*
 * a6/a7: DeepSeek-V3-like blockwise FP8 ([MP] recipe 4 and "Blockwise
 * scaling"): E4M3 only, FP32 scale per tile, formed like the per-tensor
 * scale on the tile: alpha_b = 448 / b, s_b = 1 / alpha_b.
 *   tile Q_T1x128 (activations, gradients):
 *     q_row [M, K], s_row [M, K/128];  q_colT [K, M], s_colT [K, M/128]
 *     (128x1 blocks along M of each column).  K % 128 == 0; with q_colT
 *     also M % 128 == 0.
 *   tile Q_T128x128 (weights):
 *     q_row [M, K], s_row [M/128, K/128]; q_colT [K, M] = the same codes
 *     transposed, s_colT [K/128, M/128].  M % 128 == 0 and K % 128 == 0.
 * Either direction may be NULL, not both.
 */
q_status q_blockwise(const void *x, q_dtype in, int64_t M, int64_t K, q_tile tile,
                     uint8_t *q_row, float *s_row, uint8_t *q_colT, float *s_colT,
                     int32_t *status, q_stream_t stream);

/*
 * R5: blockwise tiles held as MXFP8 ([MP] "Blockwise scaling": on Blackwell
 * the blockwise recipe is emulated with MXFP8, a 1x128 tile being 4 MXFP8
 * blocks that share one scale factor, a 128x128 tile 128 x 4 of them).  E4M3.
 * The tile scale is b/448 rounded up to a power of two (the tile maximum
 * never saturates), code = 127 + n for the smallest n with b <= 448 * 2^n,
 * clamped to [0, 254] (b = 0 -> 127; inf / NaN -> 247); it is stored once
 * per 32 elements along the quantization direction.  Elements
 * q = Q(x * 2^(127 - code)), as in MXFP8.
 *   tile Q_T1x128:   q_row [M, K], e8m0_row [M, K/32]; q_colT [K, M],
 *                    e8m0_colT [K, M/32] (128x1 blocks along M).
 *   tile Q_T128x128: q_row [M, K], e8m0_row [M, K/32] (a tile's 128 rows
 *                    share its code); q_colT [K, M] = the same codes
 *                    transposed, e8m0_colT [K, M/32].
 * Both copies dequantize with dq_mxfp8(..., Q_ROW, ...), the transposed copy
 * as the [K, M] matrix it is.  Shapes as q_blockwise; code buffers 16-byte
 * aligned, scale buffers 4-byte aligned.  Either direction may be NULL, not
 * both.  Non-finite tile maxima set Q_ST_NONFINITE in *status.
 */
q_status q_blockwise_mx(const void *x, q_dtype in, int64_t M, int64_t K, q_tile tile,
                        uint8_t *q_row, uint8_t *e8m0_row, uint8_t *q_colT, uint8_t *e8m0_colT,
                        int32_t *status, q_stream_t stream);

/*
 * a8-a11: NVFP4 ([MP] "NVFP4" and recipe 6; [LP] 2.4 items 1, 4, 5):
 * E2M1 codes packed two per byte (element 2j in bits 3-0, 2j+1 in bits 7-4),
 * one E4M3 scale per block, one FP32 tensor scale.
 *   alpha_g = 2688 / amax (= 6 * 448 / amax; amax = 0 -> 1), s_global = 1/alpha_g
 *   per block: sb = E4M3(RTNE((b * alpha_g) / 6)), b = 0 -> sb = 1.0;
 *              enc = alpha_g / sb (0 if sb == 0); q = E2M1(x * enc)
 *   rnd Q_RN: round to nearest even.  rnd Q_SR: stochastic rounding as the
 *   GB300's E2M1 conversion with random bits performs it.  The random bits
 *   come from Philox4x32-10 with key (seed lo, seed hi) and counter
 *   (g lo, g hi, stream, 0), g = offset + i / 16, where i is the draw index:
 *   stream 0 (q_row):         i = m*K + k;
 *   stream 1 (a 1x16 q_colT): i = ((m / 16)*K + k)*16 + m % 16.
 *   Output word (i % 16) / 4 serves the four draw indices 4t .. 4t + 3; its
 *   bytes 0 and 2 form a 16-bit draw U0 (byte 2 high), bytes 1 and 3 a draw
 *   U1 (byte 3 high), and the four elements take U0, U0 bit-reversed, U1,
 *   U1 bit-reversed.  With T = floor(frac * 65536), frac the position of
 *   |x * enc| between its two neighbouring E2M1 values, an element rounds
 *   up iff T + R >= 65536 for its draw R.  The index depends on K but not
 *   on M: a row shard holding rows [r0, r0 + M) of a taller tensor
 *   (r0 % 16 == 0) that passes offset + r0*K/16 draws exactly what the
 *   unsharded call draws for those rows, in both copies ([MP] "FP8
 *   communication", TP).
 *   blk Q_B1x16 (activations, gradients):
 *     q_row [M, K/2], sb_row [M, K/16];  q_colT [K, M/2], sb_colT [K, M/16]
 *     (16x1 blocks along M of each column).
 *   blk Q_B16x16 (weights): one scale per 16x16 tile,
 *     q_row [M, K/2], sb_row [M/16, K/16]; q_colT [K, M/2] = the same codes
 *     transposed, sb_colT [K/16, M/16].
 *   amax      one float, written (Q_AMAX_COMPUTE) or read (Q_AMAX_GIVEN)
 *   s_global  one float, written.
 * Shapes: K % 16 == 0 and M % 16 == 0.  Either direction may be NULL, not
 * both.
 */
q_status q_nvfp4(const void *x, q_dtype in, int64_t M, int64_t K, q_nvblk blk, q_round rnd,
                 uint64_t seed, uint64_t offset,
                 uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT,
                 float *amax, q_amax_mode amax_mode, float *s_global,
                 int32_t *status, q_stream_t stream);

/*
 * NVFP4 columnwise copy of the random-Hadamard-transformed tensor, for the
 * inputs of the weight-gradient GEMM ([LP] section 2.4, recipe item 3, and
 * section 5.6: the transform spreads block-level outliers before FP4
 * quantization).  x' = (1/4) H D x on every group of 16 consecutive rows of
 * each column (H the 16 x 16 Sylvester Hadamard matrix, D = diag(s) with
 * s_j = -1 where bit j of sign_mask is set), computed as the signs, the
 * FP32 butterfly with strides 1, 2, 4, 8, and the factor 1/4.  The groups
 * are the 16x1 blocks of the columnwise copy; H is orthogonal, so applying
 * the same transform to both wgrad operands leaves their product unchanged.
 * Then exactly the columnwise part of q_nvfp4 (Q_B1x16, rounding rnd,
 * stochastic draws of stream 1 indexed ((m / 16)*K + k)*16 + m % 16) on x':
 *   q_colT [K, M/2], sb_colT [K, M/16] (written);
 *   amax   one float: max|x'| written (Q_AMAX_COMPUTE, an extra read of x)
 *          or read (Q_AMAX_GIVEN, e.g. all-reduced over shards);
 *   s_global one float, written.
 * The rowwise (fprop) copy is quantized without the transform (q_nvfp4).
 * Shapes: M % 16 == 0, K % 16 == 0.
 */
/* max|x'| of the same transform (the amax q_nvfp4_rht_colT computes in
 * Q_AMAX_COMPUTE mode), for a caller that all-reduces it over shards first.
 * amax: one float, written.  Shapes as q_nvfp4_rht_colT. */
q_status q_nvfp4_rht_amax(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, float *amax,
                          int32_t *status, q_stream_t stream);

q_status q_nvfp4_rht_colT(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, q_round rnd,
                          uint64_t seed, uint64_t offset, uint8_t *q_colT, uint8_t *sb_colT,
                          float *amax, q_amax_mode amax_mode, float *s_global, int32_t *status, q_stream_t stream);

/*
 * Diagnostic of the host-side failure path (a library check, not an
 * operation of the pages): the next n launches attempted by the calling
 * thread fail as if the CUDA launch had returned cudaErrorLaunchFailure.
 * The entry point that meets one returns Q_ERR_CUDA with q_last_error()
 * naming the launch and the error, after its argument checks and before
 * anything is enqueued.  n = 0 clears a pending injection; n < 0 is
 * Q_ERR_ARG.
 */
q_status q_selftest_inject_launch_error(int n);

/*
 * Diagnostic of the device-side failure path (a library check, not an
 * operation of the pages).  Every wait in the kernels is bounded: a thread
 * that polls a shared-memory barrier longer than its limit gives up and ORs
 * Q_ST_TIMEOUT into the status word, and the context stays usable.  This
 * entry runs one warp that waits, with limit wait_ns, on a barrier whose
 * phase needs an arrival nobody makes, so the wait runs out and *status gets
 * Q_ST_TIMEOUT.  status: one device int32 (required); 0 < wait_ns <= 10^9.
 */
q_status q_selftest_wait_timeout(int32_t *status, uint64_t wait_ns, q_stream_t stream);

/*
 * Both maxima the NVFP4 recipe needs, in one read: *amax_rht = max|x'| (as
 * q_nvfp4_rht_amax) and *amax_x = max|x| (as q_amax).  For sharded tensors:
 * all-reduce both, then q_nvfp4_recipe with Q_AMAX_GIVEN (or q_nvfp4 rowwise
 * with amax_x and q_nvfp4_rht_colT with amax_rht, both Q_AMAX_GIVEN).
 * M % 16 == 0, K % 16 == 0.
 */
q_status q_nvfp4_rht_amax2(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, float *amax_rht,
                           float *amax_x, int32_t *status, q_stream_t stream);

/*
 * The NVFP4 training recipe's two copies of one tensor ([LP] §2.4: 1x16
 * blocks for activations and gradients, stochastic rounding on gradients,
 * the random Hadamard transform on the inputs of the weight-gradient GEMM,
 * which reads the columnwise copy): the rowwise 1x16 copy of x as q_nvfp4
 * gives it (q_row [M, K/2], sb_row [M, K/16], *s_global_row) and the
 * columnwise copy of x' (the transform of q_nvfp4_rht_amax) as
 * q_nvfp4_rht_colT gives it (q_colT [K, M/2], sb_colT [K, M/16],
 * *s_global_colT).  amax_mode Q_AMAX_COMPUTE: one pass takes both max|x| and
 * max|x'| into *amax_row / *amax_colT (as q_nvfp4_rht_amax2); Q_AMAX_GIVEN:
 * they are read from there (e.g. all-reduced over shards).  A BF16 x is then
 * read once more for both copies together, an FP32 x once for each.  With the
 * same seed and offset every output is bit-identical to q_nvfp4(rowwise
 * only) plus q_nvfp4_rht_colT (row draws from stream 0, transposed draws
 * from stream 1).  M % 16 == 0 and K % 16 == 0; all buffers required.
 */
q_status q_nvfp4_recipe(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, q_round rnd,
                        uint64_t seed, uint64_t offset, uint8_t *q_row, uint8_t *sb_row, float *amax_row,
                        float *s_global_row, uint8_t *q_colT, uint8_t *sb_colT, float *amax_colT,
                        float *s_global_colT, q_amax_mode amax_mode, int32_t *status, q_stream_t stream);

/*
 * a12: dequantizers.  Output y [R, C] in `out` (Q_F32, or Q_BF16 rounded to
 * nearest even from the FP32 value).  A transposed columnwise output is
 * passed as the [K, M] matrix it is (R = K, C = M).
 */

/* x_hat = q * s ([CS] "Current Scaling": x_hat_i = q_i * s).  q [R, C]
 * FP8 codes; scale: one device float.  Any R, C >= 0. */
q_status dq_current_scaling(const uint8_t *q, const float *scale, int64_t R, int64_t C,
                            q_fp8 fmt, q_dtype out, void *y, q_stream_t stream);

/* x_hat = q * 2^(code-127) ([MP] "MXFP8": value = element x block scale).
 * dir Q_ROW: e8m0 [R, C/32]; dir Q_COL: e8m0 [R/32, C].  C % 32 == 0
 * (Q_ROW) or R % 32 == 0 and C % 16 == 0 (Q_COL). */
q_status dq_mxfp8(const uint8_t *q, const uint8_t *e8m0, int64_t R, int64_t C, q_fp8 fmt,
                  q_dir dir, q_dtype out, void *y, q_stream_t stream);

/* x_hat = q * s_tile.  Q_T1x128: s [R, C/128]; Q_T128x128: s [R/128, C/128].
 * C % 128 == 0 (and R % 128 == 0 for Q_T128x128). */
q_status dq_blockwise(const uint8_t *q, const float *s, int64_t R, int64_t C, q_tile tile,
                      q_dtype out, void *y, q_stream_t stream);

/* x_hat = q * (sb * s_global), the block factor formed once per block.
 * q [R, C/2] packed; Q_B1x16: sb [R, C/16]; Q_B16x16: sb [R/16, C/16].
 * s_global: one device float.  C % 16 == 0 (and R % 16 == 0 for 16x16). */
q_status dq_nvfp4(const uint8_t *q, const uint8_t *sb, const float *s_global, int64_t R,
                  int64_t C, q_nvblk blk, q_dtype out, void *y, q_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q_H_ */
