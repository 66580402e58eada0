// The C ABI (include/q.h): argument validation on the host, then stream-
// ordered launches.  Nothing here allocates or synchronizes.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "q.h"
#include "q_internal.h"

namespace {

thread_local char g_err[512] = "";

q_status fail(q_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

q_status cuda_fail(const char *where, cudaError_t e)
{
    return fail(Q_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// M, K >= 0 and M*K < 2^62.
q_status check_dims(const char *fn, int64_t M, int64_t K)
{
    if (M < 0 || K < 0) return fail(Q_ERR_SHAPE, "%s: negative shape (%lld, %lld)", fn, (long long)M, (long long)K);
    if (M > 0 && K > ((int64_t)1 << 62) / M)
        return fail(Q_ERR_SHAPE, "%s: M*K too large (%lld x %lld)", fn, (long long)M, (long long)K);
    return Q_OK;
}

q_status check_in(const char *fn, const void *x, q_dtype in, int64_t n)
{
    if (in != Q_BF16 && in != Q_F32) return fail(Q_ERR_DTYPE, "%s: input dtype %d is not Q_BF16 or Q_F32", fn, (int)in);
    if (n > 0 && x == nullptr) return fail(Q_ERR_ARG, "%s: x is NULL", fn);
    if (!aligned(x, 16)) return fail(Q_ERR_ALIGN, "%s: x is not 16-byte aligned", fn);
    return Q_OK;
}

q_status need(const char *fn, const char *name, const void *p, uintptr_t align)
{
    if (p == nullptr) return fail(Q_ERR_ARG, "%s: %s is NULL", fn, name);
    if (!aligned(p, align)) return fail(Q_ERR_ALIGN, "%s: %s is not %u-byte aligned", fn, name, (unsigned)align);
    return Q_OK;
}

q_status multiple(const char *fn, const char *what, int64_t v, int64_t b)
{
    if (v % b != 0) return fail(Q_ERR_SHAPE, "%s: %s = %lld is not a multiple of %lld", fn, what, (long long)v, (long long)b);
    return Q_OK;
}

q_status check_out(const char *fn, q_dtype out)
{
    if (out != Q_BF16 && out != Q_F32) return fail(Q_ERR_DTYPE, "%s: output dtype %d is not Q_BF16 or Q_F32", fn, (int)out);
    return Q_OK;
}

#define TRY(expr)                      \
    do {                               \
        q_status s_ = (expr);          \
        if (s_ != Q_OK) return s_;     \
    } while (0)

// Launch failures injected by q_selftest_inject_launch_error: the next n
// launches of this thread fail with cudaErrorLaunchFailure before anything is
// enqueued (the error path of every entry point, exercised without a GPU).
thread_local int g_inject_launch_failures = 0;

#define LAUNCH(where, expr)                                                \
    do {                                                                   \
        if (g_inject_launch_failures > 0) {                                \
            g_inject_launch_failures--;                                    \
            return cuda_fail(where, cudaErrorLaunchFailure);               \
        }                                                                  \
        cudaError_t e_ = (expr);                                           \
        if (e_ != cudaSuccess) return cuda_fail(where, e_);                \
    } while (0)

cudaStream_t S(q_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char *q_last_error(void) { return g_err; }

int q_abi_version(void) { return 4; }

q_status q_amax(const void *x, q_dtype in, int64_t n, float *amax, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_amax";
    if (n < 0) return fail(Q_ERR_SHAPE, "%s: negative size %lld", fn, (long long)n);
    TRY(check_in(fn, x, in, n));
    TRY(need(fn, "amax", amax, 4));
    LAUNCH(fn, qk::launch_amax(x, (int)in, n, amax, status, S(stream)));
    return Q_OK;
}

q_status q_current_scaling(const void *x, q_dtype in, int64_t M, int64_t K, q_fp8 fmt, uint8_t *q_row,
                           uint8_t *q_colT, float *amax, q_amax_mode amax_mode, float *scale, int32_t *status,
                           q_stream_t stream)
{
    const char *fn = "q_current_scaling";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    if (amax_mode != Q_AMAX_COMPUTE && amax_mode != Q_AMAX_GIVEN) return fail(Q_ERR_ARG, "%s: bad amax_mode %d", fn, (int)amax_mode);
    const int64_t n = M * K;
    // an empty tensor has no codes to write (its buffers may be NULL)
    if (n > 0 && q_row == nullptr && q_colT == nullptr) return fail(Q_ERR_ARG, "%s: neither q_row nor q_colT requested", fn);
    if (n > 0 && q_row != nullptr) TRY(need(fn, "q_row", q_row, 16));
    if (n > 0 && q_colT != nullptr) {
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(multiple(fn, "M (with q_colT)", M, 16));
        TRY(multiple(fn, "K (with q_colT)", K, 16));
    }
    TRY(need(fn, "amax", amax, 4));
    TRY(need(fn, "scale", scale, 4));
    if (amax_mode == Q_AMAX_COMPUTE) LAUNCH("q_current_scaling/amax", qk::launch_amax(x, (int)in, n, amax, status, S(stream)));
    // an empty tensor takes the flat path, which only writes the scale
    LAUNCH("q_current_scaling/cast",
           qk::launch_cs_cast(x, (int)in, n == 0 ? 0 : M, n == 0 ? 0 : K, (int)fmt, amax, q_row,
                              n == 0 ? nullptr : q_colT, scale, status, S(stream), amax_mode == Q_AMAX_COMPUTE));
    return Q_OK;
}

q_status q_delayed_scaling(const void *x, q_dtype in, int64_t M, int64_t K, q_fp8 fmt, uint8_t *q_row,
                           uint8_t *q_colT, const float *ds, float *amax_out, float *scale, int32_t *status,
                           q_stream_t stream)
{
    const char *fn = "q_delayed_scaling";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    const int64_t n = M * K;
    if (n > 0 && q_row == nullptr && q_colT == nullptr) return fail(Q_ERR_ARG, "%s: neither q_row nor q_colT requested", fn);
    if (n > 0 && q_row != nullptr) TRY(need(fn, "q_row", q_row, 16));
    if (n > 0 && q_colT != nullptr) {
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(multiple(fn, "M (with q_colT)", M, 16));
        TRY(multiple(fn, "K (with q_colT)", K, 16));
    }
    TRY(need(fn, "ds", ds, 4));
    TRY(need(fn, "amax_out", amax_out, 4));
    TRY(need(fn, "scale", scale, 4));
    // an empty tensor takes the flat path: it writes the scale and a zero amax
    LAUNCH(fn, qk::launch_ds_cast(x, (int)in, n == 0 ? 0 : M, n == 0 ? 0 : K, (int)fmt, ds, amax_out, q_row,
                                  n == 0 ? nullptr : q_colT, scale, status, S(stream)));
    return Q_OK;
}

q_status q_delayed_scale_update(const float *hist, int64_t N, int64_t pos, q_hist_algo algo, q_fp8 fmt, float *ds,
                                q_stream_t stream)
{
    const char *fn = "q_delayed_scale_update";
    if (N < 1) return fail(Q_ERR_SHAPE, "%s: window length N = %lld must be >= 1", fn, (long long)N);
    if (pos < 0 || pos >= N) return fail(Q_ERR_ARG, "%s: pos %lld is outside [0, %lld)", fn, (long long)pos, (long long)N);
    if (algo != Q_HIST_MAX && algo != Q_HIST_MOST_RECENT) return fail(Q_ERR_ARG, "%s: bad algo %d", fn, (int)algo);
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    TRY(need(fn, "hist", hist, 4));
    TRY(need(fn, "ds", ds, 4));
    LAUNCH(fn, qk::launch_ds_update(hist, N, pos, (int)algo, (int)fmt, ds, S(stream)));
    return Q_OK;
}

q_status q_mxfp8(const void *x, q_dtype in, int64_t M, int64_t K, q_fp8 fmt, uint8_t *q_row, uint8_t *e8m0_row,
                 uint8_t *q_col, uint8_t *e8m0_col, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_mxfp8";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    TRY(multiple(fn, "K", K, 32));
    if (M * K == 0) return Q_OK;
    if (q_row == nullptr && q_col == nullptr) return fail(Q_ERR_ARG, "%s: neither direction requested", fn);
    if (q_row != nullptr) {
        TRY(need(fn, "q_row", q_row, 16));
        TRY(need(fn, "e8m0_row", e8m0_row, 1));
    }
    if (q_col != nullptr) {
        TRY(need(fn, "q_col", q_col, 16));
        TRY(need(fn, "e8m0_col", e8m0_col, 16));
        TRY(multiple(fn, "M (with q_col)", M, 32));
    }
    LAUNCH(fn, qk::launch_mxfp8(x, (int)in, M, K, (int)fmt, q_row, e8m0_row, q_col, e8m0_col, status, S(stream)));
    return Q_OK;
}

q_status q_mxfp8_requant_col(const uint8_t *q_row, const uint8_t *e8m0_row, int64_t M, int64_t K, q_fp8 fmt,
                             uint8_t *q_col, uint8_t *e8m0_col, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_mxfp8_requant_col";
    TRY(check_dims(fn, M, K));
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    TRY(multiple(fn, "K", K, 32));
    TRY(multiple(fn, "M", M, 32));
    if (M * K == 0) return Q_OK;
    TRY(need(fn, "q_row", q_row, 16));
    TRY(need(fn, "e8m0_row", e8m0_row, 1));
    TRY(need(fn, "q_col", q_col, 16));
    TRY(need(fn, "e8m0_col", e8m0_col, 16));
    LAUNCH(fn, qk::launch_mxfp8_requant_col(q_row, e8m0_row, M, K, (int)fmt, q_col, e8m0_col, status, S(stream)));
    return Q_OK;
}

q_status q_blockwise(const void *x, q_dtype in, int64_t M, int64_t K, q_tile tile, uint8_t *q_row, float *s_row,
                     uint8_t *q_colT, float *s_colT, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_blockwise";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (tile != Q_T1x128 && tile != Q_T128x128) return fail(Q_ERR_ARG, "%s: tile %d is not Q_T1x128 or Q_T128x128", fn, (int)tile);
    TRY(multiple(fn, "K", K, 128));
    if (tile == Q_T128x128) TRY(multiple(fn, "M (128x128 tiles)", M, 128));
    if (M * K == 0) return Q_OK;
    if (q_row == nullptr && q_colT == nullptr) return fail(Q_ERR_ARG, "%s: neither direction requested", fn);
    if (q_row != nullptr) {
        TRY(need(fn, "q_row", q_row, 16));
        TRY(need(fn, "s_row", s_row, 4));
    }
    if (q_colT != nullptr) {
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(need(fn, "s_colT", s_colT, 4));
        TRY(multiple(fn, "M (with q_colT)", M, 128));
    }
    LAUNCH(fn, qk::launch_blockwise(x, (int)in, M, K, (int)tile, q_row, s_row, q_colT, s_colT, status, S(stream)));
    return Q_OK;
}

q_status q_blockwise_mx(const void *x, q_dtype in, int64_t M, int64_t K, q_tile tile, uint8_t *q_row,
                        uint8_t *e8m0_row, uint8_t *q_colT, uint8_t *e8m0_colT, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_blockwise_mx";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (tile != Q_T1x128 && tile != Q_T128x128) return fail(Q_ERR_ARG, "%s: tile %d is not Q_T1x128 or Q_T128x128", fn, (int)tile);
    TRY(multiple(fn, "K", K, 128));
    if (tile == Q_T128x128) TRY(multiple(fn, "M (128x128 tiles)", M, 128));
    if (M * K == 0) return Q_OK;
    if (q_row == nullptr && q_colT == nullptr) return fail(Q_ERR_ARG, "%s: neither direction requested", fn);
    if (q_row != nullptr) {
        TRY(need(fn, "q_row", q_row, 16));
        TRY(need(fn, "e8m0_row", e8m0_row, 4));
    }
    if (q_colT != nullptr) {
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(need(fn, "e8m0_colT", e8m0_colT, 4));
        TRY(multiple(fn, "M (with q_colT)", M, 128));
    }
    LAUNCH(fn, qk::launch_blockwise_mx(x, (int)in, M, K, (int)tile, q_row, e8m0_row, q_colT, e8m0_colT, status,
                                       S(stream)));
    return Q_OK;
}

q_status q_nvfp4(const void *x, q_dtype in, int64_t M, int64_t K, q_nvblk blk, q_round rnd, uint64_t seed,
                 uint64_t offset, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT, float *amax,
                 q_amax_mode amax_mode, float *s_global, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_nvfp4";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (blk != Q_B1x16 && blk != Q_B16x16) return fail(Q_ERR_ARG, "%s: blk %d is not Q_B1x16 or Q_B16x16", fn, (int)blk);
    if (rnd != Q_RN && rnd != Q_SR) return fail(Q_ERR_ARG, "%s: rnd %d is not Q_RN or Q_SR", fn, (int)rnd);
    if (amax_mode != Q_AMAX_COMPUTE && amax_mode != Q_AMAX_GIVEN) return fail(Q_ERR_ARG, "%s: bad amax_mode %d", fn, (int)amax_mode);
    TRY(multiple(fn, "K", K, 16));
    TRY(multiple(fn, "M", M, 16));
    const bool empty = M * K == 0;   // no codes to write; buffers may be NULL
    if (!empty && q_row == nullptr && q_colT == nullptr) return fail(Q_ERR_ARG, "%s: neither direction requested", fn);
    if (!empty && q_row != nullptr) {
        TRY(need(fn, "q_row", q_row, 16));
        TRY(need(fn, "sb_row", sb_row, 1));
    }
    if (!empty && q_colT != nullptr) {
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(need(fn, "sb_colT", sb_colT, 16));
    }
    TRY(need(fn, "amax", amax, 4));
    TRY(need(fn, "s_global", s_global, 4));
    if (amax_mode == Q_AMAX_COMPUTE) LAUNCH("q_nvfp4/amax", qk::launch_amax(x, (int)in, M * K, amax, status, S(stream)));
    LAUNCH("q_nvfp4/cast", qk::launch_nvfp4(x, (int)in, M, K, (int)blk, (int)rnd, seed, offset, amax, q_row, sb_row,
                                            q_colT, sb_colT, s_global, status, S(stream), amax_mode == Q_AMAX_COMPUTE));
    return Q_OK;
}

q_status q_nvfp4_rht_amax(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, float *amax,
                          int32_t *status, q_stream_t stream)
{
    const char *fn = "q_nvfp4_rht_amax";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (sign_mask > 0xFFFFu) return fail(Q_ERR_ARG, "%s: sign_mask 0x%x has bits above bit 15", fn, sign_mask);
    TRY(multiple(fn, "K", K, 16));
    TRY(multiple(fn, "M", M, 16));
    TRY(need(fn, "amax", amax, 4));
    LAUNCH(fn, qk::launch_rht_amax(x, (int)in, M, K, sign_mask, amax, nullptr, status, S(stream)));
    return Q_OK;
}

q_status q_nvfp4_rht_amax2(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, float *amax_rht,
                           float *amax_x, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_nvfp4_rht_amax2";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (sign_mask > 0xFFFFu) return fail(Q_ERR_ARG, "%s: sign_mask 0x%x has bits above bit 15", fn, sign_mask);
    TRY(multiple(fn, "K", K, 16));
    TRY(multiple(fn, "M", M, 16));
    TRY(need(fn, "amax_rht", amax_rht, 4));
    TRY(need(fn, "amax_x", amax_x, 4));
    LAUNCH(fn, qk::launch_rht_amax(x, (int)in, M, K, sign_mask, amax_rht, amax_x, status, S(stream)));
    return Q_OK;
}

q_status q_nvfp4_recipe(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, q_round rnd,
                        uint64_t seed, uint64_t offset, uint8_t *q_row, uint8_t *sb_row, float *amax_row,
                        float *s_global_row, uint8_t *q_colT, uint8_t *sb_colT, float *amax_colT,
                        float *s_global_colT, q_amax_mode amax_mode, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_nvfp4_recipe";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (rnd != Q_RN && rnd != Q_SR) return fail(Q_ERR_ARG, "%s: rnd %d is not Q_RN or Q_SR", fn, (int)rnd);
    if (amax_mode != Q_AMAX_COMPUTE && amax_mode != Q_AMAX_GIVEN) return fail(Q_ERR_ARG, "%s: bad amax_mode %d", fn, (int)amax_mode);
    if (sign_mask > 0xFFFFu) return fail(Q_ERR_ARG, "%s: sign_mask 0x%x has bits above bit 15", fn, sign_mask);
    TRY(multiple(fn, "K", K, 16));
    TRY(multiple(fn, "M", M, 16));
    TRY(need(fn, "amax_row", amax_row, 4));
    TRY(need(fn, "s_global_row", s_global_row, 4));
    TRY(need(fn, "amax_colT", amax_colT, 4));
    TRY(need(fn, "s_global_colT", s_global_colT, 4));
    if (M * K != 0) {
        TRY(need(fn, "q_row", q_row, 16));
        TRY(need(fn, "sb_row", sb_row, 1));
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(need(fn, "sb_colT", sb_colT, 16));   // written in 8-byte pieces
    }
    // one read for both maxima (unless given), then the rowwise cast and the
    // transformed columnwise cast with them: for BF16 in one pass over x,
    // for FP32 in two
    const bool compute = amax_mode == Q_AMAX_COMPUTE;
    if (compute) LAUNCH(fn, qk::launch_rht_amax(x, (int)in, M, K, sign_mask, amax_colT, amax_row, status, S(stream)));
    if (in == Q_BF16) {
        LAUNCH(fn, qk::launch_nvfp4_bf16_recipe(x, M, K, sign_mask, (int)rnd, seed, offset, amax_row, q_row, sb_row,
                                                s_global_row, amax_colT, q_colT, sb_colT, s_global_colT, status,
                                                S(stream), compute));
        return Q_OK;
    }
    LAUNCH(fn, qk::launch_nvfp4(x, (int)in, M, K, (int)Q_B1x16, (int)rnd, seed, offset, amax_row, q_row, sb_row, nullptr,
                                nullptr, s_global_row, status, S(stream), compute));
    LAUNCH(fn, qk::launch_nvfp4_rht_colT(x, (int)in, M, K, sign_mask, (int)rnd, seed, offset, false, amax_colT, q_colT,
                                         sb_colT, s_global_colT, status, S(stream)));
    return Q_OK;
}

q_status q_nvfp4_rht_colT(const void *x, q_dtype in, int64_t M, int64_t K, uint32_t sign_mask, q_round rnd,
                          uint64_t seed, uint64_t offset, uint8_t *q_colT, uint8_t *sb_colT, float *amax,
                          q_amax_mode amax_mode, float *s_global, int32_t *status, q_stream_t stream)
{
    const char *fn = "q_nvfp4_rht_colT";
    TRY(check_dims(fn, M, K));
    TRY(check_in(fn, x, in, M * K));
    if (rnd != Q_RN && rnd != Q_SR) return fail(Q_ERR_ARG, "%s: rnd %d is not Q_RN or Q_SR", fn, (int)rnd);
    if (amax_mode != Q_AMAX_COMPUTE && amax_mode != Q_AMAX_GIVEN) return fail(Q_ERR_ARG, "%s: bad amax_mode %d", fn, (int)amax_mode);
    if (sign_mask > 0xFFFFu) return fail(Q_ERR_ARG, "%s: sign_mask 0x%x has bits above bit 15", fn, sign_mask);
    TRY(multiple(fn, "K", K, 16));
    TRY(multiple(fn, "M", M, 16));
    if (M * K > 0) {
        TRY(need(fn, "q_colT", q_colT, 16));
        TRY(need(fn, "sb_colT", sb_colT, 16));
    }
    TRY(need(fn, "amax", amax, 4));
    TRY(need(fn, "s_global", s_global, 4));
    LAUNCH(fn, qk::launch_nvfp4_rht_colT(x, (int)in, M, K, sign_mask, (int)rnd, seed, offset, amax_mode == Q_AMAX_COMPUTE,
                                         amax, q_colT, sb_colT, s_global, status, S(stream)));
    return Q_OK;
}

q_status q_selftest_inject_launch_error(int n)
{
    if (n < 0) return fail(Q_ERR_ARG, "q_selftest_inject_launch_error: n = %d is negative", n);
    g_inject_launch_failures = n;
    return Q_OK;
}

q_status q_selftest_wait_timeout(int32_t *status, uint64_t wait_ns, q_stream_t stream)
{
    const char *fn = "q_selftest_wait_timeout";
    TRY(need(fn, "status", status, 4));
    if (wait_ns == 0 || wait_ns > 1000000000ull) return fail(Q_ERR_ARG, "%s: wait_ns %llu is outside (0, 1e9]", fn, (unsigned long long)wait_ns);
    LAUNCH(fn, qk::launch_selftest_wait(status, (unsigned long long)wait_ns, S(stream)));
    return Q_OK;
}

q_status dq_current_scaling(const uint8_t *q, const float *scale, int64_t R, int64_t C, q_fp8 fmt, q_dtype out,
                            void *y, q_stream_t stream)
{
    const char *fn = "dq_current_scaling";
    TRY(check_dims(fn, R, C));
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    TRY(check_out(fn, out));
    if (R * C == 0) return Q_OK;
    TRY(need(fn, "q", q, 16));
    TRY(need(fn, "scale", scale, 4));
    TRY(need(fn, "y", y, 16));
    LAUNCH(fn, qk::launch_dq_cs(q, scale, R, C, (int)fmt, (int)out, y, S(stream)));
    return Q_OK;
}

q_status dq_mxfp8(const uint8_t *q, const uint8_t *e8m0, int64_t R, int64_t C, q_fp8 fmt, q_dir dir, q_dtype out,
                  void *y, q_stream_t stream)
{
    const char *fn = "dq_mxfp8";
    TRY(check_dims(fn, R, C));
    if (fmt != Q_E4M3 && fmt != Q_E5M2) return fail(Q_ERR_ARG, "%s: fmt %d is not Q_E4M3 or Q_E5M2", fn, (int)fmt);
    if (dir != Q_ROW && dir != Q_COL) return fail(Q_ERR_ARG, "%s: dir %d is not Q_ROW or Q_COL", fn, (int)dir);
    TRY(check_out(fn, out));
    if (dir == Q_ROW) TRY(multiple(fn, "C", C, 32));
    else {
        TRY(multiple(fn, "R (Q_COL)", R, 32));
        TRY(multiple(fn, "C (Q_COL)", C, 16));
    }
    if (R * C == 0) return Q_OK;
    TRY(need(fn, "q", q, 16));
    TRY(need(fn, "e8m0", e8m0, dir == Q_COL ? 16 : 1));
    TRY(need(fn, "y", y, 16));
    LAUNCH(fn, qk::launch_dq_mxfp8(q, e8m0, R, C, (int)fmt, (int)dir, (int)out, y, S(stream)));
    return Q_OK;
}

q_status dq_blockwise(const uint8_t *q, const float *s, int64_t R, int64_t C, q_tile tile, q_dtype out, void *y,
                      q_stream_t stream)
{
    const char *fn = "dq_blockwise";
    TRY(check_dims(fn, R, C));
    if (tile != Q_T1x128 && tile != Q_T128x128) return fail(Q_ERR_ARG, "%s: tile %d is not Q_T1x128 or Q_T128x128", fn, (int)tile);
    TRY(check_out(fn, out));
    TRY(multiple(fn, "C", C, 128));
    if (tile == Q_T128x128) TRY(multiple(fn, "R (128x128)", R, 128));
    if (R * C == 0) return Q_OK;
    TRY(need(fn, "q", q, 16));
    TRY(need(fn, "s", s, 4));
    TRY(need(fn, "y", y, 16));
    LAUNCH(fn, qk::launch_dq_blockwise(q, s, R, C, (int)tile, (int)out, y, S(stream)));
    return Q_OK;
}

q_status dq_nvfp4(const uint8_t *q, const uint8_t *sb, const float *s_global, int64_t R, int64_t C, q_nvblk blk,
                  q_dtype out, void *y, q_stream_t stream)
{
    const char *fn = "dq_nvfp4";
    TRY(check_dims(fn, R, C));
    if (blk != Q_B1x16 && blk != Q_B16x16) return fail(Q_ERR_ARG, "%s: blk %d is not Q_B1x16 or Q_B16x16", fn, (int)blk);
    TRY(check_out(fn, out));
    TRY(multiple(fn, "C", C, 16));
    if (blk == Q_B16x16) TRY(multiple(fn, "R (16x16)", R, 16));
    if (R * C == 0) return Q_OK;
    TRY(need(fn, "q", q, 16));
    TRY(need(fn, "sb", sb, 1));
    TRY(need(fn, "s_global", s_global, 4));
    TRY(need(fn, "y", y, 16));
    LAUNCH(fn, qk::launch_dq_nvfp4(q, sb, s_global, R, C, (int)blk, (int)out, y, S(stream)));
    return Q_OK;
}

}  // extern "C"
