// Launchers shared between the C-ABI layer (q_api.cu) and the kernel files.
// Every launcher enqueues on `st` and returns cudaGetLastError().
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qk {

int sm_count();

// Launch `kernel`; with pdl = true, as a programmatic dependent of the kernel
// before it in the stream (the kernel then calls griddep_wait() before it
// reads that kernel's output).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? at : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// A 2-D TMA tensor map over a row-major [M, K] input (dt: BF16, F32, or U8
// for code matrices, K even) whose box is box_rows rows x 512 bytes (the tile
// engine's stage; box_rows <= 256).  The x coordinate counts elements of 2
// bytes (BF16, U8) or 4 bytes (F32).  Fails with cudaErrorNotSupported if the
// driver entry point is unavailable.
cudaError_t make_tile_map(void *map /* CUtensorMap, 64-byte aligned */, const void *x, int dt, int64_t M, int64_t K,
                          int box_rows = 128);

// A 2-D TMA tensor map for bulk stores into a row-major byte matrix of
// `rows` rows of row_bytes bytes (row_bytes a multiple of 16, base 16-byte
// aligned), box box_bytes x box_rows (box_bytes a multiple of 16, both <= 256).
cudaError_t make_store_map_u8(void *map /* CUtensorMap, 64-byte aligned */, void *base, int64_t row_bytes,
                              int64_t rows, int box_bytes, int box_rows);

// current scaling
cudaError_t launch_amax(const void *x, int dt, int64_t n, float *amax, int32_t *status, cudaStream_t st);
cudaError_t launch_cs_cast(const void *x, int dt, int64_t M, int64_t K, int fmt, const float *amax,
                           uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st,
                           bool after_amax);

// MXFP8
cudaError_t launch_mxfp8(const void *x, int dt, int64_t M, int64_t K, int fmt, uint8_t *q_row,
                         uint8_t *e_row, uint8_t *q_col, uint8_t *e_col, int32_t *status, cudaStream_t st);

// one warp waits wait_ns on a barrier nothing completes, then reports Q_ST_TIMEOUT
cudaError_t launch_selftest_wait(int32_t *status, unsigned long long wait_ns, cudaStream_t st);

// *w = 0 (and *w2 = 0 when given; one thread), stream-ordered before a reduction into it
cudaError_t launch_zero_word(float *w, cudaStream_t st, float *w2 = nullptr);

// max|x'| of the random Hadamard transform along M, and max|x| into *amax_x
// when it is given, in one read (zeroes both words first)
cudaError_t launch_rht_amax(const void *x, int dt, int64_t M, int64_t K, uint32_t sign_mask, float *amax,
                            float *amax_x, int32_t *status, cudaStream_t st);

// random Hadamard transform along M + columnwise NVFP4 of the result; the
// amax of the transformed tensor is reduced into *amax first unless given
cudaError_t launch_nvfp4_rht_colT(const void *x, int dt, int64_t M, int64_t K, uint32_t sign_mask, int rnd,
                                  uint64_t seed, uint64_t offset, bool compute_amax, float *amax, uint8_t *q_colT,
                                  uint8_t *sb_colT, float *s_global, int32_t *status, cudaStream_t st);

// delayed scaling: cast with the pair ds = [alpha, s], recording max|x| into
// *amax_rec (zeroed first); next pair from the window of N amaxes
cudaError_t launch_ds_cast(const void *x, int dt, int64_t M, int64_t K, int fmt, const float *ds, float *amax_rec,
                           uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st);
cudaError_t launch_ds_update(const float *hist, int64_t N, int64_t pos, int algo, int fmt, float *ds, cudaStream_t st);

// MXFP8 rowwise codes -> columnwise codes (dequantize + re-quantize)
cudaError_t launch_mxfp8_requant_col(const uint8_t *q_row, const uint8_t *e_row, int64_t M, int64_t K, int fmt,
                                     uint8_t *q_col, uint8_t *e_col, int32_t *status, cudaStream_t st);

// blockwise
cudaError_t launch_blockwise(const void *x, int dt, int64_t M, int64_t K, int tile, uint8_t *q_row,
                             float *s_row, uint8_t *q_colT, float *s_colT, int32_t *status, cudaStream_t st);
cudaError_t launch_blockwise_mx(const void *x, int dt, int64_t M, int64_t K, int tile, uint8_t *q_row,
                                uint8_t *e_row, uint8_t *q_colT, uint8_t *e_colT, int32_t *status, cudaStream_t st);

// NVFP4 (the amax is already in *amax)
cudaError_t launch_nvfp4(const void *x, int dt, int64_t M, int64_t K, int blk, int rnd, uint64_t seed,
                         uint64_t offset, const float *amax, uint8_t *q_row, uint8_t *sb_row,
                         uint8_t *q_colT, uint8_t *sb_colT, float *s_global, int32_t *status,
                         cudaStream_t st, bool after_amax);

// NVFP4 of a BF16 tensor (the BF16 path of launch_nvfp4)
cudaError_t launch_nvfp4_bf16(const void *x, int64_t M, int64_t K, int blk, int rnd, uint64_t seed, uint64_t offset,
                              const float *amax, uint8_t *q_row, uint8_t *sb_row, uint8_t *q_colT, uint8_t *sb_colT,
                              float *s_global, int32_t *status, cudaStream_t st, bool after_amax);
// NVFP4 recipe, BF16 input: rowwise 1x16 copy of x and columnwise copy of its
// random Hadamard transform in one pass, with the two tensor maxima given
// (after_amax: launched behind the kernel that reduced them)
cudaError_t launch_nvfp4_bf16_recipe(const void *x, int64_t M, int64_t K, uint32_t sign_mask, int rnd, uint64_t seed,
                                     uint64_t offset, const float *amax_row, uint8_t *q_row, uint8_t *sb_row,
                                     float *s_global_row, const float *amax_col, uint8_t *q_colT, uint8_t *sb_colT,
                                     float *s_global_col, int32_t *status, cudaStream_t st, bool after_amax);

// dequantizers
cudaError_t launch_dq_cs(const uint8_t *q, const float *s, int64_t R, int64_t C, int fmt, int out,
                         void *y, cudaStream_t st);
cudaError_t launch_dq_mxfp8(const uint8_t *q, const uint8_t *e, int64_t R, int64_t C, int fmt, int dir,
                            int out, void *y, cudaStream_t st);
cudaError_t launch_dq_blockwise(const uint8_t *q, const float *s, int64_t R, int64_t C, int tile, int out,
                                void *y, cudaStream_t st);
cudaError_t launch_dq_nvfp4(const uint8_t *q, const uint8_t *sb, const float *s_g, int64_t R, int64_t C,
                            int blk, int out, void *y, cudaStream_t st);

// Scales of an empty tensor (amax 0): writes *amax = 0 (if amax_out), *scale = 1.
cudaError_t launch_empty_scales(float *amax_out, float *scale, cudaStream_t st);

}  // namespace qk
