// Per-tensor current scaling: the amax pass (a1), the scale (a2) and the
// scale + cast pass (a3) with its optional transposed copy.
//
// "FP8 Current Scaling: quantization, scaling and precision bounds", section
// "Current Scaling": a = max|x|, alpha = Fmax / a, q = Q(alpha x), s = 1/alpha;
// section "Cost and multi-GPU use": the tensor is read twice.
// "Mixed-precision training: fp16 to fp8", "Per-tensor Current Scaling"
// (Hopper flow): one kernel writes the cast and the cast_transpose.
//
// The two passes are two launches in stream order (no grid-wide barrier, no
// spin-wait).  Every CTA of the cast pass recomputes alpha from the amax
// word (identical in every CTA); CTA 0 writes s.  The cast pass walks the
// tensor from its end, so the last part the amax pass streamed (still in L2)
// is consumed first.
#include "q_common.cuh"
#include "q_internal.h"

namespace qk {

int sm_count()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    }
    return n;
}

// ---------------------------------------------------------------------------
// a1: amax.  Grid-stride 16-byte loads (four in flight per thread), |x| max
// on bit patterns, warp reduce, CTA reduce, one atomicMax per CTA.
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(512) k_amax(const void *__restrict__ x, int64_t n, uint32_t *__restrict__ amax)
{
    constexpr int VEC = In<DT>::VEC;
    const uint4 *xv = static_cast<const uint4 *>(x);
    const int64_t nv = n / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t m = 0;
    for (; i + 3 * stride < nv; i += 4 * stride) {
        uint4 a = ldg_stream(xv + i), b = ldg_stream(xv + i + stride);
        uint4 c = ldg_stream(xv + i + 2 * stride), d = ldg_stream(xv + i + 3 * stride);
        m = max(m, max(max(absmax_bits<DT>(a), absmax_bits<DT>(b)), max(absmax_bits<DT>(c), absmax_bits<DT>(d))));
    }
    for (; i < nv; i += stride) m = max(m, absmax_bits<DT>(ldg_stream(xv + i)));
    // the last n % VEC elements, one per thread of CTA 0
    if (blockIdx.x == 0 && threadIdx.x < n - nv * VEC) {
        int64_t t = nv * VEC + threadIdx.x;
        uint32_t u = DT == BF16 ? (uint32_t)static_cast<const uint16_t *>(x)[t] << 16
                                : __float_as_uint(static_cast<const float *>(x)[t]);
        m = max(m, u & 0x7FFFFFFFu);
    }
    m = warp_max(m);
    __shared__ uint32_t red[16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
        m = warp_max(m);
        if (lane == 0 && m != 0) atomicMax(amax, m);
    }
}

// ---------------------------------------------------------------------------
// a3, rowwise only: flat streaming cast, 16 elements -> one 16-byte store.
// ---------------------------------------------------------------------------
template <int DT, int FMT>
__global__ void __launch_bounds__(256) k_cs_cast_flat(const void *__restrict__ x, int64_t n,
                                                      const float *__restrict__ amax, uint8_t *__restrict__ q,
                                                      float *__restrict__ scale, int32_t *status)
{
    constexpr int VEC = In<DT>::VEC;
    constexpr int VPC = 16 / VEC;   // 16-byte input vectors per 16-element chunk
    const float a = *amax;
    const float alpha = alpha_from_amax(Fp8<FMT>::FMAX, a);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *scale = __fdiv_rn(1.0f, alpha);
        flag_nonfinite(status, __float_as_uint(a) & 0x7FFFFFFFu);
    }
    const uint4 *xv = static_cast<const uint4 *>(x);
    const int64_t nc = n / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nc; i += 2 * stride) {
        const int64_t c0 = nc - 1 - i, c1 = c0 - stride;   // backwards: L2-resident data first
        uint4 v0[VPC], v1[VPC];
#pragma unroll
        for (int j = 0; j < VPC; j++) v0[j] = ldg_stream(xv + c0 * VPC + j);
        if (c1 >= 0) {
#pragma unroll
            for (int j = 0; j < VPC; j++) v1[j] = ldg_stream(xv + c1 * VPC + j);
        }
        uint32_t o[4];
#pragma unroll
        for (int w = 0; w < 4; w++) {
            const int e = 4 * w;   // element index within the chunk
            o[w] = cvt_fp8x4<FMT>(__fmul_rn(alpha, elem<DT>(v0[e / VEC], e % VEC)),
                                  __fmul_rn(alpha, elem<DT>(v0[(e + 1) / VEC], (e + 1) % VEC)),
                                  __fmul_rn(alpha, elem<DT>(v0[(e + 2) / VEC], (e + 2) % VEC)),
                                  __fmul_rn(alpha, elem<DT>(v0[(e + 3) / VEC], (e + 3) % VEC)));
        }
        stg16(q + c0 * 16, make_uint4(o[0], o[1], o[2], o[3]));
        if (c1 >= 0) {
#pragma unroll
            for (int w = 0; w < 4; w++) {
                const int e = 4 * w;
                o[w] = cvt_fp8x4<FMT>(__fmul_rn(alpha, elem<DT>(v1[e / VEC], e % VEC)),
                                      __fmul_rn(alpha, elem<DT>(v1[(e + 1) / VEC], (e + 1) % VEC)),
                                      __fmul_rn(alpha, elem<DT>(v1[(e + 2) / VEC], (e + 2) % VEC)),
                                      __fmul_rn(alpha, elem<DT>(v1[(e + 3) / VEC], (e + 3) % VEC)));
            }
            stg16(q + c1 * 16, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
    // the last n % 16 elements, one per thread of CTA 0
    if (blockIdx.x == 0 && threadIdx.x < n - nc * 16) {
        const int64_t t = nc * 16 + threadIdx.x;
        float v = DT == BF16 ? __uint_as_float((uint32_t)static_cast<const uint16_t *>(x)[t] << 16)
                             : static_cast<const float *>(x)[t];
        q[t] = (uint8_t)(cvt_fp8x4<FMT>(__fmul_rn(alpha, v), 0.f, 0.f, 0.f) & 0xFFu);
    }
}

// ---------------------------------------------------------------------------
// a3 with the transposed copy: a CTA owns a 128 x (32*VEC) tile.  The codes
// are computed once; rowwise they are stored straight from registers, and
// for the transpose each thread turns its 16 x VEC byte block around with
// byte permutes, parks it in shared memory ([column][128 rows], 16-byte
// chunks XOR-swizzled by column group so that neither side conflicts), and
// the CTA then writes full 128-byte rows of q_colT.
// Requires M % 16 == 0 and K % 16 == 0 (checked by the host).
// ---------------------------------------------------------------------------
template <int DT, int FMT>
__global__ void __launch_bounds__(kThreads) k_cs_cast_tiled(const void *__restrict__ x, int64_t M, int64_t K,
                                                            const float *__restrict__ amax,
                                                            uint8_t *__restrict__ q_row,
                                                            uint8_t *__restrict__ q_colT,
                                                            float *__restrict__ scale, int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, BYTES = In<DT>::BYTES, TC = 32 * VEC, CW = VEC / 4;
    __shared__ __align__(16) uint8_t sT[TC * kTileRows];

    const float a = *amax;
    const float alpha = alpha_from_amax(Fp8<FMT>::FMAX, a);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *scale = __fdiv_rn(1.0f, alpha);
        flag_nonfinite(status, __float_as_uint(a) & 0x7FFFFFFFu);
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_k = (K + TC - 1) / TC;
    const int64_t t = (int64_t)gridDim.x - 1 - blockIdx.x;    // backwards
    const int64_t tm = t / tiles_k, tk = t - tm * tiles_k;
    const int64_t m0 = tm * kTileRows + warp * kRowsPerWarp;
    const int64_t k0 = tk * TC + lane * VEC;
    const bool ok = (m0 < M) && (k0 < K);

    uint32_t code[kRowsPerWarp][CW];
    if (ok) {
        uint4 v[kRowsPerWarp];
        const char *base = static_cast<const char *>(x) + (m0 * K + k0) * BYTES;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++) v[r] = ldg_stream(base + (int64_t)r * K * BYTES);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; r++)
#pragma unroll
            for (int w = 0; w < CW; w++)
                code[r][w] = cvt_fp8x4<FMT>(__fmul_rn(alpha, elem<DT>(v[r], 4 * w)),
                                            __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 1)),
                                            __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 2)),
                                            __fmul_rn(alpha, elem<DT>(v[r], 4 * w + 3)));
        if (q_row != nullptr) {
            uint8_t *dst = q_row + m0 * K + k0;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; r++) {
                if (CW == 2) stg8(dst + (int64_t)r * K, code[r][0], code[r][CW - 1]);
                else stg4(dst + (int64_t)r * K, code[r][0]);
            }
        }
        if (q_colT != nullptr) {
#pragma unroll
            for (int w = 0; w < CW; w++) {
                uint32_t c[4][4];   // c[i][g]: column 4w+i, rows 4g..4g+3
#pragma unroll
                for (int g = 0; g < 4; g++)
                    transpose4x4(code[4 * g][w], code[4 * g + 1][w], code[4 * g + 2][w], code[4 * g + 3][w],
                                 c[0][g], c[1][g], c[2][g], c[3][g]);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int col = lane * VEC + 4 * w + i;
                    const int chunk = warp ^ (lane & 7);
                    *reinterpret_cast<uint4 *>(sT + col * kTileRows + chunk * 16) =
                        make_uint4(c[i][0], c[i][1], c[i][2], c[i][3]);
                }
            }
        }
    }
    if (q_colT == nullptr) return;
    __syncthreads();
    // 8 lanes per column row: each writes one 16-byte chunk (16 rows of m)
#pragma unroll
    for (int it = 0; it < TC * 8 / kThreads; it++) {
        const int idx = it * kThreads + threadIdx.x;
        const int col = idx >> 3, ch = idx & 7;
        const int64_t kg = tk * TC + col, mg = tm * kTileRows + ch * 16;
        if (kg < K && mg < M) {
            const int phys = ch ^ ((col / VEC) & 7);
            uint4 val = *reinterpret_cast<const uint4 *>(sT + col * kTileRows + phys * 16);
            stg16(q_colT + kg * M + mg, val);
        }
    }
}

// Scales of an empty tensor.
__global__ void k_empty_scales(float *amax_out, float *scale)
{
    if (amax_out != nullptr) *amax_out = 0.0f;
    if (scale != nullptr) *scale = 1.0f;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

cudaError_t launch_amax(const void *x, int dt, int64_t n, float *amax, int32_t *status, cudaStream_t st)
{
    (void)status;
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
    if (e != cudaSuccess || n == 0) return e;
    const int vec = dt == BF16 ? 8 : 4;
    const int64_t nv = n / vec;
    int64_t blocks = (nv + 511) / 512;
    const int64_t cap = (int64_t)sm_count() * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (dt == BF16) k_amax<BF16><<<(unsigned)blocks, 512, 0, st>>>(x, n, reinterpret_cast<uint32_t *>(amax));
    else k_amax<F32><<<(unsigned)blocks, 512, 0, st>>>(x, n, reinterpret_cast<uint32_t *>(amax));
    return cudaGetLastError();
}

template <int DT, int FMT>
static cudaError_t cs_cast_t(const void *x, int64_t M, int64_t K, const float *amax, uint8_t *q_row,
                             uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st)
{
    if (q_colT == nullptr) {
        const int64_t n = M * K, nc = n / 16;
        int64_t blocks = (nc + 2 * 256 - 1) / (2 * 256);
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        k_cs_cast_flat<DT, FMT><<<(unsigned)blocks, 256, 0, st>>>(x, n, amax, q_row, scale, status);
    } else {
        constexpr int TC = 32 * In<DT>::VEC;
        const int64_t tiles = ((M + kTileRows - 1) / kTileRows) * ((K + TC - 1) / TC);
        k_cs_cast_tiled<DT, FMT><<<(unsigned)tiles, kThreads, 0, st>>>(x, M, K, amax, q_row, q_colT, scale, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_cs_cast(const void *x, int dt, int64_t M, int64_t K, int fmt, const float *amax,
                           uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st)
{
    if (dt == BF16) {
        return fmt == E4M3 ? cs_cast_t<BF16, E4M3>(x, M, K, amax, q_row, q_colT, scale, status, st)
                           : cs_cast_t<BF16, E5M2>(x, M, K, amax, q_row, q_colT, scale, status, st);
    }
    return fmt == E4M3 ? cs_cast_t<F32, E4M3>(x, M, K, amax, q_row, q_colT, scale, status, st)
                       : cs_cast_t<F32, E5M2>(x, M, K, amax, q_row, q_colT, scale, status, st);
}

cudaError_t launch_empty_scales(float *amax_out, float *scale, cudaStream_t st)
{
    k_empty_scales<<<1, 1, 0, st>>>(amax_out, scale);
    return cudaGetLastError();
}

}  // namespace qk
