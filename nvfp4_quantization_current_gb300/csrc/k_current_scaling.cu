// Per-tensor current scaling: the amax pass (a1), the scale (a2) and the
// scale + cast pass (a3) with its optional transposed copy.
//
// "FP8 Current Scaling: quantization, scaling and precision bounds", section
// "Current Scaling": a = max|x|, alpha = Fmax / a, q = Q(alpha x), s = 1/alpha;
// section "Cost and multi-GPU use": the tensor is read twice.
// "Mixed-precision training: fp16 to fp8", "Per-tensor Current Scaling"
// (Hopper flow): one kernel writes the cast and the cast_transpose.
//
// Per-tensor delayed scaling ("Mixed-precision training: fp16 to fp8",
// "Per-tensor delayed scaling") runs the same cast kernels with DS = true:
// alpha and s come from a device pair written by the previous step's scale
// update, and the pass also reduces max|x| into this step's slot of the amax
// window, so x is read once.  k_ds_update derives the next pair from the
// window.
//
// The two passes are two launches in stream order (no grid-wide barrier, no
// spin-wait).  Every CTA of the cast pass recomputes alpha from the amax
// word (identical in every CTA); CTA 0 writes s.  The cast pass walks the
// tensor from its end, so the last part the amax pass streamed (still in L2)
// is consumed first.
#include "q_engine.cuh"
#include "q_internal.h"

namespace qk {

// SM count of the current device, cached per device (grids are sized by it;
// a failed query falls back to GB300's 152, which only affects grid sizes).
int sm_count()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// ---------------------------------------------------------------------------
// a1: amax.  Grid-stride 16-byte loads, eight in flight per thread (each
// batch predicated, so the tail costs one memory round trip, not one per
// leftover load), |x| max on bit patterns, warp reduce, CTA reduce, one
// atomicMax per CTA.
// ---------------------------------------------------------------------------
constexpr int kAmaxThreads = 256, kAmaxUnroll = 8;

template <int DT>
__global__ void __launch_bounds__(kAmaxThreads, 4) k_amax(const void *__restrict__ x, int64_t n, uint32_t *__restrict__ amax)
{
    constexpr int VEC = In<DT>::VEC;
    griddep_launch_dependents();   // the cast behind this pass may be scheduled; it waits for the amax
    const uint4 *xv = static_cast<const uint4 *>(x);
    const int64_t nv = n / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t m = 0;
    for (; i < nv; i += kAmaxUnroll * stride) {
        uint4 a[kAmaxUnroll];
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; u++)
            a[u] = i + u * stride < nv ? ldg_stream(xv + i + u * stride) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kAmaxUnroll; u++) m = max(m, absmax_bits<DT>(a[u]));
    }
    // the last n % VEC elements, one per thread of CTA 0
    if (blockIdx.x == 0 && threadIdx.x < n - nv * VEC) {
        const int64_t t = nv * VEC + threadIdx.x;
        const uint32_t u = DT == BF16 ? (uint32_t)static_cast<const uint16_t *>(x)[t] << 16
                                      : __float_as_uint(static_cast<const float *>(x)[t]);
        m = max(m, u & 0x7FFFFFFFu);
    }
    m = warp_max(m);
    __shared__ uint32_t red[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kAmaxThreads / 32 ? red[lane] : 0u;
        m = warp_max(m);
        griddep_wait();   // the zeroing of *amax (the kernel ahead of this one) is complete
        // same-address atomics serialize in L2: only a CTA that raises the
        // running maximum pays for one
        if (lane == 0 && m > *reinterpret_cast<volatile uint32_t *>(amax)) atomicMax(amax, m);
    }
}

// alpha of the cast: from the amax (current scaling) or the pair [alpha, s]
// (delayed scaling); CTA 0 writes s and reports a non-finite amax or alpha.
template <int FMT, bool DS>
QD float cast_alpha(const float *amax, const float *ds, float *scale, int32_t *status)
{
    griddep_wait();   // the amax pass (or the zeroing of the delayed-scaling slot) ahead of this kernel is complete
    const float a = DS ? 0.0f : *amax;
    const float alpha = DS ? ds[0] : alpha_from_amax(Fp8<FMT>::FMAX, a);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *scale = DS ? ds[1] : __fdiv_rn(1.0f, alpha);
        flag_nonfinite(status, DS ? __float_as_uint(alpha) & 0x7FFFFFFFu : __float_as_uint(a) & 0x7FFFFFFFu);
    }
    return alpha;
}

// ---------------------------------------------------------------------------
// a3, rowwise only: flat streaming cast, 16 elements -> one 16-byte store.
// ---------------------------------------------------------------------------
template <int DT, int FMT, bool DS>
__global__ void __launch_bounds__(256) k_cs_cast_flat(const void *__restrict__ x, int64_t n,
                                                      const float *__restrict__ amax, const float *__restrict__ ds,
                                                      uint32_t *amax_rec, uint8_t *__restrict__ q,
                                                      float *__restrict__ scale, int32_t *status)
{
    constexpr int VEC = In<DT>::VEC;
    constexpr int VPC = 16 / VEC;   // 16-byte input vectors per 16-element chunk
    constexpr int U = 4;            // chunks in flight per thread
    const float alpha = cast_alpha<FMT, DS>(amax, ds, scale, status);
    uint32_t mx = 0;                // DS: max |x| bits seen by this thread
    const uint4 *xv = static_cast<const uint4 *>(x);
    const int64_t nc = n / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nc; i += U * stride) {
        uint4 v[U][VPC];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t c = nc - 1 - (i + u * stride);   // backwards: L2-resident data first
            if (c >= 0)
#pragma unroll
                for (int j = 0; j < VPC; j++) v[u][j] = ldg_stream(xv + c * VPC + j);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t c = nc - 1 - (i + u * stride);
            if (c < 0) break;
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < VPC; j++) {
                if (DS) mx = max(mx, absmax_bits<DT>(v[u][j]));
                chunk_fp8<DT, FMT>(v[u][j], alpha, o + j * (VEC / 4));
            }
            stg16(q + c * 16, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
    // the last n % 16 elements, one per thread of CTA 0
    if (blockIdx.x == 0 && threadIdx.x < n - nc * 16) {
        const int64_t t = nc * 16 + threadIdx.x;
        const float v = DT == BF16 ? __uint_as_float((uint32_t)static_cast<const uint16_t *>(x)[t] << 16)
                                   : static_cast<const float *>(x)[t];
        q[t] = (uint8_t)(cvt_fp8x4<FMT>(__fmul_rn(alpha, v), 0.f, 0.f, 0.f) & 0xFFu);
        mx = max(mx, __float_as_uint(v) & 0x7FFFFFFFu);
    }
    if (DS) cta_max_to(mx, amax_rec, status);
}

// ---------------------------------------------------------------------------
// a3 with the transposed copy, on the tile engine.  Per 128 x TC tile,
// thread (warp w, lane l) casts rows 8w..8w+7 of its 16-byte column chunk
// once; q_row leaves straight from registers, and the same codes, turned
// around by byte transposes, are parked in the consumed stage and written as
// full 128-byte q_colT rows.  Requires M % 16 == 0 and K % 16 == 0.
// ---------------------------------------------------------------------------
template <int DT, int FMT, bool DS>
__global__ void __launch_bounds__(kEngThreads, 1) k_cs_tiles(const __grid_constant__ CUtensorMap tmap, int64_t M, int64_t K,
                                                             const float *__restrict__ amax, const float *__restrict__ ds,
                                                             uint32_t *amax_rec, uint8_t *__restrict__ q_row,
                                                             uint8_t *__restrict__ q_colT, float *__restrict__ scale,
                                                             int32_t *status)
{
    constexpr int VEC = In<DT>::VEC, TC = 32 * VEC, CW = VEC / 4;
    const float alpha = cast_alpha<FMT, DS>(amax, ds, scale, status);
    uint32_t mx = 0;   // DS: max |x| bits of this thread's tile chunks (OOB fill is 0)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_m = (M + kTileRowsE - 1) / kTileRowsE, tiles_k = (K + TC - 1) / TC;

    run_tiles(&tmap, tiles_m, tiles_k, TC, true, status, [&](uint8_t *st, int64_t tm, int64_t tk) {
        const int64_t mb = tm * kTileRowsE, kb = tk * TC;
        const int64_t k = kb + lane * VEC, m0 = mb + 8 * warp;
        uint32_t code[8][CW];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const uint4 v = lds16(st + (8 * warp + j) * kRowBytes + lane * 16);
            if (DS) mx = max(mx, absmax_bits<DT>(v));
            chunk_fp8<DT, FMT>(v, alpha, code[j]);
        }
        if (q_row != nullptr && k < K) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (m0 + j >= M) break;
                uint8_t *dst = q_row + (m0 + j) * K + k;
                if (CW == 2) stg8(dst, code[j][0], code[j][CW - 1]);
                else stg4(dst, code[j][0]);
            }
        }
        if (q_colT == nullptr) return;
        __syncthreads();   // every read of the stage is done: park the transposed codes in it
        park_fp8T<VEC>(st, code, warp, lane);
        __syncthreads();
        copy_out_fp8T<VEC>(st, q_colT, M, K, mb, kb);
    });
    if (DS) cta_max_to(mx, amax_rec, status);
}

// ---------------------------------------------------------------------------
// Delayed scaling: the pair [alpha, s] for the next step from the window of
// N recorded amaxes (a ring; slot pos is the latest).  algo 0: the largest
// |entry| (bit patterns, a NaN entry wins); algo 1: |hist[pos]|.  Then the
// current-scaling rule (amax 0 -> 1, overflowing alpha -> FLT_MAX).
// ---------------------------------------------------------------------------
constexpr int kDsThreads = 256;

__global__ void __launch_bounds__(kDsThreads) k_ds_update(const float *__restrict__ hist, int64_t N, int64_t pos, int algo,
                                                          float fmax, float *__restrict__ ds)
{
    uint32_t m = 0;
    if (algo == 1) {
        if (threadIdx.x == 0) m = __float_as_uint(hist[pos]) & 0x7FFFFFFFu;
    } else {
        for (int64_t i = threadIdx.x; i < N; i += kDsThreads) m = max(m, __float_as_uint(hist[i]) & 0x7FFFFFFFu);
    }
    m = warp_max(m);
    __shared__ uint32_t red[kDsThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kDsThreads / 32 ? red[lane] : 0u;
        m = warp_max(m);
        if (lane == 0) {
            const float alpha = alpha_from_amax(fmax, __uint_as_float(m));
            ds[0] = alpha;
            ds[1] = __fdiv_rn(1.0f, alpha);
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

// Zeroes the amax word before the reduction (a kernel on the same stream: the
// next kernel starts right behind it, which a driver memset does not).
__global__ void k_zero_word(uint32_t *w, uint32_t *w2)
{
    griddep_launch_dependents();   // the reduction behind may start; it waits before its atomic
    *w = 0u;
    if (w2 != nullptr) *w2 = 0u;
}

cudaError_t launch_zero_word(float *w, cudaStream_t st, float *w2)
{
    k_zero_word<<<1, 1, 0, st>>>(reinterpret_cast<uint32_t *>(w), reinterpret_cast<uint32_t *>(w2));
    return cudaGetLastError();
}

cudaError_t launch_amax(const void *x, int dt, int64_t n, float *amax, int32_t *status, cudaStream_t st)
{
    (void)status;
    k_zero_word<<<1, 1, 0, st>>>(reinterpret_cast<uint32_t *>(amax), nullptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || n == 0) return e;
    const int vec = dt == BF16 ? 8 : 4;
    const int64_t nv = n / vec;
    int64_t blocks = (nv + (int64_t)kAmaxThreads * kAmaxUnroll - 1) / ((int64_t)kAmaxThreads * kAmaxUnroll);
    const int64_t cap = (int64_t)sm_count() * 8;   // two waves of the 4 resident CTAs: a shorter tail
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    uint32_t *w = reinterpret_cast<uint32_t *>(amax);
    return dt == BF16 ? launch_k(true, k_amax<BF16>, dim3((unsigned)blocks), dim3(kAmaxThreads), 0, st, x, n, w)
                      : launch_k(true, k_amax<F32>, dim3((unsigned)blocks), dim3(kAmaxThreads), 0, st, x, n, w);
}

template <int DT, int FMT, bool DS>
static cudaError_t cs_cast_t(const void *x, int64_t M, int64_t K, const float *amax, const float *ds, float *amax_rec,
                             uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st,
                             bool after_amax)
{
    const bool pdl = DS || after_amax;   // behind the zeroing kernel (DS) or the amax pass
    uint32_t *rec = reinterpret_cast<uint32_t *>(amax_rec);
    if (DS) {
        k_zero_word<<<1, 1, 0, st>>>(rec, nullptr);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (q_colT == nullptr) {
        const int64_t n = M * K, nc = n / 16;
        int64_t blocks = (nc + 4 * 256 - 1) / (4 * 256);
        const int64_t cap = (int64_t)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        return launch_k(pdl, k_cs_cast_flat<DT, FMT, DS>, dim3((unsigned)blocks), dim3(256), 0, st, x, n, amax, ds, rec,
                        q_row, scale, status);
    }
    constexpr int TC = 32 * In<DT>::VEC;
    alignas(64) CUtensorMap map;
    cudaError_t e = make_tile_map(&map, x, DT, M, K);
    if (e != cudaSuccess) return e;
    {
        const cudaError_t ea = engine_smem_ready<k_cs_tiles<DT, FMT, DS>>();
        if (ea != cudaSuccess) return ea;
    }
    const int64_t tiles = ((M + kTileRowsE - 1) / kTileRowsE) * ((K + TC - 1) / TC);
    const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
    return launch_k(pdl, k_cs_tiles<DT, FMT, DS>, dim3(grid), dim3(kEngThreads), kEngSmem, st, map, M, K, amax, ds, rec,
                    q_row, q_colT, scale, status);
}

template <bool DS>
static cudaError_t cast_dispatch(const void *x, int dt, int64_t M, int64_t K, int fmt, const float *amax, const float *ds,
                                 float *amax_rec, uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status,
                                 cudaStream_t st, bool after_amax)
{
#define CS_ARGS x, M, K, amax, ds, amax_rec, q_row, q_colT, scale, status, st, after_amax
    if (dt == BF16) return fmt == E4M3 ? cs_cast_t<BF16, E4M3, DS>(CS_ARGS) : cs_cast_t<BF16, E5M2, DS>(CS_ARGS);
    return fmt == E4M3 ? cs_cast_t<F32, E4M3, DS>(CS_ARGS) : cs_cast_t<F32, E5M2, DS>(CS_ARGS);
#undef CS_ARGS
}

cudaError_t launch_cs_cast(const void *x, int dt, int64_t M, int64_t K, int fmt, const float *amax,
                           uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st,
                           bool after_amax)
{
    return cast_dispatch<false>(x, dt, M, K, fmt, amax, nullptr, nullptr, q_row, q_colT, scale, status, st, after_amax);
}

cudaError_t launch_ds_cast(const void *x, int dt, int64_t M, int64_t K, int fmt, const float *ds, float *amax_rec,
                           uint8_t *q_row, uint8_t *q_colT, float *scale, int32_t *status, cudaStream_t st)
{
    return cast_dispatch<true>(x, dt, M, K, fmt, nullptr, ds, amax_rec, q_row, q_colT, scale, status, st, false);
}

cudaError_t launch_ds_update(const float *hist, int64_t N, int64_t pos, int algo, int fmt, float *ds, cudaStream_t st)
{
    k_ds_update<<<1, kDsThreads, 0, st>>>(hist, N, pos, algo, fmt == E4M3 ? Fp8<E4M3>::FMAX : Fp8<E5M2>::FMAX, ds);
    return cudaGetLastError();
}

// Diagnostic of the bounded waits: one warp waits on a barrier whose first
// phase needs an arrival that no thread makes, so every wait can only end by
// its time limit; each thread that gives up ORs Q_ST_TIMEOUT into *status.
// Nothing is in flight when the CTA exits.
__global__ void k_selftest_wait(int32_t *status, unsigned long long wait_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(&bar, 0u, wait_ns)) atomicOr(status, kStTimeout);
}

cudaError_t launch_selftest_wait(int32_t *status, unsigned long long wait_ns, cudaStream_t st)
{
    k_selftest_wait<<<1, 32, 0, st>>>(status, wait_ns);
    return cudaGetLastError();
}

cudaError_t launch_empty_scales(float *amax_out, float *scale, cudaStream_t st)
{
    k_empty_scales<<<1, 1, 0, st>>>(amax_out, scale);
    return cudaGetLastError();
}

}  // namespace qk
