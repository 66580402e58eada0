// Tile engine: a persistent, TMA-fed, multi-stage pipeline that streams
// 128-row x 512-byte tiles of the input through shared memory.
//
// One CTA of 512 threads per SM.  Thread 0 keeps kStages tiles in flight:
// each is one cp.async.bulk.tensor.2d load (the tensor map's box is 128 rows
// x 512 bytes; rows or columns past the tensor's edge arrive as zeros) that
// completes on the stage's mbarrier.  Every thread waits on that mbarrier
// itself (its acquire makes the tile visible to the thread, so no CTA
// barrier is needed at the start of a tile), runs the recipe's tile body on
// the stage, and when all are done (barrier) thread 0 refills the stage with
// the tile kStages tiles ahead.  Bytes in flight per SM are set by the
// stages, not by registers or occupancy, so the bodies can spend registers
// on arithmetic.
//
// Every wait is bounded: a thread polls the stage barrier with try_wait and
// gives up after kWaitNs of %globaltimer.  A thread that gives up ORs
// Q_ST_TIMEOUT into the status word, raises the CTA's abort flag and runs
// the rest of the tile with the others (every barrier of the body is still
// reached by all threads; the outputs of such a launch are not meaningful).
// At the end of that tile the whole CTA sees the flag and leaves the loop:
// no further copy is issued.  Thread 0 then waits (bounded again) for every
// copy it issued and did not see complete, so that no copy is in flight when
// the CTA's shared memory goes away -- unless one of those waits also runs
// out, in which case the CTA exits anyway and the status word already says
// Q_ST_TIMEOUT.
#pragma once

#include <atomic>
#include <cuda.h>
#include "q_common.cuh"

namespace qk {

constexpr int kEngThreads = 512;
constexpr int kEngWarps = kEngThreads / 32;
constexpr int kStages = 3;
constexpr int kTileRowsE = 128;
constexpr int kRowBytes = 512;                          // one tile row in shared memory
constexpr int kTileBytes = kTileRowsE * kRowBytes;      // 64 KiB
constexpr int kEngSmem = kStages * kTileBytes;          // dynamic shared memory of an engine CTA
constexpr int32_t kStTimeout = 2;
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s

// The engine's dynamic shared memory exceeds the default per-CTA limit; the
// opt-in is a per-device attribute of each kernel, set once per device.
template <auto Kernel>
inline cudaError_t engine_smem_ready()
{
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kEngSmem);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

QD uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

QD void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
QD void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
QD void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

QD void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

QD bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done != 0;
}

QD unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Poll until the barrier's phase with this parity completes; false after
// limit_ns (kWaitNs unless given).
QD bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, unsigned long long limit_ns = kWaitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// One 2-D tile (x = first column in elements, y = first row) into shared memory.
QD void tma_load_tile(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

QD uint4 lds16(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Transposed FP8 codes of a tile, staged for full-line writes: each thread
// holds 8 rows (8w..8w+7) x VEC columns of codes, as VEC/4 words per row
// (byte c = column c).  4x4 byte transposes turn them into 8 bytes per column,
// parked at [column][128 rows] in `stage` with the 8-byte chunks XOR-swizzled
// by lane; after a barrier, copy_out_fp8T writes 128-byte q_colT rows.
template <int VEC> QD void park_fp8T(uint8_t *stage, const uint32_t (*code)[VEC / 4], int warp, int lane)
{
#pragma unroll
    for (int q = 0; q < VEC / 4; q++) {
        uint32_t lo[4], hi[4];
        transpose4x4(code[0][q], code[1][q], code[2][q], code[3][q], lo[0], lo[1], lo[2], lo[3]);
        transpose4x4(code[4][q], code[5][q], code[6][q], code[7][q], hi[0], hi[1], hi[2], hi[3]);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int col = lane * VEC + 4 * q + i;
            *reinterpret_cast<uint2 *>(stage + col * 128 + ((warp ^ (lane & 15)) * 8)) = make_uint2(lo[i], hi[i]);
        }
    }
}

// Writes the parked [TC][128] code tile as q_colT rows (8 threads x 16 bytes
// per 128-byte row; M % 16 == 0).  Chunks 2p and 2p+1 (rows 16p..16p+15)
// sit in the aligned pair of 8-byte slots 2p ^ (s & ~1), in swapped order
// when the swizzle s is odd.
template <int VEC>
QD void copy_out_fp8T(const uint8_t *stage, uint8_t *q_colT, int64_t M, int64_t K, int64_t mb, int64_t kb)
{
    constexpr int TC = 32 * VEC;
#pragma unroll
    for (int it = 0; it < TC * 8 / kEngThreads; it++) {
        const int idx = it * kEngThreads + threadIdx.x;
        const int col = idx >> 3, pr = idx & 7;
        const int s = (col / VEC) & 15;
        const int64_t kg = kb + col, mg = mb + 16 * pr;
        if (kg < K && mg < M) {
            uint4 v = *reinterpret_cast<const uint4 *>(stage + col * 128 + ((2 * pr) ^ (s & ~1)) * 8);
            if (s & 1) v = make_uint4(v.z, v.w, v.x, v.y);
            stg16(q_colT + kg * M + mg, v);
        }
    }
}

// Tiles of this CTA: t = blockIdx.x + i * gridDim.x (reversed when `reverse`,
// so that a second pass over a tensor meets the part the first pass left in
// L2 first).  body(stage, tm, tk) runs with all threads; it may use
// __syncthreads() and may overwrite its stage.
template <class Body>
__device__ __forceinline__ void run_tiles(const CUtensorMap *tmap, int64_t tiles_m, int64_t tiles_k, int tile_cols,
                                          bool reverse, int32_t *status, Body &&body)
{
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kStages];

    const int64_t ntiles = tiles_m * tiles_k;
    const int64_t count = ntiles > (int64_t)blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_of = [&](int64_t i) -> int64_t {
        const int64_t t = (int64_t)blockIdx.x + i * gridDim.x;
        return reverse ? ntiles - 1 - t : t;
    };
    auto issue = [&](int64_t i, int s) {
        const int64_t t = tile_of(i);
        const int64_t tm = t / tiles_k, tk = t - tm * tiles_k;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kTileBytes);
        tma_load_tile(dsm + s * kTileBytes, tmap, (int)(tk * tile_cols), (int)(tm * kTileRowsE), &full[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int64_t i = 0; i < count && i < kStages; i++) issue(i, (int)i);

    // Tile i is issued before iteration i - kStages + 1 at the latest, so when
    // the loop leaves after tile i the copies of tiles i + 1 .. i + kStages - 1
    // are outstanding, and tile i's own if thread 0's wait for it gave up.
    int64_t drain_from = -1, drain_to = -1;
    for (int64_t i = 0; i < count; i++) {
        const int s = (int)(i % kStages);
        const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((i / kStages) & 1));
        if (!ok && status != nullptr) atomicOr(status, kStTimeout);
        const int64_t t = tile_of(i);
        const int64_t tm = t / tiles_k, tk = t - tm * tiles_k;
        body(dsm + s * kTileBytes, tm, tk);
        // every thread is done with the stage; any wait of this tile that gave up stops the whole CTA
        if (__syncthreads_or(!ok)) {
            drain_from = ok ? i + 1 : i;
            drain_to = i + kStages - 1 < count - 1 ? i + kStages - 1 : count - 1;
            break;
        }
        if (threadIdx.x == 0 && i + kStages < count) {
            fence_proxy_async();   // generic-proxy accesses of the stage before the async-proxy refill
            issue(i + kStages, s);
        }
    }
    if (threadIdx.x == 0 && drain_from >= 0) {
        // copies still in flight land before the CTA's shared memory goes away
        for (int64_t j = drain_from; j <= drain_to; j++)
            (void)mbar_wait_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1));
    }
}

}  // namespace qk
