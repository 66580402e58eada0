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

// Tile geometry of an engine kernel: ROWS x 512-byte tiles, STAGES in
// flight, THREADS per CTA.  The default is one 512-thread CTA per SM with
// 128-row tiles; TileCfg<64, 256> runs two 256-thread CTAs per SM (each with
// its own stages), so that one CTA's barriers and latency-bound phases
// overlap the other's work.
template <int ROWS, int THREADS, int STAGES = 3> struct TileCfg {
    static constexpr int kRows = ROWS, kThreads = THREADS, kStages = STAGES;
    static constexpr int kTileBytes = ROWS * kRowBytes;
    static constexpr int kSmem = STAGES * kTileBytes;   // dynamic shared memory of the stages
};
using EngCfg = TileCfg<kTileRowsE, kEngThreads, kStages>;

// The engine's dynamic shared memory exceeds the default per-CTA limit; the
// opt-in is a per-device attribute of each kernel, set once per device.
// max_shared also asks for the largest shared-memory carveout (kernels that
// keep two CTAs per SM).
template <auto Kernel>
inline cudaError_t engine_smem_ready(int bytes = kEngSmem, bool max_shared = false)
{
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && max_shared)
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
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

// A 2-D tile from shared memory to global memory (x = first column in
// elements, y = first row; the parts of the box outside the tensor are not
// written), in this thread's bulk-async group.
QD void tma_store_tile(const CUtensorMap *map, const void *src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(map), "r"(x), "r"(y), "r"(smem_u32(src)) : "memory");
}
QD void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's committed bulk stores have finished reading shared memory.
QD void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's committed bulk stores are complete.
QD void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Barrier `id` (1..15) among `count` threads (whole warps).
QD void named_barrier(int id, int count) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory"); }

QD uint4 lds16(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }
// The same load, issued again even when the compiler could reuse an earlier
// one (a second pass over a stage re-reads it instead of keeping registers).
QD uint4 lds16_again(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
    return v;
}

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

// In-place transpose of an 8x8 nibble matrix: a[i] nibble j -> a[j] nibble i.
QD void transpose8x8_nibbles(uint32_t *a)
{
#pragma unroll
    for (int i = 0; i < 4; i++) {   // 4x4 blocks
        uint32_t t = ((a[i] >> 16) ^ a[i + 4]) & 0x0000FFFFu;
        a[i + 4] ^= t;
        a[i] ^= t << 16;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 4)
#pragma unroll
        for (int j = 0; j < 2; j++) {   // 2x2 blocks
            uint32_t t = ((a[i + j] >> 8) ^ a[i + j + 2]) & 0x00FF00FFu;
            a[i + j + 2] ^= t;
            a[i + j] ^= t << 8;
        }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {   // single nibbles
        uint32_t t = ((a[i] >> 4) ^ a[i + 1]) & 0x0F0F0F0Fu;
        a[i + 1] ^= t;
        a[i] ^= t << 4;
    }
}

// Transposed FP4 codes of a tile: col[c] holds, for column c of this
// thread's chunk, the 8 codes of rows 8w..8w+7 (row 8w in bits 3-0).  They
// are parked at [column][64 bytes] in the consumed stage (4-byte slot w,
// XOR-swizzled by lane) and written as q_colT rows by copy_out_fp4T.
template <int VEC> QD void park_fp4T(uint8_t *stage, const uint32_t *col, int warp, int lane)
{
#pragma unroll
    for (int c = 0; c < VEC; c++)
        *reinterpret_cast<uint32_t *>(stage + (lane * VEC + c) * 64 + ((warp ^ (lane & 15)) * 4)) = col[c];
}

// Writes the parked transposed FP4 codes of a ROWS-row tile as q_colT rows.
// Parking layout: [tile column][ROWS / 2 bytes], the ROWS / 8 4-byte slots of
// a column (slot sl = its rows 8 sl .. 8 sl + 7) XOR-swizzled by
// s = (column / VEC) & (ROWS / 8 - 1).  With M % 32 == 0 the rows go out as
// 16-byte pieces (ROWS / 32 per column): slots 4g..4g+3 sit in the aligned
// group 4g ^ (s & ~3), word k holding slot 4g + (k ^ (s & 3)).
template <int VEC, int ROWS = kTileRowsE, int THREADS = kEngThreads>
QD void copy_out_fp4T(const uint8_t *stage, uint8_t *q_colT, int64_t M, int64_t K, int64_t mb, int64_t kb)
{
    constexpr int TC = 32 * VEC, CB = ROWS / 2, SL = ROWS / 8, PC = ROWS / 32;
    if ((M & 31) == 0) {
#pragma unroll
        for (int it = 0; it < TC * PC / THREADS; it++) {
            const int idx = it * THREADS + threadIdx.x;
            const int col = idx / PC, g = idx % PC;   // rows 32g..32g+31 of the tile
            const int s = (col / VEC) & (SL - 1);
            const int64_t kg = kb + col, mg = mb + 32 * g;
            if (kg < K && mg < M) {
                uint4 w = *reinterpret_cast<const uint4 *>(stage + col * CB + ((4 * g) ^ (s & ~3)) * 4);
                if (s & 1) w = make_uint4(w.y, w.x, w.w, w.z);
                if (s & 2) w = make_uint4(w.z, w.w, w.x, w.y);
                stg16(q_colT + kg * (M / 2) + mg / 2, w);
            }
        }
        return;
    }
#pragma unroll
    for (int it = 0; it < TC * SL / THREADS; it++) {
        const int idx = it * THREADS + threadIdx.x;
        const int col = idx / SL, sl = idx % SL;   // slot sl = rows 8sl..8sl+7 of the tile
        const int64_t kg = kb + col, mg = mb + 8 * sl;
        if (kg < K && mg < M)
            stg4(q_colT + kg * (M / 2) + mg / 2,
                 *reinterpret_cast<const uint32_t *>(stage + col * CB + ((sl ^ ((col / VEC) & (SL - 1))) * 4)));
    }
}

// Columnwise block scales of a ROWS-row tile, sSB[g][col] for the 16-row
// group g of tile column col, written as sb_colT[kb + col][mb/16 + g]: one
// store of ROWS / 16 bytes per column when the whole tile height is inside
// the tensor and aligned, byte stores otherwise.
template <int TC, int ROWS = kTileRowsE, int THREADS = kEngThreads>
QD void copy_out_sbT(const uint8_t (*sSB)[TC], uint8_t *sb_colT, int64_t M, int64_t K, int64_t mb, int64_t kb)
{
    constexpr int G = ROWS / 16;
    const int64_t left = (M - mb) / 16;
    const int nb = left < G ? (int)left : G;
    for (int col = threadIdx.x; col < TC; col += THREADS) {
        const int64_t kg = kb + col;
        if (kg >= K) continue;
        uint8_t *dst = sb_colT + kg * (M / 16) + mb / 16;
        if (nb == G && (M % (16 * G)) == 0) {
            uint32_t w[G / 4] = {};
#pragma unroll
            for (int q = 0; q < G; q++) w[q / 4] |= (uint32_t)sSB[q][col] << (8 * (q & 3));
            if constexpr (G == 8) stg8(dst, w[0], w[1]);
            else stg4(dst, w[0]);
        } else {
            for (int q = 0; q < nb; q++) dst[q] = sSB[q][col];
        }
    }
}

// Tiles of this CTA (Cfg: tile rows, stages): t = blockIdx.x + i * gridDim.x (reversed when `reverse`,
// so that a second pass over a tensor meets the part the first pass left in
// L2 first).  pre() runs with all threads once the first kStages copies are
// issued and before the first tile is awaited (a kernel whose input tensor is
// ready but whose scalar inputs come from the kernel ahead of it can wait for
// those there, while its first tiles load).  body(stage, tm, tk) runs with
// all threads; it may use __syncthreads() and may overwrite its stage.
template <class Cfg = EngCfg, class Pre, class Body>
__device__ __forceinline__ void run_tiles(const CUtensorMap *tmap, int64_t tiles_m, int64_t tiles_k, int tile_cols,
                                          bool reverse, int32_t *status, Pre &&pre, Body &&body);

template <class Cfg = EngCfg, class Body>
__device__ __forceinline__ void run_tiles(const CUtensorMap *tmap, int64_t tiles_m, int64_t tiles_k, int tile_cols,
                                          bool reverse, int32_t *status, Body &&body)
{
    run_tiles<Cfg>(tmap, tiles_m, tiles_k, tile_cols, reverse, status, [] {}, static_cast<Body &&>(body));
}

template <class Cfg, class Pre, class Body>
__device__ __forceinline__ void run_tiles(const CUtensorMap *tmap, int64_t tiles_m, int64_t tiles_k, int tile_cols,
                                          bool reverse, int32_t *status, Pre &&pre, Body &&body)
{
    constexpr int kStages = Cfg::kStages, kTileBytes = Cfg::kTileBytes, kTileRowsE = Cfg::kRows;
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[kStages];

    const int64_t ntiles = tiles_m * tiles_k;
    const int64_t count = ntiles > (int64_t)blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    // Tile t = blockIdx.x + i * gridDim.x as (row, column) of the tile grid,
    // advanced without a division per tile: the stride gridDim.x is
    // q rows + r columns.  Reversed walks use (tiles_m - 1 - tm, tiles_k - 1 - tk).
    const int64_t tkd = tiles_k > 0 ? tiles_k : 1;   // an empty tensor has no tiles to walk
    const int64_t q = (int64_t)gridDim.x / tkd, r = (int64_t)gridDim.x - q * tkd;
    struct Cursor {
        int64_t tm, tk;
    };
    auto advance = [&](Cursor &c) {
        c.tk += r;
        c.tm += q;
        if (c.tk >= tiles_k) {
            c.tk -= tiles_k;
            c.tm += 1;
        }
    };
    Cursor first;
    first.tm = (int64_t)blockIdx.x / tkd;
    first.tk = (int64_t)blockIdx.x - first.tm * tkd;
    Cursor ahead = first;   // thread 0: the next tile to request
    auto issue = [&](int s) {
        const int64_t tm = reverse ? tiles_m - 1 - ahead.tm : ahead.tm, tk = reverse ? tiles_k - 1 - ahead.tk : ahead.tk;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kTileBytes);
        tma_load_tile(dsm + s * kTileBytes, tmap, (int)(tk * tile_cols), (int)(tm * kTileRowsE), &full[s]);
        advance(ahead);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int64_t i = 0; i < count && i < kStages; i++) issue((int)i);
    pre();

    // Tile i is issued before iteration i - kStages + 1 at the latest, so when
    // the loop leaves after tile i the copies of tiles i + 1 .. i + kStages - 1
    // are outstanding, and tile i's own if thread 0's wait for it gave up.
    int64_t drain_from = -1, drain_to = -1;
    Cursor cur = first;
    int s = 0;
    uint32_t parity = 0;
    for (int64_t i = 0; i < count; i++) {
        const bool ok = mbar_wait_bounded(&full[s], parity);
        if (!ok && status != nullptr) atomicOr(status, kStTimeout);
        body(dsm + s * kTileBytes, reverse ? tiles_m - 1 - cur.tm : cur.tm, reverse ? tiles_k - 1 - cur.tk : cur.tk);
        advance(cur);
        // every thread is done with the stage; any wait of this tile that gave up stops the whole CTA
        if (__syncthreads_or(!ok)) {
            drain_from = ok ? i + 1 : i;
            drain_to = i + kStages - 1 < count - 1 ? i + kStages - 1 : count - 1;
            break;
        }
        if (threadIdx.x == 0 && i + kStages < count) {
            fence_proxy_async();   // generic-proxy accesses of the stage before the async-proxy refill
            issue(s);
        }
        if (++s == kStages) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (threadIdx.x == 0 && drain_from >= 0) {
        // copies still in flight land before the CTA's shared memory goes away
        for (int64_t j = drain_from; j <= drain_to; j++)
            (void)mbar_wait_bounded(&full[j % kStages], (uint32_t)((j / kStages) & 1));
    }
}

}  // namespace qk
