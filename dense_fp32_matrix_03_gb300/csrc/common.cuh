// common.cuh -- device-side building blocks shared by the SGEMM kernels:
// mbarrier waits with an iteration bound, TMA tile loads, cp.async copies,
// the 128-byte shared-memory swizzle and the persistent grouped tile order.
//
// Everything here is inline PTX or plain CUDA written for sm_103a.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace sg {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete yet is
// suspended until it completes or about `hint_ns` nanoseconds pass, instead
// of returning at once: a waiting warp then takes no issue slots and no
// shared-memory bandwidth from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Suspend hint of the bounded waits (the wait still ends as soon as the
// phase completes).
constexpr uint32_t kWaitSleepNs = 200000;

// Per-CTA abort state kept in shared memory.  A wait that runs out of
// iterations records why in the device status word, raises the CTA's abort
// flag so that every other role stops waiting too, and reports failure.
struct Abort {
    volatile int *flag;     // shared memory, 0 = running
    unsigned int *status;   // global device status word
    long long limit;        // clock64 cycles a wait may spin
};

// Waits until the phase with the given parity of `bar` has completed.
// Returns false (and aborts the CTA) if the wait exceeds ab.limit cycles or
// another role of the CTA has aborted.  Critical-path waits poll; `sleep`
// waits, for roles that wait long off the critical path, suspend between
// polls so that they take no issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const Abort &ab,
                                          unsigned int code, bool sleep = false)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (sleep ? mbar_try_wait_sleep(bar, parity, kWaitSleepNs) : mbar_try_wait(bar, parity))
            return true;
        if (*ab.flag) return false;
        if (clock64() - t0 > ab.limit) {
            atomicOr(ab.status, code);
            *ab.flag = 1;
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag: used to let copies already in
// flight land before the CTA exits after an abort.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, long long limit)
{
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

// Warp-wide bounded wait: every lane polls the barrier (and so acquires the
// stage's contents itself); the lanes then agree on the outcome, keeping the
// warp converged whatever happens.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const Abort &ab,
                                          unsigned int code, int lane)
{
    (void)lane;
    const bool ok = mbar_wait(bar, parity, ab, code);
    return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------ producers

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *m, uint64_t *bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ---------------------------------------------------------------- cp.async

// Copies `src_bytes` (0..16) bytes and zero-fills the rest of 16 bytes.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Copies `src_bytes` (0 or 4) bytes and zero-fills the rest of 4 bytes.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// The mbarrier counts one (pre-declared) arrival when all of this thread's
// earlier cp.async copies have landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------------ layout

// Byte offset of element (row, k) in a tile of 32-float (128-byte) rows laid
// out with the 128-byte swizzle that TMA's SWIZZLE_128B mode writes: the
// 16-byte chunk index inside a row is XORed with the row index modulo 8.
// The tile base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_offset(int row, int k)
{
    return static_cast<uint32_t>(row * 128 + ((((k >> 2) ^ row) & 7) << 4) + ((k & 3) << 2));
}

// K extent of one pipeline stage: one 128-byte swizzle row of fp32.
constexpr int kTileK = 32;

// One operand tile by cp.async, spread over `nthr` threads.  KIN: tile rows
// are ROWS (M or N) rows of 32 k-values, swizzled; otherwise the tile is
// [32 k][ROWS] unswizzled.  Global element (r, k) of a K-inner operand is at
// base[r*ld + k]; of an M/N-inner operand at base[k*ld + r].  Out-of-range
// elements are zero-filled (source size 0), never read.
template <int ROWS, bool KIN, bool EVEN_K>
__device__ __forceinline__ void cp_async_tile(uint8_t *dst, const float *base, long long ld,
                                              int r0, int rlim, int k0, int K, bool vec4, int tid,
                                              int nthr)
{
    const uint32_t d0 = smem_u32(dst);
    if (vec4) {
        if (KIN) {
            constexpr int UNITS = ROWS * (kTileK / 4);
            for (int u = tid; u < UNITS; u += nthr) {
                const int r = u >> 3, c = u & 7;
                const int gr = r0 + r, gk = k0 + 4 * c;
                int nval = (gr < rlim) ? (EVEN_K ? 4 : min(4, K - gk)) : 0;
                nval = max(nval, 0);
                const float *src = nval ? base + gr * ld + gk : base;
                cp_async_16(d0 + sw128_offset(r, 4 * c), src, nval * 4);
            }
        } else {
            constexpr int UNITS = kTileK * (ROWS / 4);
            for (int u = tid; u < UNITS; u += nthr) {
                const int k = u / (ROWS / 4), c = u % (ROWS / 4);
                const int gk = k0 + k, gr = r0 + 4 * c;
                int nval = (EVEN_K || gk < K) ? min(4, rlim - gr) : 0;
                nval = max(nval, 0);
                const float *src = nval ? base + gk * ld + gr : base;
                cp_async_16(d0 + (k * ROWS + 4 * c) * 4, src, nval * 4);
            }
        }
    } else {
        if (KIN) {
            constexpr int UNITS = ROWS * kTileK;
            for (int u = tid; u < UNITS; u += nthr) {
                const int r = u >> 5, k = u & 31;
                const int gr = r0 + r, gk = k0 + k;
                const bool v = gr < rlim && (EVEN_K || gk < K);
                cp_async_4(d0 + sw128_offset(r, k), v ? base + gr * ld + gk : base, v ? 4 : 0);
            }
        } else {
            constexpr int UNITS = kTileK * ROWS;
            for (int u = tid; u < UNITS; u += nthr) {
                const int k = u / ROWS, r = u % ROWS;
                const int gk = k0 + k, gr = r0 + r;
                const bool v = gr < rlim && (EVEN_K || gk < K);
                cp_async_4(d0 + (k * ROWS + r) * 4, v ? base + gk * ld + gr : base, v ? 4 : 0);
            }
        }
    }
}

// --------------------------------------------------------------- scheduler

// Persistent grouped tile order.  Linear tile id t -> (q, tm, tn): batch
// outermost; inside a batch, GROUP_M rows of tiles are walked column by column
// so that CTAs running at the same time share A rows and B columns in L2.
struct TileCoord {
    int q, tm, tn;
};

__device__ __forceinline__ TileCoord tile_coord(long long t, const GemmParams &p)
{
    const long long per_q = static_cast<long long>(p.tiles_m) * p.tiles_n;
    TileCoord c;
    c.q = static_cast<int>(t / per_q);
    int r = static_cast<int>(t - c.q * per_q);
    const int in_group = p.group_m * p.tiles_n;
    const int g = r / in_group;
    const int first_m = g * p.group_m;
    const int gsize = min(p.tiles_m - first_m, p.group_m);
    const int rr = r - g * in_group;
    c.tm = first_m + rr % gsize;
    c.tn = rr / gsize;
    return c;
}

// One work unit of the persistent scheduler: a tile and its k-block slice.
struct WorkUnit {
    TileCoord tc;
    long long tile;   // linear tile index
    long long sidx;   // index among the split tiles (tile - dp_tiles); -1 if whole
    int slice;        // 0 .. splits-1 (0 if whole)
    int kb_lo, kb_hi; // k-blocks [kb_lo, kb_hi) of this unit (never empty)
    bool split;       // part of a split tile: hand the partial over
};

__device__ __forceinline__ WorkUnit work_unit(long long u, const GemmParams &p)
{
    WorkUnit w;
    if (p.splits <= 1 || u < p.dp_tiles) {
        w.tile = u;
        w.sidx = -1;
        w.slice = 0;
        w.kb_lo = 0;
        w.kb_hi = p.k_blocks;
        w.split = false;
    } else {
        const long long v = u - p.dp_tiles;
        w.sidx = v / p.splits;
        w.tile = p.dp_tiles + w.sidx;
        w.slice = static_cast<int>(v - w.sidx * p.splits);
        w.kb_lo = static_cast<int>((static_cast<long long>(w.slice) * p.k_blocks) / p.splits);
        w.kb_hi = static_cast<int>((static_cast<long long>(w.slice + 1) * p.k_blocks) / p.splits);
        w.split = true;
    }
    w.tc = tile_coord(w.tile, p);
    return w;
}

// Where a work unit's BM x BN result goes.  A whole tile goes to C with the
// caller's alpha and beta; one slice of a split tile goes, unscaled, to its
// own row-major BM x BN slot of the split-K workspace (slot
// sidx * splits + slice), from where the fix-up kernel sums the slices.
struct OutTile {
    float *base;        // element (0, 0) of the tile
    long long ld;       // row pitch in elements
    float alpha, beta;  // beta == 0: the destination is not read
    int rows, cols;     // valid extent: min(BM, M - m0), min(BN, N - n0)
    bool vec4;          // 16-byte accesses allowed (base and ld allow them)
};

template <int BM, int BN>
__device__ __forceinline__ OutTile out_tile(const GemmParams &p, const WorkUnit &wu)
{
    OutTile o;
    const int m0 = wu.tc.tm * BM, n0 = wu.tc.tn * BN;
    o.rows = min(BM, p.M - m0);
    o.cols = min(BN, p.N - n0);
    if (!wu.split) {
        o.base = p.C + wu.tc.q * p.sC + static_cast<long long>(m0) * p.ldc + n0;
        o.ld = p.ldc;
        o.alpha = p.alpha;
        o.beta = p.beta;
        o.vec4 = p.c_vec4 != 0;
    } else {
        o.base = p.ws_part + (wu.sidx * p.splits + wu.slice) * static_cast<long long>(BM * BN);
        o.ld = BN;
        o.alpha = 1.f;
        o.beta = 0.f;
        o.vec4 = true;
    }
    return o;
}

}  // namespace sg
