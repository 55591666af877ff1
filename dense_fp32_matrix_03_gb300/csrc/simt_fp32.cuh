// simt_fp32.cuh -- the FP32 CUDA-core SGEMM kernel.
//
// C = alpha * op(A) @ op(B) + beta * C on the FP32 FFMA pipe, following the
// ladder of "From 1% to 94% of cuBLAS, one kernel at a time"
// (arpit2412.github.io/blog/cuda-sgemm.html): shared-memory cache blocking,
// 2D register blocking, float4 (128-bit) shared and global accesses,
// warptiling, and the "future work" the page lists (double buffering,
// swizzled conflict-free layouts, hardware copy engines, warp
// specialisation), built for sm_103a:
//
//  * one producer warp fills a STAGES-deep ring of shared-memory stages.
//    With TMA it issues two tiled tensor loads per stage (out-of-bounds rows,
//    columns and the K tail are zero-filled by the copy engine, so no mask is
//    evaluated in the main loop); for operands TMA cannot describe (a row
//    pitch that is not a multiple of 16 bytes, an unaligned base) it copies
//    with cp.async, masked, into the same layout.  An mbarrier per stage
//    signals "full"; another signals "empty" when the consumers are done.
//  * operands whose contiguous dimension is K ("K-inner": A, or B when
//    transposed) are stored as 32-float rows with the 128-byte swizzle, so a
//    warp's 128-bit loads of eight different rows at the same k hit eight
//    distinct 16-byte bank groups; operands whose contiguous dimension is M
//    or N are stored [k][m|n] unswizzled and read as 128-bit loads along the
//    row, as the page's kernel 6 does by transposing As.
//  * each consumer warp owns a WM x WN warp tile; its 32 lanes form an 8 x 4
//    grid and each lane accumulates (WM/32) x (WN/16) sub-blocks of 4 x 4
//    outputs in registers (the page's kernel 10 warptiling).  K is walked in
//    groups of 4 so that one 128-bit load of a K-inner row yields four k.
//  * tiles are visited in a persistent, grouped order (one CTA per SM).
//  * the epilogue fuses alpha and beta: C is read only when beta != 0.
#pragma once

#include "common.cuh"

namespace sg {

constexpr int kBK = 32;  // K per pipeline stage (one 128-byte swizzle row of fp32)

template <int BM_, int BN_, int WM_, int WN_, int STAGES_>
struct SimtCfg {
    static constexpr int BM = BM_, BN = BN_, WM = WM_, WN = WN_, STAGES = STAGES_;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    static constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
    static constexpr int WMITER = WM / 32, WNITER = WN / 16;
    static constexpr int TM = 4 * WMITER, TN = 4 * WNITER;
    static constexpr int A_BYTES = BM * kBK * 4, B_BYTES = BN * kBK * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int BAR_BYTES = 2 * STAGES * 8 + 16;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
    static_assert(BM % WM == 0 && BN % WN == 0 && WM % 32 == 0 && WN % 16 == 0, "tile shape");
    static_assert(BM <= 256 && BN <= 256, "a TMA box spans at most 256 rows");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Bounded wait that ignores the abort flag: used to let copies already in
// flight land before the CTA exits after an abort.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, long long limit)
{
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

// Warp-wide bounded wait: lane 0 spins (bounded), the verdict is broadcast,
// then every lane observes the completed phase itself (which returns at once)
// so that each lane acquires the stage's contents.  Keeps the warp converged
// whatever the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const Abort &ab,
                                          unsigned int code, int lane)
{
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, ab, code) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_drain(bar, parity, ab.limit);
    return ok != 0;
}

// ------------------------------------------------------------ producers

template <class Cfg, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void simt_tma_producer(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                                  const GemmParams &p, uint8_t *smem,
                                                  uint64_t *full, uint64_t *empty,
                                                  const Abort &ab)
{
    tma_prefetch_desc(tmA);
    tma_prefetch_desc(tmB);
    long long it = 0;
    bool ok = true;
    for (long long t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, p);
        const int m0 = tc.tm * Cfg::BM, n0 = tc.tn * Cfg::BN;
        const int qa = tc.q * p.a_q_step, qb = tc.q * p.b_q_step;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
            const int s = static_cast<int>(it % Cfg::STAGES);
            const uint32_t ph = static_cast<uint32_t>((it / Cfg::STAGES) & 1);
            if (!mbar_wait(&empty[s], ph ^ 1u, ab, kStatusWaitEmpty)) {
                ok = false;
                break;
            }
            uint8_t *sa = smem + s * Cfg::STAGE_BYTES;
            uint8_t *sb = sa + Cfg::A_BYTES;
            mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
            const int k0 = kb * kBK;
            if (A_KIN) tma_load_3d(sa, tmA, &full[s], k0, m0, qa);
            else       tma_load_3d(sa, tmA, &full[s], m0, k0, qa);
            if (B_KIN) tma_load_3d(sb, tmB, &full[s], k0, n0, qb);
            else       tma_load_3d(sb, tmB, &full[s], n0, k0, qb);
        }
    }
    if (!ok) {  // let the copies already issued land before leaving
        for (long long j = it - 1; j >= 0 && j >= it - Cfg::STAGES; --j)
            mbar_drain(&full[j % Cfg::STAGES], static_cast<uint32_t>((j / Cfg::STAGES) & 1),
                       ab.limit);
    }
}

// One operand tile by cp.async.  KIN: tile rows are `rows` (M or N) of 32
// k-values, swizzled; otherwise the tile is [32 k][ROWS] unswizzled.
// Global element (r, k) of a K-inner operand is at base[r*ld + k]; of an
// M/N-inner operand at base[k*ld + r].
template <int ROWS, bool KIN, bool EVEN_K>
__device__ __forceinline__ void cp_async_tile(uint8_t *dst, const float *base, long long ld,
                                              int r0, int rlim, int k0, int K, bool vec4,
                                              int lane)
{
    const uint32_t d0 = smem_u32(dst);
    if (vec4) {
        if (KIN) {
            constexpr int UNITS = ROWS * (kBK / 4);
#pragma unroll 4
            for (int u = lane; u < UNITS; u += 32) {
                const int r = u >> 3, c = u & 7;
                const int gr = r0 + r, gk = k0 + 4 * c;
                int nval = (gr < rlim) ? (EVEN_K ? 4 : min(4, K - gk)) : 0;
                nval = max(nval, 0);
                const float *src = nval ? base + gr * ld + gk : base;
                cp_async_16(d0 + sw128_offset(r, 4 * c), src, nval * 4);
            }
        } else {
            constexpr int UNITS = kBK * (ROWS / 4);
#pragma unroll 4
            for (int u = lane; u < UNITS; u += 32) {
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
            constexpr int UNITS = ROWS * kBK;
#pragma unroll 4
            for (int u = lane; u < UNITS; u += 32) {
                const int r = u >> 5, k = u & 31;
                const int gr = r0 + r, gk = k0 + k;
                const bool v = gr < rlim && (EVEN_K || gk < K);
                cp_async_4(d0 + sw128_offset(r, k), v ? base + gr * ld + gk : base, v ? 4 : 0);
            }
        } else {
            constexpr int UNITS = kBK * ROWS;
#pragma unroll 4
            for (int u = lane; u < UNITS; u += 32) {
                const int k = u / ROWS, r = u % ROWS;
                const int gk = k0 + k, gr = r0 + r;
                const bool v = gr < rlim && (EVEN_K || gk < K);
                cp_async_4(d0 + (k * ROWS + r) * 4, v ? base + gk * ld + gr : base, v ? 4 : 0);
            }
        }
    }
}

template <class Cfg, bool A_KIN, bool B_KIN, bool EVEN_K>
__device__ __forceinline__ void simt_cpasync_producer(const GemmParams &p, uint8_t *smem,
                                                      uint64_t *full, uint64_t *empty,
                                                      const Abort &ab, int lane)
{
    long long it = 0;
    bool ok = true;
    for (long long t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, p);
        const int m0 = tc.tm * Cfg::BM, n0 = tc.tn * Cfg::BN;
        const float *Aq = p.A + tc.q * p.sA;
        const float *Bq = p.B + tc.q * p.sB;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
            const int s = static_cast<int>(it % Cfg::STAGES);
            const uint32_t ph = static_cast<uint32_t>((it / Cfg::STAGES) & 1);
            if (!warp_wait(&empty[s], ph ^ 1u, ab, kStatusWaitEmpty, lane)) {
                ok = false;
                break;
            }
            uint8_t *sa = smem + s * Cfg::STAGE_BYTES;
            uint8_t *sb = sa + Cfg::A_BYTES;
            const int k0 = kb * kBK;
            cp_async_tile<Cfg::BM, A_KIN, EVEN_K>(sa, Aq, p.lda, m0, p.M, k0, p.K,
                                                  p.a_vec4 != 0, lane);
            cp_async_tile<Cfg::BN, B_KIN, EVEN_K>(sb, Bq, p.ldb, n0, p.N, k0, p.K,
                                                  p.b_vec4 != 0, lane);
            cp_async_arrive_noinc(&full[s]);
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------- consumer

template <class Cfg, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void simt_consumer(const GemmParams &p, uint8_t *smem, uint64_t *full,
                                              uint64_t *empty, const Abort &ab, int cw, int lane)
{
    constexpr int WMITER = Cfg::WMITER, WNITER = Cfg::WNITER, TM = Cfg::TM, TN = Cfg::TN;
    const int wm0 = (cw / Cfg::WARPS_N) * Cfg::WM;
    const int wn0 = (cw % Cfg::WARPS_N) * Cfg::WN;
    const int lr = lane >> 2, lc = lane & 3;

    // Rows/columns (inside the CTA tile) of this lane's outputs.  K-inner
    // operands interleave the lane rows (stride 8 / 4) so that the lanes of a
    // load instruction touch consecutive swizzled rows; M/N-inner operands give
    // each lane 4 consecutive elements (one 128-bit load).
    auto row_of = [&](int wm, int i) {
        return wm0 + wm * 32 + (A_KIN ? i * 8 + lr : lr * 4 + i);
    };
    auto col_of = [&](int wn, int j) {
        return wn0 + wn * 16 + (B_KIN ? j * 4 + lc : lc * 4 + j);
    };

    long long it = 0;
    for (long long t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, p);
        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
            const int s = static_cast<int>(it % Cfg::STAGES);
            const uint32_t ph = static_cast<uint32_t>((it / Cfg::STAGES) & 1);
            if (!warp_wait(&full[s], ph, ab, kStatusWaitFull, lane)) return;
            const uint8_t *sa = smem + s * Cfg::STAGE_BYTES;
            const uint8_t *sb = sa + Cfg::A_BYTES;
#pragma unroll 2
            for (int g = 0; g < kBK / 4; ++g) {
                float a[4][TM], b[4][TN];
                if (A_KIN) {
#pragma unroll
                    for (int wm = 0; wm < WMITER; ++wm)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 v = *reinterpret_cast<const float4 *>(
                                sa + sw128_offset(row_of(wm, i), 4 * g));
                            a[0][wm * 4 + i] = v.x;
                            a[1][wm * 4 + i] = v.y;
                            a[2][wm * 4 + i] = v.z;
                            a[3][wm * 4 + i] = v.w;
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int wm = 0; wm < WMITER; ++wm) {
                            const float4 v = *reinterpret_cast<const float4 *>(
                                sa + ((4 * g + kk) * Cfg::BM + row_of(wm, 0)) * 4);
                            a[kk][wm * 4 + 0] = v.x;
                            a[kk][wm * 4 + 1] = v.y;
                            a[kk][wm * 4 + 2] = v.z;
                            a[kk][wm * 4 + 3] = v.w;
                        }
                }
                if (B_KIN) {
#pragma unroll
                    for (int wn = 0; wn < WNITER; ++wn)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 v = *reinterpret_cast<const float4 *>(
                                sb + sw128_offset(col_of(wn, j), 4 * g));
                            b[0][wn * 4 + j] = v.x;
                            b[1][wn * 4 + j] = v.y;
                            b[2][wn * 4 + j] = v.z;
                            b[3][wn * 4 + j] = v.w;
                        }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int wn = 0; wn < WNITER; ++wn) {
                            const float4 v = *reinterpret_cast<const float4 *>(
                                sb + ((4 * g + kk) * Cfg::BN + col_of(wn, 0)) * 4);
                            b[kk][wn * 4 + 0] = v.x;
                            b[kk][wn * 4 + 1] = v.y;
                            b[kk][wn * 4 + 2] = v.z;
                            b[kk][wn * 4 + 3] = v.w;
                        }
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int j = 0; j < TN; ++j)
                            acc[i][j] = fmaf(a[kk][i], b[kk][j], acc[i][j]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // ---- epilogue: C = alpha * acc + beta * C, masked at the M/N edges
        const int mt = tc.tm * Cfg::BM, nt = tc.tn * Cfg::BN;
        float *Cq = p.C + tc.q * p.sC;
        const bool use_beta = p.beta != 0.f;
#pragma unroll
        for (int wm = 0; wm < WMITER; ++wm)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = mt + row_of(wm, i);
                if (r >= p.M) continue;
                float *crow = Cq + r * p.ldc;
#pragma unroll
                for (int wn = 0; wn < WNITER; ++wn) {
                    const float *av = &acc[wm * 4 + i][wn * 4];
                    if (!B_KIN) {
                        const int c0 = nt + col_of(wn, 0);
                        if (p.c_vec4 && c0 + 3 < p.N) {
                            float4 o;
                            o.x = p.alpha * av[0];
                            o.y = p.alpha * av[1];
                            o.z = p.alpha * av[2];
                            o.w = p.alpha * av[3];
                            float4 *dst = reinterpret_cast<float4 *>(crow + c0);
                            if (use_beta) {
                                const float4 old = *dst;
                                o.x = fmaf(p.beta, old.x, o.x);
                                o.y = fmaf(p.beta, old.y, o.y);
                                o.z = fmaf(p.beta, old.z, o.z);
                                o.w = fmaf(p.beta, old.w, o.w);
                            }
                            *dst = o;
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int c = c0 + j;
                                if (c < p.N) {
                                    float o = p.alpha * av[j];
                                    if (use_beta) o = fmaf(p.beta, crow[c], o);
                                    crow[c] = o;
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int c = nt + col_of(wn, j);
                            if (c < p.N) {
                                float o = p.alpha * av[j];
                                if (use_beta) o = fmaf(p.beta, crow[c], o);
                                crow[c] = o;
                            }
                        }
                    }
                }
            }
    }
}

// ---------------------------------------------------------------- kernel

template <class Cfg, bool A_KIN, bool B_KIN, bool USE_TMA, bool EVEN_K>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    simt_sgemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + Cfg::STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], USE_TMA ? 1u : 32u);
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Abort ab{abort_flag, p.status, p.wait_limit};

    if (warp == Cfg::CONSUMER_WARPS) {
        if (USE_TMA) {
            if (lane == 0) simt_tma_producer<Cfg, A_KIN, B_KIN>(&tmA, &tmB, p, smem, full, empty, ab);
        } else {
            simt_cpasync_producer<Cfg, A_KIN, B_KIN, EVEN_K>(p, smem, full, empty, ab, lane);
        }
    } else {
        simt_consumer<Cfg, A_KIN, B_KIN>(p, smem, full, empty, ab, warp, lane);
    }
    __syncwarp();
    __syncthreads();
}

}  // namespace sg
