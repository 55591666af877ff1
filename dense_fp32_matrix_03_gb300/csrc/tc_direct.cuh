// tc_direct.cuh -- tcgen05 tensor-core SGEMM whose converter warps read the
// operands straight from global memory.
//
// Same arithmetic as tc_tf32.cuh (3xTF32 hi/lo split or one TF32 pass, A
// planes in TMEM, B planes in shared memory as K-major 128-byte-swizzled
// tiles, fp32 accumulators in TMEM), without the raw shared-memory stage:
// in the TMA design every operand byte is written to shared memory by the
// copy engine and read back by a converter before the split planes are
// written, 64 of the 144 KB of shared-memory traffic per k-block.  Here each
// converter thread loads its share of the next k-block into registers while
// it converts the current one, and touches the k-block four ahead with an
// L2 prefetch so that the register loads hit L2.  Loads are 16 bytes wide
// where the operand allows it and scalar (masked) elsewhere, so operands TMA
// cannot describe (an odd row pitch, an unaligned base) take the same path.
//
// Warp roles (13 warps): warp 0 TMEM allocator and single-thread MMA issuer;
// warps 1-4 A converters (thread = A row = TMEM lane, warp w owns lanes
// 32*(w mod 4)...); warps 5-8 B converters; warps 9-12 epilogue (TMEM lane
// quarter = warp mod 4).
#pragma once

#include "tc_tf32.cuh"

namespace sg {
namespace tcd {

using tc::BK;
using tc::BM;
using tc::UK;

constexpr int kMmaWarp = 0;
constexpr int kAConvWarp0 = 1;                   // warps 1-4
constexpr int kBConvWarp0 = 5, kBConvWarps = 4;  // warps 5-8
constexpr int kEpiWarp0 = 9;                     // warps 9-12
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kConvWarps = 4 + kBConvWarps;      // arrivals that complete a stage
constexpr uint32_t kTmemCols = 512;
#ifndef SG_TCD_PREFETCH
#define SG_TCD_PREFETCH 4
#endif
constexpr int kPrefetchDist = SG_TCD_PREFETCH;   // k-blocks ahead for the L2 prefetch

template <int BN_, bool SPLIT3_, bool A_KIN_, bool B_KIN_>
struct Cfg {
    static constexpr int BN = BN_;
    static constexpr bool SPLIT3 = SPLIT3_, A_KIN = A_KIN_, B_KIN = B_KIN_;
    static constexpr int B_BYTES = BN * BK * 4;
    static constexpr int PLANES = SPLIT3 ? 2 : 1;         // hi (+ lo)
    static constexpr int SPLIT_BYTES = PLANES * B_BYTES;  // B planes of one stage
    // TMEM columns: two accumulator buffers of BN fp32 columns, then the A
    // planes of every stage (BK columns per plane, one row per lane).
    static constexpr int ACC_COLS = 2 * BN;
    static constexpr int A_COLS = PLANES * BK;
    static constexpr int STAGES = (static_cast<int>(kTmemCols) - ACC_COLS) / A_COLS;
    static constexpr int NBAR = 2 * STAGES + 4 + 1;
    static constexpr int EPI_BYTES = 4 * tc::kStageFloats * 4;  // epilogue staging (4 warps)
    static constexpr int SMEM_BYTES = STAGES * SPLIT_BYTES + EPI_BYTES + NBAR * 8 + 16 + 1024;
    static constexpr int OFF_BHI = 0, OFF_BLO = B_BYTES;
    static_assert(BN == 128, "one UMMA N per tile (BN = 128 keeps two accumulators in TMEM)");
    static_assert(STAGES >= 2, "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Walks the (work unit, k-block) sequence of one CTA.
struct KWalk {
    long long unit;
    int kb, kb_end;
    TileCoord tc;
    bool valid;

    __device__ __forceinline__ void load(const GemmParams &p)
    {
        valid = unit < p.num_units;
        if (valid) {
            const WorkUnit w = work_unit(unit, p);
            tc = w.tc;
            kb = w.kb_lo;
            kb_end = w.kb_hi;
        }
    }
    __device__ __forceinline__ void start(const GemmParams &p)
    {
        unit = blockIdx.x;
        load(p);
    }
    __device__ __forceinline__ void advance(const GemmParams &p)
    {
        if (!valid) return;
        if (++kb == kb_end) {
            unit += gridDim.x;
            load(p);
        }
    }
};

__device__ __forceinline__ float4 ldg4(const float *p)
{
    return __ldg(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ void prefetch_l2(const float *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// 32 consecutive values src[0..31] of a K-inner row segment starting at k0;
// values at k >= K are zero and never read.
__device__ __forceinline__ void load_row32(float (&x)[32], const float *src, int k0, int K,
                                           bool vec4)
{
    if (vec4 && k0 + BK <= K) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 v = ldg4(src + 4 * c);
            x[4 * c] = v.x;
            x[4 * c + 1] = v.y;
            x[4 * c + 2] = v.z;
            x[4 * c + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float v = 0.f;
            if (k0 + k < K) v = __ldg(src + k);
            x[k] = v;
        }
    }
}

// A converter thread's operand: row r of the A tile of k-block w, k along x.
template <bool KIN>
__device__ __forceinline__ void load_a(float (&x)[32], const GemmParams &p, const KWalk &w,
                                       int r)
{
    const int gm = w.tc.tm * BM + r, k0 = w.kb * BK;
    const float *Aq = p.A + w.tc.q * p.sA;
    if (gm >= p.M) {
#pragma unroll
        for (int k = 0; k < BK; ++k) x[k] = 0.f;
        return;
    }
    if (KIN) {
        load_row32(x, Aq + static_cast<long long>(gm) * p.lda + k0, k0, p.K, p.a_vec4 != 0);
    } else {
        // A stored K x M: element (m, k) at Aq[k*lda + m]; lanes read consecutive m
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float v = 0.f;
            if (k0 + k < p.K) v = __ldg(Aq + static_cast<long long>(k0 + k) * p.lda + gm);
            x[k] = v;
        }
    }
}

template <bool KIN>
__device__ __forceinline__ void prefetch_a(const GemmParams &p, const KWalk &w, int r)
{
    const int k0 = w.kb * BK;
    const float *Aq = p.A + w.tc.q * p.sA;
    if (KIN) {
        const int gm = w.tc.tm * BM + r;
        if (gm < p.M) prefetch_l2(Aq + static_cast<long long>(gm) * p.lda + k0);
    } else {
        // 32 k rows x 128 m = 128 lines of 128 bytes, one per thread
        const int k = k0 + (r >> 2), m = w.tc.tm * BM + (r & 3) * 32;
        if (k < p.K && m < p.M) prefetch_l2(Aq + static_cast<long long>(k) * p.lda + m);
    }
}

// B converter thread's operand (ct = 0..127).
//  K-inner B (stored N x K): x = the 32 k of plane row n = ct.
//  N-inner B (stored K x N): two 4 x 4 blocks, x[16*sh + 4*kk + i] =
//  B(k = 4*kb4(sh) + kk, n = 4*lane + i) with kb4 rotated by lane/2 so that
//  the plane stores of a quarter-warp hit eight distinct bank groups.
template <int BN>
__device__ __forceinline__ int b_kb4(int ct, int sh)
{
    const int warp = ct >> 5, lane = ct & 31;
    return (warp * 2 + sh + (lane >> 1)) & 7;
}

template <int BN, bool KIN>
__device__ __forceinline__ void load_b(float (&x)[32], const GemmParams &p, const KWalk &w,
                                       int ct)
{
    const int n0 = w.tc.tn * BN, k0 = w.kb * BK;
    const float *Bq = p.B + w.tc.q * p.sB;
    if (KIN) {
        const int gn = n0 + ct;
        if (gn >= p.N) {
#pragma unroll
            for (int k = 0; k < BK; ++k) x[k] = 0.f;
            return;
        }
        load_row32(x, Bq + static_cast<long long>(gn) * p.ldb + k0, k0, p.K, p.b_vec4 != 0);
    } else {
        static_assert(BN == 128, "one 4-column block per lane");
        const int lane = ct & 31;
        const int gn = n0 + 4 * lane;
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
            const int kb4 = b_kb4<BN>(ct, sh);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int gk = k0 + 4 * kb4 + kk;
                const float *src = Bq + static_cast<long long>(gk) * p.ldb + gn;
                float *d = &x[16 * sh + 4 * kk];
                if (gk < p.K && p.b_vec4 && gn + 3 < p.N) {
                    const float4 v = ldg4(src);
                    d[0] = v.x;
                    d[1] = v.y;
                    d[2] = v.z;
                    d[3] = v.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float v = 0.f;
                        if (gk < p.K && gn + i < p.N) v = __ldg(src + i);
                        d[i] = v;
                    }
                }
            }
        }
    }
}

template <int BN, bool KIN>
__device__ __forceinline__ void prefetch_b(const GemmParams &p, const KWalk &w, int ct)
{
    const int n0 = w.tc.tn * BN, k0 = w.kb * BK;
    const float *Bq = p.B + w.tc.q * p.sB;
    if (KIN) {
        const int gn = n0 + ct;
        if (gn < p.N) prefetch_l2(Bq + static_cast<long long>(gn) * p.ldb + k0);
    } else {
        // 32 k rows x BN n = 128 lines of 128 bytes, one per thread
        const int k = k0 + (ct >> 2), n = n0 + (ct & 3) * 32;
        if (k < p.K && n < p.N) prefetch_l2(Bq + static_cast<long long>(k) * p.ldb + n);
    }
}

// Writes this thread's values as hi (and lo) planes: A into its TMEM row
// (columns [t_hi, t_hi + 32) and [t_lo, ...)), B into the stage's K-major
// 128-byte-swizzled planes in shared memory.
template <bool SPLIT3>
__device__ __forceinline__ void store_a(const float (&x)[32], uint32_t t_hi, uint32_t t_lo)
{
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float h[16], l[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) tc::split_value<SPLIT3>(x[16 * half + k], h[k], l[k]);
        tc::tmem_st16(t_hi + half * 16, h);
        if (SPLIT3) tc::tmem_st16(t_lo + half * 16, l);
    }
}

__device__ __forceinline__ void sts4(uint32_t a, float x0, float x1, float x2, float x3)
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x0), "f"(x1), "f"(x2),
                 "f"(x3)
                 : "memory");
}

template <int BN, bool KIN, bool SPLIT3>
__device__ __forceinline__ void store_b(const float (&x)[32], uint32_t hi_a, uint32_t lo_a,
                                        int ct)
{
    if (KIN) {
        // plane row ct: chunk c (k = 4c..4c+3) at chunk c ^ (row mod 8)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t off = sw128_offset(ct, 4 * c);
            float h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) tc::split_value<SPLIT3>(x[4 * c + i], h[i], l[i]);
            sts4(hi_a + off, h[0], h[1], h[2], h[3]);
            if (SPLIT3) sts4(lo_a + off, l[0], l[1], l[2], l[3]);
        }
    } else {
        const int lane = ct & 31;
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
            const int kb4 = b_kb4<BN>(ct, sh);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t off = sw128_offset(4 * lane + i, 4 * kb4);
                float h[4], l[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::split_value<SPLIT3>(x[16 * sh + 4 * kk + i], h[kk], l[kk]);
                sts4(hi_a + off, h[0], h[1], h[2], h[3]);
                if (SPLIT3) sts4(lo_a + off, l[0], l[1], l[2], l[3]);
            }
        }
    }
}

template <class C>
struct Smem {
    uint8_t *split;  // STAGES x (B_hi | B_lo)
    float4 *epi;     // the epilogue warps' staging buffers
    uint64_t *split_full, *split_empty, *acc_full, *acc_empty, *mma_done;
    uint32_t *tmem_base;
    volatile int *abort_flag;
};

template <class C>
__global__ void __launch_bounds__(kThreads, 1) tcd_sgemm_kernel(const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Smem<C> sm;
    sm.split = base;
    sm.epi = reinterpret_cast<float4 *>(base + C::STAGES * C::SPLIT_BYTES);
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(base + C::STAGES * C::SPLIT_BYTES + C::EPI_BYTES);
    sm.split_full = bars;
    sm.split_empty = sm.split_full + C::STAGES;
    sm.acc_full = sm.split_empty + C::STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.mma_done = sm.acc_empty + 2;
    sm.tmem_base = reinterpret_cast<uint32_t *>(sm.mma_done + 1);
    sm.abort_flag = reinterpret_cast<volatile int *>(sm.tmem_base + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&sm.split_full[s], kConvWarps);
            mbar_init(&sm.split_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);
            mbar_init(&sm.acc_empty[b], 4);
        }
        mbar_init(sm.mma_done, 1);
        *sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(sm.tmem_base, kTmemCols);
        tc::tc_fence_before();
    }
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *sm.tmem_base;
    const Abort ab{sm.abort_flag, p.status, p.wait_limit};

    if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            tc::Ring<C::STAGES> sr;
            tc::Ring<2> acc;
            constexpr uint32_t idesc = tc::idesc_tf32<C::BN>();
            bool ok = true;
            bool any = false;
            for (long long u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                const WorkUnit wu = work_unit(u, p);
                if (!mbar_wait(&sm.acc_empty[acc.s], acc.ph ^ 1u, ab, kStatusWaitAcc)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc.s * C::BN);
                for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                    if (!mbar_wait(&sm.split_full[sr.s], sr.ph, ab, kStatusWaitConv)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t st = smem_u32(sm.split + sr.s * C::SPLIT_BYTES);
                    const uint32_t a_hi = tmem + C::ACC_COLS + sr.s * C::A_COLS;
                    const uint32_t a_lo = a_hi + BK;
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk) {
                        const uint32_t koff = kk * UK * 4;  // bytes along the 128-byte row
                        const uint64_t b_hi = tc::kmajor_sw128_desc(st + C::OFF_BHI + koff);
                        const uint32_t acc_in = (kb > wu.kb_lo || kk > 0) ? 1u : 0u;
                        if (C::SPLIT3) {
                            const uint64_t b_lo = tc::kmajor_sw128_desc(st + C::OFF_BLO + koff);
                            tc::umma_tf32_ts(d_tmem, a_lo + kk * UK, b_hi, idesc, acc_in);
                            tc::umma_tf32_ts(d_tmem, a_hi + kk * UK, b_lo, idesc, 1u);
                            tc::umma_tf32_ts(d_tmem, a_hi + kk * UK, b_hi, idesc, 1u);
                        } else {
                            tc::umma_tf32_ts(d_tmem, a_hi + kk * UK, b_hi, idesc, acc_in);
                        }
                    }
                    any = true;
                    tc::umma_commit(&sm.split_empty[sr.s]);  // frees the stage
                    sr.next();
                }
                if (!ok) break;
                tc::umma_commit(&sm.acc_full[acc.s]);  // accumulator ready for the epilogue
                acc.next();
            }
            // wait until every MMA issued has completed (TMEM is freed next)
            if (any) {
                tc::umma_commit(sm.mma_done);
                mbar_drain(sm.mma_done, 0, ab.limit);
            }
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ converters
        const bool is_a = warp < kBConvWarp0;
        const int quarter = warp & 3;  // TMEM lanes this warp may access (A converters)
        const int row = quarter * 32 + lane;
        const int ct = threadIdx.x - kBConvWarp0 * 32;
        KWalk cur, pf;
        cur.start(p);
        pf = cur;
        for (int i = 0; i < kPrefetchDist; ++i) pf.advance(p);
        float xa[32], xb[32];
        auto load = [&](float (&x)[32], const KWalk &w) {
            if (is_a)
                load_a<C::A_KIN>(x, p, w, row);
            else
                load_b<C::BN, C::B_KIN>(x, p, w, ct);
        };
        auto prefetch = [&](const KWalk &w) {
            if (is_a)
                prefetch_a<C::A_KIN>(p, w, row);
            else
                prefetch_b<C::BN, C::B_KIN>(p, w, ct);
        };
        tc::Ring<C::STAGES> sr;
        // Converts the k-block whose values are in `use` (position `cur`)
        // while the next k-block's loads, issued into `fill`, are in flight.
        auto step = [&](float (&use)[32], float (&fill)[32]) -> bool {
            KWalk nx = cur;
            nx.advance(p);
            if (nx.valid) load(fill, nx);
            if (pf.valid) {
                prefetch(pf);
                pf.advance(p);
            }
            if (!warp_wait(&sm.split_empty[sr.s], sr.ph ^ 1u, ab, kStatusWaitMma, lane))
                return false;
            if (is_a) {
                tc::tc_fence_after();  // the MMA that read this TMEM stage has completed
                const uint32_t t_hi = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                      C::ACC_COLS + sr.s * C::A_COLS;
                store_a<C::SPLIT3>(use, t_hi, t_hi + BK);
                tc::tmem_wait_st();
                tc::tc_fence_before();  // our TMEM stores -> visible to the MMA
            } else {
                const uint32_t st = smem_u32(sm.split + sr.s * C::SPLIT_BYTES);
                store_b<C::BN, C::B_KIN, C::SPLIT3>(use, st + C::OFF_BHI, st + C::OFF_BLO, ct);
                tc::fence_proxy_async_smem();  // our stores -> visible to the tensor core
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.split_full[sr.s]);
            sr.next();
            cur = nx;
            return true;
        };
        if (cur.valid) load(xa, cur);
        while (cur.valid) {
            if (!step(xa, xb) || !cur.valid) break;
            if (!step(xb, xa)) break;
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int r0 = q * 32;  // this warp's first row
        float4 *stage = sm.epi + q * (tc::kStageFloats / 4);
        tc::Ring<2> acc;
        for (long long u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const WorkUnit wu = work_unit(u, p);
            // C, or this slice's workspace slot (unscaled) when the tile is split
            const OutTile o = out_tile<BM, C::BN>(p, wu);
            tc::prefetch_c_rows(o, r0, lane);
            int w = 1;
            if (lane == 0) w = mbar_wait(&sm.acc_full[acc.s], acc.ph, ab, kStatusWaitAcc, true);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            mbar_drain(&sm.acc_full[acc.s], acc.ph, ab.limit);
            tc::tc_fence_after();
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc.s * C::BN);
#pragma unroll 1
            for (int c0 = 0; c0 < C::BN; c0 += 32) {
                float v[32];
                tc::tmem_ld32(tbase + c0, v);  // all lanes take part, rows in range or not
                tc::store_chunk_staged(o, r0, c0, v, stage, lane);
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[acc.s]);
            acc.next();
        }
    }

    // ---- teardown: every role is done; free TMEM
    tc::tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace tcd
}  // namespace sg
