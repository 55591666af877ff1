// tc_pair.cuh -- the tcgen05 SGEMM kernel on CTA pairs (3xTF32 and TF32).
//
// Same arithmetic as tc_tf32.cuh (hi/lo split, three kind::tf32 MMAs per
// k step for 3xTF32, one for TF32), on 256 x 128 output tiles computed by a
// cluster of two CTAs on two multiprocessors with cta_group::2 MMAs
// (M = 256, N = 128, K = 8):
//   - each CTA loads, splits and keeps in its own TMEM the A rows of its
//     half of the tile (128 rows), as the single-CTA kernel does;
//   - each CTA loads and splits only HALF of the B tile (64 of its 128
//     rows of B^T) into its own shared memory; one MMA reads both halves;
//   - one thread of the even CTA issues every MMA; its commits arrive on the
//     barriers of both CTAs (multicast), and both CTAs' converters and
//     epilogue warps arrive on the even CTA's barriers (remote arrives).
// Per CTA and 32-wide k-block that halves the B work: 24 KB of TMA writes
// (A 16 + B 8), 24 KB of converter reads and 16 KB of B-plane writes,
// against 32 + 32 + 32 KB for a 128 x 128 tile on one CTA (each CTA's
// tensor core still reads the whole B tile, half of it from the other CTA),
// and 25% less L2 -> shared-memory traffic per flop.  Measured on GB300 at
// 4092^3 against the single-CTA 128 x 128 kernel it replaces: 3xTF32
// 238.7 -> 276 TFLOP/s, TF32 316.6 -> 464.
//
// Warps and barriers as in tc_tf32.cuh.  Barriers that both CTAs arrive on
// live in the even CTA (split_full: 16 converter warps; acc_empty: 8
// epilogue warps); the others are per CTA.  Waits on barriers another CTA
// signals use cluster-scope acquire.  Every wait is bounded; the CTAs meet
// at a cluster barrier before they free their TMEM (jointly) and exit, so
// that neither leaves while the other may still touch its shared memory.
#pragma once

#include "tc_tf32.cuh"

// A pipeline stage covers SG_TCP_KSUB k-blocks of 32 (one 128-byte swizzle
// row of fp32 each): the MMA thread's per-stage work (wait, fence, commit)
// leaves the tensor pipe idle for a few hundred cycles whatever the stage's
// size, since its queue holds little more than the MMA in flight, so longer
// stages waste less.  Ring depths (raw fp32 tiles / split stages): TMEM
// holds (512 - 256) / (32 * KSUB * planes) split stages of A planes beside
// the two accumulators.
#ifndef SG_TCP_KSUB
#define SG_TCP_KSUB 2
#endif
// the wide (256 x 256) configuration's sub-blocks per stage and ring depths
// (measured on GB300, TF32 4092^3 nn / nt, TFLOP/s: 1/4/4 556/428, 1/5/4
// 543/424, 1/4/6 561/431, 2/2/2 520/441, 2/2/3 526/442; the epilogue's
// staging buffer takes the room of the sixth split stage)
#ifndef SG_TCP_WIDE_KSUB
#define SG_TCP_WIDE_KSUB 1
#define SG_TCP_WIDE_RAW 4
#define SG_TCP_WIDE_SPLIT 5
#endif
#ifndef SG_TCP_RAW3
#if SG_TCP_KSUB == 2
#define SG_TCP_RAW3 3
#define SG_TCP_SPLIT3 2
#define SG_TCP_RAW1 3
#define SG_TCP_SPLIT1 4
#else
#define SG_TCP_RAW3 6
#define SG_TCP_SPLIT3 4
#define SG_TCP_RAW1 6
#define SG_TCP_SPLIT1 8
#endif
#endif

namespace sg {
namespace tcp {

using tc::BK;
using tc::kAConvWarp0;
using tc::kBConvThreads;
using tc::kBConvWarp0;
using tc::kConvWarps;
using tc::kEpiWarp0;
using tc::kThreads;
using tc::kTmemCols;
using tc::Ring;
using tc::UK;

constexpr int BM = 128;      // rows of C per CTA
constexpr int PM = 2 * BM;   // rows per pair tile (the MMA's M)

// WIDE: 256 x 256 pair tiles (MMA N = 256) with one accumulator buffer and
// 32-wide stages -- for plain TF32, whose 256 x 128 tiles are bound by L2 ->
// shared-memory traffic (25% less per flop here; measured on GB300, TF32
// 4092^3 nn 460 -> 561 TFLOP/s); the accumulator is then drained before the
// next tile's MMAs start.  Otherwise (3xTF32, bound by the MMA issue, not
// by L2) 256 x 128 tiles, two accumulator buffers, SG_TCP_KSUB sub-blocks
// per stage.
template <bool SPLIT3_, bool A_KIN_, bool B_KIN_, bool WIDE_ = false>
struct Cfg {
    static constexpr bool SPLIT3 = SPLIT3_, A_KIN = A_KIN_, B_KIN = B_KIN_, WIDE = WIDE_;
    static constexpr int BN = WIDE ? 256 : 128;   // columns per pair tile (the MMA's N)
    static constexpr int HN = BN / 2;             // rows of B^T each CTA holds
    static constexpr int KSUB = WIDE ? SG_TCP_WIDE_KSUB : SG_TCP_KSUB;  // 32-wide sub-blocks
    static constexpr int STAGE_K = KSUB * BK;
    static constexpr int ACC_BUFS = WIDE ? 1 : 2;
    static constexpr int SUB_A = BM * BK * 4;   // raw A of one 32-wide sub-block
    static constexpr int SUB_B = HN * BK * 4;   // raw B of one sub-block
    static constexpr int A_BYTES = KSUB * SUB_A;
    static constexpr int B_BYTES = KSUB * SUB_B;
    static constexpr int RAW_BYTES = A_BYTES + B_BYTES;
    static constexpr int PLANES = SPLIT3 ? 2 : 1;
    static constexpr int SUB_SPLIT = PLANES * SUB_B;  // B planes of one sub-block
    static constexpr int SPLIT_BYTES = KSUB * SUB_SPLIT;
    static constexpr int RAW_STAGES =
        WIDE ? SG_TCP_WIDE_RAW : (SPLIT3 ? SG_TCP_RAW3 : SG_TCP_RAW1);
    static constexpr int SPLIT_STAGES =
        WIDE ? SG_TCP_WIDE_SPLIT : (SPLIT3 ? SG_TCP_SPLIT3 : SG_TCP_SPLIT1);
    static constexpr int ACC_COLS = ACC_BUFS * BN;
    static constexpr int SUB_COLS = PLANES * BK;      // TMEM A columns of one sub-block
    static constexpr int A_COLS = KSUB * SUB_COLS;
    static constexpr int NBAR = 2 * RAW_STAGES + 2 * SPLIT_STAGES + 4 + 1;
    // the four epilogue warps' staging buffers (tc::store_chunk_staged)
    static constexpr int EPI_BYTES = 4 * tc::kStageFloats * 4;
    static constexpr int SMEM_BYTES = RAW_STAGES * RAW_BYTES + SPLIT_STAGES * SPLIT_BYTES +
                                      EPI_BYTES + NBAR * 8 + 16 + 1024;
    static_assert(ACC_COLS + SPLIT_STAGES * A_COLS <= static_cast<int>(kTmemCols), "TMEM columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    // a sub-block's split planes: B_hi | B_lo
    static constexpr int OFF_BHI = 0, OFF_BLO = SUB_B;
    // Instruction descriptor: kind::tf32, fp32 accumulate, both operands
    // K-major, M = 256 (two CTAs), N = BN.
    static constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                                      (static_cast<uint32_t>(BN >> 3) << 17) |
                                      (static_cast<uint32_t>(PM >> 4) << 24);
};

// Plain TF32 runs on the wide tiles when K is at least this long: with a
// shorter K each tile is short, and the wide configuration's undrained
// single accumulator and fewer tiles per wave cost more than its lighter
// traffic saves (measured on GB300, TF32 wide / narrow, TFLOP/s: 4092^3
// 574 / 490, 2048^3 396 / 336, 1024^3 95 / 105, batched 1024 x 1024 x 512
// 224 / 240).
constexpr int kWideMinK = 1536;

inline bool pair_wide(bool split3, int K) { return !split3 && K >= kWideMinK; }

// The tile shape the pair kernel uses: columns per pair tile, rows of B^T
// per CTA (the B tensor map's box), k per pipeline stage.
struct PairShape {
    int bn, hn, stage_k;
};
constexpr PairShape pair_shape(bool wide)
{
    using W = Cfg<false, true, false, true>;
    using N = Cfg<true, true, false, false>;
    return wide ? PairShape{W::BN, W::HN, W::STAGE_K} : PairShape{N::BN, N::HN, N::STAGE_K};
}

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t cta_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One warp of EACH CTA of the pair takes part: both receive the same address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// The MMAs (issue_stage) compute D[tmem] (+)= A[tmem] * B[smem]^T over both
// CTAs: rows 0..127 of A and D in the even CTA's TMEM, 128..255 in the odd
// CTA's, at the same addresses; B's first 64 rows in the even CTA's shared
// memory, the rest in the odd CTA's, at the descriptor's offset in each.
// Issues one split stage's MMAs (four k steps of 8) into accumulator d: for
// 3xTF32 lo_a*hi_b, hi_a*lo_b, hi_a*hi_b per step, else hi_a*hi_b; the
// stage's first MMA overwrites d unless acc0.  The A planes are TMEM
// columns a_hi / a_lo (+8 per step), the B planes descriptors b_hi / b_lo
// (+2 per step: 32 bytes in 16-byte units).  In the same instruction block
// it tests, without blocking, whether the barrier at shared address nbar has
// completed the phase of parity npar (the next stage's), and returns that:
// the test's latency then overlaps the MMA issue instead of leaving the
// tensor pipe idle between stages (its queue holds little more than the MMA
// in flight).  A true result carries the test's cluster-scope acquire.
template <bool SPLIT3>
__device__ __forceinline__ uint32_t issue_stage(uint32_t d, uint32_t a_hi, uint32_t a_lo,
                                                uint64_t b_hi, uint64_t b_lo, uint32_t acc0,
                                                uint32_t nbar, uint32_t npar, uint32_t idesc)
{
    uint32_t ready;
    if (SPLIT3) {
        asm volatile(
            "{\n\t.reg .pred q, p0, p1;\n\t.reg .b64 bh, bl;\n\t.reg .b32 ah, al;\n\t"
            "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q, [%7], %8;\n\t"
            "setp.ne.b32 p0, %6, 0;\n\t"
            "setp.eq.b32 p1, %6, %6;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [%3], %4, %9, p0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [%2], %5, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [%2], %4, %9, p1;\n\t"
            "add.u32 ah, %2, 8;\n\tadd.u32 al, %3, 8;\n\tadd.s64 bh, %4, 2;\n\tadd.s64 bl, %5, 2;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [al], bh, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bl, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bh, %9, p1;\n\t"
            "add.u32 ah, %2, 16;\n\tadd.u32 al, %3, 16;\n\tadd.s64 bh, %4, 4;\n\tadd.s64 bl, %5, 4;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [al], bh, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bl, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bh, %9, p1;\n\t"
            "add.u32 ah, %2, 24;\n\tadd.u32 al, %3, 24;\n\tadd.s64 bh, %4, 6;\n\tadd.s64 bl, %5, 6;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [al], bh, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bl, %9, p1;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bh, %9, p1;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(ready)
            : "r"(d), "r"(a_hi), "r"(a_lo), "l"(b_hi), "l"(b_lo), "r"(acc0), "r"(nbar),
              "r"(npar), "r"(idesc)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred q, p0, p1;\n\t.reg .b64 bh;\n\t.reg .b32 ah;\n\t"
            "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q, [%4], %5;\n\t"
            "setp.ne.b32 p0, %3, 0;\n\t"
            "setp.eq.b32 p1, %3, %3;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [%2], %6, %7, p0;\n\t"
            "add.u32 ah, %2, 8;\n\tadd.s64 bh, %6, 2;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bh, %7, p1;\n\t"
            "add.u32 ah, %2, 16;\n\tadd.s64 bh, %6, 4;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bh, %7, p1;\n\t"
            "add.u32 ah, %2, 24;\n\tadd.s64 bh, %6, 6;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%1], [ah], bh, %7, p1;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(ready)
            : "r"(d), "r"(a_hi), "r"(acc0), "r"(nbar), "r"(npar), "l"(b_hi), "r"(idesc)
            : "memory");
        (void)a_lo;
        (void)b_lo;
    }
    return ready;
}

// Both CTAs' barriers at this offset receive one arrival once every MMA the
// thread issued before has completed.
__device__ __forceinline__ void umma_commit_both(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// Arrives on the barrier at this offset in CTA `rank` of the pair, with the
// arrive's default (CTA-scope release) semantics.  The data it announces --
// split planes in this CTA's shared memory, A planes in this CTA's TMEM --
// has been made visible to the tensor core before the arrive, by
// fence.proxy.async (shared-memory stores) or tcgen05.wait::st (TMEM
// stores); the MMA that reads it is issued only after the even CTA's
// cluster-scope acquire of the barrier.  (A cluster-scope release here
// costs each converter warp ~1200 cycles per stage on GB300, more than the
// whole stage's work.)
__device__ __forceinline__ void arrive_on(uint64_t *bar, uint32_t rank)
{
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
        "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar)),
        "r"(rank)
        : "memory");
}

__device__ __forceinline__ bool try_wait_cl(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool try_wait_cl_sleep(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitSleepNs)
        : "memory");
    return ok != 0;
}

// mbar_wait with cluster-scope acquire (the barrier is signalled from the
// other CTA or by a multicast commit).
__device__ __forceinline__ bool wait_cl(uint64_t *bar, uint32_t parity, const Abort &ab,
                                        unsigned int code, bool sleep = false)
{
    if (try_wait_cl(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (sleep ? try_wait_cl_sleep(bar, parity) : try_wait_cl(bar, parity)) return true;
        if (*ab.flag) return false;
        if (clock64() - t0 > ab.limit) {
            atomicOr(ab.status, code);
            *ab.flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void drain_cl(uint64_t *bar, uint32_t parity, long long limit)
{
    const long long t0 = clock64();
    while (!try_wait_cl(bar, parity)) {
        if (clock64() - t0 > limit) return;
    }
}

__device__ __forceinline__ bool warp_wait_cl(uint64_t *bar, uint32_t parity, const Abort &ab,
                                             unsigned int code)
{
    const bool ok = wait_cl(bar, parity, ab, code);
    return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------ the kernel

template <class C>
struct Smem {
    uint8_t *raw;
    uint8_t *split;
    float4 *epi;
    uint64_t *raw_full, *raw_empty, *split_full, *split_empty, *acc_full, *acc_empty, *mma_done;
    uint32_t *tmem_base;
    volatile int *abort_flag;
};

template <class C>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tcp_sgemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Smem<C> sm;
    sm.raw = base;
    sm.split = base + C::RAW_STAGES * C::RAW_BYTES;
    sm.epi = reinterpret_cast<float4 *>(sm.split + C::SPLIT_STAGES * C::SPLIT_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sm.epi) +
                                                  C::EPI_BYTES);
    sm.raw_full = bars;
    sm.raw_empty = sm.raw_full + C::RAW_STAGES;
    sm.split_full = sm.raw_empty + C::RAW_STAGES;
    sm.split_empty = sm.split_full + C::SPLIT_STAGES;
    sm.acc_full = sm.split_empty + C::SPLIT_STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.mma_done = sm.acc_empty + 2;
    sm.tmem_base = reinterpret_cast<uint32_t *>(sm.mma_done + 1);
    sm.abort_flag = reinterpret_cast<volatile int *>(sm.tmem_base + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cta_rank();
    const long long cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::RAW_STAGES; ++s) {
            mbar_init(&sm.raw_full[s], 1u);
            mbar_init(&sm.raw_empty[s], kConvWarps);
        }
        for (int s = 0; s < C::SPLIT_STAGES; ++s) {
            mbar_init(&sm.split_full[s], 2 * kConvWarps);  // both CTAs' converters
            mbar_init(&sm.split_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.acc_full[b], 1);
            mbar_init(&sm.acc_empty[b], 2 * 4);  // both CTAs' epilogue warps
        }
        mbar_init(sm.mma_done, 1);
        *sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(sm.tmem_base, kTmemCols);
    tc::tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated
    tc::tc_fence_after();
    const uint32_t tmem = *sm.tmem_base;
    const Abort ab{sm.abort_flag, p.status, p.wait_limit};

    if (warp == 0) {
        // ------------------------------------------------ producer (own CTA's rows)
        Ring<C::RAW_STAGES> rr;
        long long issued = 0;
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
        }
        for (long long u = cid; ok && u < p.num_units; u += ncl) {
            const WorkUnit wu = work_unit(u, p);
            const TileCoord &tc = wu.tc;
            const int m0 = tc.tm * PM + static_cast<int>(rank) * BM;
            const int n0 = tc.tn * C::BN + static_cast<int>(rank) * C::HN;
            for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                uint8_t *sa = sm.raw + rr.s * C::RAW_BYTES;
                uint8_t *sb = sa + C::A_BYTES;
                if (lane == 0) {
                    if (!mbar_wait(&sm.raw_empty[rr.s], rr.ph ^ 1u, ab, kStatusWaitEmpty)) {
                        ok = false;
                    } else {
                        const int qa = tc.q * p.a_q_step, qb = tc.q * p.b_q_step;
                        mbar_arrive_expect_tx(&sm.raw_full[rr.s], C::RAW_BYTES);
#pragma unroll
                        for (int j = 0; j < C::KSUB; ++j) {
                            const int k0 = kb * C::STAGE_K + j * BK;
                            uint8_t *ja = sa + j * C::SUB_A;
                            uint8_t *jb = sb + j * C::SUB_B;
                            if (C::A_KIN) tma_load_3d(ja, &tmA, &sm.raw_full[rr.s], k0, m0, qa);
                            else          tma_load_3d(ja, &tmA, &sm.raw_full[rr.s], m0, k0, qa);
                            if (C::B_KIN) tma_load_3d(jb, &tmB, &sm.raw_full[rr.s], k0, n0, qb);
                            else          tma_load_3d(jb, &tmB, &sm.raw_full[rr.s], n0, k0, qb);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                ++issued;
                rr.next();
            }
        }
        // when this CTA is stopping early (its own wait ran out, or another
        // role's did), the stages issued last may still be landing: wait
        // (bounded) for them before the teardown.  On the normal path every
        // stage has been consumed, and the loop is not run (running it cost
        // 2.4% at 4092^3 on GB300).
        if (lane == 0 && (!ok || *sm.abort_flag)) {
            Ring<C::RAW_STAGES> d;
            for (long long j = 0; j < issued; ++j) {
                if (j + C::RAW_STAGES >= issued) mbar_drain(&sm.raw_full[d.s], d.ph, ab.limit);
                d.next();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA only)
        if (rank == 0 && lane == 0) {
            Ring<C::SPLIT_STAGES> sr;
            Ring<C::ACC_BUFS> acc;
            bool ok = true;
            bool any = false;
            // B descriptors of split stage 0; stage s and k step kk are at
            // + s * SPLIT_BYTES + 32 * kk bytes (the start address field
            // counts 16-byte units), so the issue loop only adds constants.
            const uint64_t bdesc0 = tc::kmajor_sw128_desc(smem_u32(sm.split) + C::OFF_BHI);
            for (long long u = cid; ok && u < p.num_units; u += ncl) {
                const WorkUnit wu = work_unit(u, p);
                if (!wait_cl(&sm.acc_empty[acc.s], acc.ph ^ 1u, ab, kStatusWaitAcc)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc.s * C::BN);
                uint32_t ready = 0;  // split_full[sr] already seen complete
                for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                    if (!ready && !wait_cl(&sm.split_full[sr.s], sr.ph, ab, kStatusWaitConv)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint64_t b_st =
                        bdesc0 + static_cast<uint64_t>(sr.s * (C::SPLIT_BYTES >> 4));
                    const uint32_t a_st = tmem + C::ACC_COLS + sr.s * C::A_COLS;
                    Ring<C::SPLIT_STAGES> nx = sr;
                    nx.next();
#pragma unroll
                    for (int j = 0; j < C::KSUB; ++j) {
                        const uint64_t b_hi = b_st + static_cast<uint64_t>(j * (C::SUB_SPLIT >> 4));
                        const uint32_t a_hi = a_st + j * C::SUB_COLS;
                        ready = issue_stage<C::SPLIT3>(
                            d_tmem, a_hi, a_hi + BK, b_hi, b_hi + (C::OFF_BLO >> 4),
                            (kb > wu.kb_lo || j > 0) ? 1u : 0u, smem_u32(&sm.split_full[nx.s]),
                            nx.ph, C::IDESC);
                    }
                    if (kb + 1 == wu.kb_hi) ready = 0;  // the next unit waits afresh
                    any = true;
                    umma_commit_both(&sm.split_empty[sr.s]);
                    sr.next();
                }
                if (!ok) break;
                umma_commit_both(&sm.acc_full[acc.s]);
                acc.next();
            }
            if (any) {
                umma_commit_both(sm.mma_done);
                drain_cl(sm.mma_done, 0, ab.limit);
            }
        }
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ converters (own CTA's halves)
        const bool is_a = warp < kBConvWarp0;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int ct = threadIdx.x - kBConvWarp0 * 32;
        Ring<C::RAW_STAGES> rr;
        Ring<C::SPLIT_STAGES> sr;
        bool ok = true;
        for (long long u = cid; ok && u < p.num_units; u += ncl) {
            const WorkUnit wu = work_unit(u, p);
            for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                if (!warp_wait(&sm.raw_full[rr.s], rr.ph, ab, kStatusWaitFull, lane) ||
                    !warp_wait_cl(&sm.split_empty[sr.s], sr.ph ^ 1u, ab, kStatusWaitMma)) {
                    ok = false;
                    break;
                }
                const uint8_t *sa = sm.raw + rr.s * C::RAW_BYTES;
                const uint8_t *sb = sa + C::A_BYTES;
                if (is_a) {
                    tc::tc_fence_after();
                    const uint32_t t_st = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                          C::ACC_COLS + sr.s * C::A_COLS;
#pragma unroll 1
                    for (int j = 0; j < C::KSUB; ++j) {
                        const uint32_t t_hi = t_st + j * C::SUB_COLS;
                        tc::convert_a_row<C::A_KIN, C::SPLIT3>(sa + j * C::SUB_A, row, t_hi,
                                                               t_hi + BK);
                    }
                    tc::tmem_wait_st();
                    tc::tc_fence_before();
                } else {
                    uint8_t *st = sm.split + sr.s * C::SPLIT_BYTES;
#pragma unroll 1
                    for (int j = 0; j < C::KSUB; ++j) {
                        uint8_t *jt = st + j * C::SUB_SPLIT;
                        tc::convert_b_tile<C::HN, C::B_KIN, C::SPLIT3>(sb + j * C::SUB_B,
                                                                    jt + C::OFF_BHI,
                                                                    jt + C::OFF_BLO, ct);
                    }
                    tc::fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sm.raw_empty[rr.s]);
                    arrive_on(&sm.split_full[sr.s], 0);
                }
                rr.next();
                sr.next();
            }
        }
    } else {
        // ------------------------------------------------ epilogue (own CTA's rows)
        const int q = warp & 3;
        const int r0 = static_cast<int>(rank) * BM + q * 32;  // this warp's first row
        float4 *stage = sm.epi + q * (tc::kStageFloats / 4);
        Ring<C::ACC_BUFS> acc;
        for (long long u = cid; u < p.num_units; u += ncl) {
            const WorkUnit wu = work_unit(u, p);
            const OutTile o = out_tile<PM, C::BN>(p, wu);
            tc::prefetch_c_rows(o, r0, lane);
            int w = 1;
            if (lane == 0) w = wait_cl(&sm.acc_full[acc.s], acc.ph, ab, kStatusWaitAcc, true);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            drain_cl(&sm.acc_full[acc.s], acc.ph, ab.limit);
            tc::tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc.s * C::BN);
#pragma unroll 1
            for (int c0 = 0; c0 < C::BN; c0 += 32) {
                float v[32];
                tc::tmem_ld32(tbase + c0, v);
                tc::store_chunk_staged(o, r0, c0, v, stage, lane);
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_on(&sm.acc_empty[acc.s], 0);
            acc.next();
        }
    }

    // ---- teardown: both CTAs done with each other's memory; free TMEM jointly
    tc::tc_fence_before();
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace tcp
}  // namespace sg
