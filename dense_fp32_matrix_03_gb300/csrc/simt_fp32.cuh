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
//  * lane 0 of warp 0 fills a STAGES-deep ring of shared-memory stages,
//    each SUBS x 32 deep in K.  With TMA it issues two tiled tensor loads per
//    sub-block (out-of-bounds rows,
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
//    The FMAs are issued two per instruction (fma.rn.f32x2) where one operand
//    arrives in adjacent registers (see Acc below).
//  * tiles are visited in a persistent, grouped order (one CTA per SM).
//  * the epilogue fuses alpha and beta: C is read only when beta != 0.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace sg {

// K per sub-block: one 128-byte swizzle row of fp32, the widest box a
// 128-byte-swizzled TMA copy takes along its contiguous dimension.
constexpr int kSubK = 32;


// A stage holds SUBS sub-blocks of K (BK = 32 * SUBS): all of A's
// sub-blocks (each BM x 32), then all of B's.  More sub-blocks per stage
// means fewer barrier round trips per FFMA.
template <int BM_, int BN_, int WM_, int WN_, int STAGES_, int SUBS_ = 1, int LAG_ = 1,
          int KSTEP_ = 4>
struct SimtCfg {
    static constexpr int BM = BM_, BN = BN_, WM = WM_, WN = WN_, STAGES = STAGES_;
    static constexpr int SUBS = SUBS_, BK = kSubK * SUBS_;
    static constexpr int LAG = LAG_;      // see "Who fills the stages" below
    static constexpr int KSTEP = KSTEP_;  // k per fragment load (see Frag)
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    // The consumer warps issue the copies themselves (no producer warp), so
    // that each warp may use up to 255 registers.
    static constexpr int THREADS = CONSUMER_WARPS * 32;
    static constexpr int WMITER = WM / 32, WNITER = WN / 16;
    static constexpr int TM = 4 * WMITER, TN = 4 * WNITER;
    static constexpr int A_SUB = BM * kSubK * 4, B_SUB = BN * kSubK * 4;
    static constexpr int A_BYTES = SUBS * A_SUB, B_BYTES = SUBS * B_SUB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // full/empty barriers, abort flag, release counters, the issue cursor
    static constexpr int BAR_BYTES = 2 * STAGES * 8 + 16 + 4 * STAGES + 4 + 64;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + BAR_BYTES;
    static_assert(BM % WM == 0 && BN % WN == 0 && WM % 32 == 0 && WN % 16 == 0, "tile shape");
    static_assert(BM <= 256 && BN <= 256, "a TMA box spans at most 256 rows");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(LAG >= 0 && LAG < STAGES, "copies must run ahead of the consumers");
    static_assert(KSTEP == 2 || KSTEP == 4, "fragment step");
};

// Who fills the stages.  The CTA's k-blocks are numbered j = 0, 1, ... over
// all of its tiles in order; k-block j lives in stage j % STAGES.  All stages
// are filled up front; after the warps have consumed k-block `it`, the stage
// of k-block it-LAG (which every warp has normally released by then) is
// refilled, so the copies run STAGES-1-LAG k-blocks ahead of the consumers.
// The wait for that release is bounded like every other wait.  Positions are
// advanced incrementally: no division on the per-k-block path.
// Unroll of the consumer's k-step loop; CTAs per SM the kernel is compiled for.
#ifndef SG_SIMT_UNROLL
#define SG_SIMT_UNROLL 4
#endif
#ifndef SG_SIMT_MINB
#define SG_SIMT_MINB 1
#endif
constexpr int kGroupUnroll = SG_SIMT_UNROLL;
constexpr int kMinBlocks = SG_SIMT_MINB;

// Walks the (work unit, k-block) sequence of one CTA.
struct KPos {
    long long unit;   // global work-unit index
    int kb, kb_end;   // current k-block and end of the unit's slice
    int stage;        // stage of this k-block
    uint32_t phase;   // round parity of this k-block's stage
    TileCoord tc;

    __device__ __forceinline__ void load_unit(const GemmParams &p)
    {
        if (unit < p.num_units) {
            const WorkUnit w = work_unit(unit, p);
            tc = w.tc;
            kb = w.kb_lo;
            kb_end = w.kb_hi;
        }
    }
    __device__ __forceinline__ void start(const GemmParams &p)
    {
        unit = blockIdx.x;
        stage = 0;
        phase = 0;
        load_unit(p);
    }
    template <int STAGES>
    __device__ __forceinline__ void next(const GemmParams &p)
    {
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
        if (++kb == kb_end) {
            unit += gridDim.x;
            load_unit(p);
        }
    }
};

// Where the next k-block to load comes from: the cursor lives in shared
// memory and is advanced by whichever warp issues the next copy.
struct IssueCursor {
    KPos pos;
    long long issued;  // k-blocks issued so far
};

// TMA: the stages are refilled by the last warp to release them.  Every warp
// counts its release of a stage on that stage's counter (an acq_rel atomic);
// the warp that completes a round of the count knows that every warp is
// done reading the stage, and at once issues the copies of the k-block that
// goes there next (STAGES k-blocks later), so no warp ever waits for a
// stage to become free.  The stages are released in k-block order (a warp
// releases k-block j before j + 1), so the refills, and the cursor they
// advance, follow k-block order too; each refill reads the cursor the
// previous one wrote (ordered by the release-acquire chain of the counters).
// Lane 0 of warp 0 issues the first STAGES k-blocks.
template <class Cfg, bool A_KIN, bool B_KIN>
struct TmaIssuer {
    static constexpr unsigned kFullCount = 1;
    const CUtensorMap *tmA, *tmB;
    const GemmParams *p;
    uint8_t *smem;
    uint64_t *full, *empty;
    unsigned int *released;  // per stage: warps that released it, ever (mod 2^32)
    IssueCursor *cur;
    long long total;         // k-blocks this CTA will consume

    __device__ __forceinline__ void issue(KPos &pos)
    {
        const int s = pos.stage;
        uint8_t *sa = smem + s * Cfg::STAGE_BYTES;
        uint8_t *sb = sa + Cfg::A_BYTES;
        const int m0 = pos.tc.tm * Cfg::BM, n0 = pos.tc.tn * Cfg::BN;
        const int qa = pos.tc.q * p->a_q_step, qb = pos.tc.q * p->b_q_step;
        mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
#pragma unroll
        for (int sub = 0; sub < Cfg::SUBS; ++sub) {
            const int k0 = pos.kb * Cfg::BK + sub * kSubK;
            if (A_KIN) tma_load_3d(sa + sub * Cfg::A_SUB, tmA, &full[s], k0, m0, qa);
            else       tma_load_3d(sa + sub * Cfg::A_SUB, tmA, &full[s], m0, k0, qa);
            if (B_KIN) tma_load_3d(sb + sub * Cfg::B_SUB, tmB, &full[s], k0, n0, qb);
            else       tma_load_3d(sb + sub * Cfg::B_SUB, tmB, &full[s], n0, k0, qb);
        }
        pos.template next<Cfg::STAGES>(*p);
    }

    // Fills every stage once; the CTA synchronises before the first refill.
    __device__ __forceinline__ void prologue(int warp, int lane, const Abort &)
    {
        if (warp != 0 || lane != 0) return;
        tma_prefetch_desc(tmA);
        tma_prefetch_desc(tmB);
        KPos pos;
        pos.start(*p);
        long long n = 0;
        for (; n < Cfg::STAGES && n < total; ++n) issue(pos);
        cur->pos = pos;
        cur->issued = n;
        for (int s = 0; s < Cfg::STAGES; ++s) released[s] = 0u;
    }

    // Called by every lane of every consumer warp after it consumed the
    // k-block in stage `s`.  Never waits.
    __device__ __forceinline__ bool refill(long long, const Abort &, int, int lane, int s)
    {
        __syncwarp();
        if (lane == 0) {
            unsigned int before;
            asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                         : "=r"(before)
                         : "r"(smem_u32(&released[s]))
                         : "memory");
            if (before % Cfg::CONSUMER_WARPS == Cfg::CONSUMER_WARPS - 1) {
                const long long n = cur->issued;
                if (n < total) {
                    KPos pos = cur->pos;
                    issue(pos);
                    cur->pos = pos;
                    cur->issued = n + 1;
                }
            }
        }
        return true;
    }

    // After an abort (every warp has left its loop): let every issued copy
    // land before the CTA exits.
    __device__ __forceinline__ void drain(long long limit, int warp, int lane)
    {
        if (warp != 0 || lane != 0) return;
        const long long issued = cur->issued;
        for (long long j = issued - 1; j >= 0 && j >= issued - Cfg::STAGES; --j)
            mbar_drain(&full[j % Cfg::STAGES], static_cast<uint32_t>((j / Cfg::STAGES) & 1),
                       limit);
    }
};

// cp.async: every thread copies its share of the stage (operands TMA cannot
// describe: unaligned bases, row pitches or batch strides that are not
// multiples of 16 bytes) and the stage's full barrier counts one arrival per
// thread when that thread's copies have landed.
template <class Cfg, bool A_KIN, bool B_KIN, bool EVEN_K>
struct CpAsyncIssuer {
    static constexpr unsigned kFullCount = Cfg::THREADS;
    const GemmParams *p;
    uint8_t *smem;
    uint64_t *full, *empty;
    long long total;
    long long issued;
    KPos pos;

    __device__ __forceinline__ bool issue_to(long long target, const Abort &ab, int warp,
                                             int lane)
    {
        if (target > total) target = total;
        const int tid = warp * 32 + lane;
        while (issued < target) {
            const int s = pos.stage;
            if (!warp_wait(&empty[s], pos.phase ^ 1u, ab, kStatusWaitEmpty, lane)) return false;
            uint8_t *sa = smem + s * Cfg::STAGE_BYTES;
            uint8_t *sb = sa + Cfg::A_BYTES;
            const TileCoord &tc = pos.tc;
#pragma unroll
            for (int sub = 0; sub < Cfg::SUBS; ++sub) {
                const int k0 = pos.kb * Cfg::BK + sub * kSubK;
                cp_async_tile<Cfg::BM, A_KIN, EVEN_K>(sa + sub * Cfg::A_SUB, p->A + tc.q * p->sA,
                                                      p->lda, tc.tm * Cfg::BM, p->M, k0, p->K,
                                                      p->a_vec4 != 0, tid, Cfg::THREADS);
                cp_async_tile<Cfg::BN, B_KIN, EVEN_K>(sb + sub * Cfg::B_SUB, p->B + tc.q * p->sB,
                                                      p->ldb, tc.tn * Cfg::BN, p->N, k0, p->K,
                                                      p->b_vec4 != 0, tid, Cfg::THREADS);
            }
            cp_async_arrive_noinc(&full[s]);
            ++issued;
            pos.template next<Cfg::STAGES>(*p);
        }
        return true;
    }

    __device__ __forceinline__ void prologue(int warp, int lane, const Abort &ab)
    {
        issued = 0;
        pos.start(*p);
        issue_to(Cfg::STAGES, ab, warp, lane);
    }

    // Called by every lane of every consumer warp after it consumed the
    // k-block `it` in stage `s`: releases the stage, then copies what this
    // thread owes of the k-blocks up to it + 1 - LAG + STAGES (waiting, with
    // a bound, until every warp has released the stages they go to).
    __device__ __forceinline__ bool refill(long long it, const Abort &ab, int warp, int lane,
                                           int s)
    {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        return issue_to(it + 1 - Cfg::LAG + Cfg::STAGES, ab, warp, lane);
    }

    __device__ __forceinline__ void drain(long long, int, int)
    {
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
};

// ------------------------------------------------------------- consumer

__device__ __forceinline__ float4 lds128(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

// Operand fragments of one k-step (Cfg::KSTEP k values: 4 with 128-bit
// loads of K-inner rows, 2 with 64-bit loads) for one lane:
// a[kk][i] = op(A)[row i of the lane, k = KSTEP*g + kk], b[kk][j] likewise.
template <class Cfg>
struct Frag {
    float a[Cfg::KSTEP][Cfg::TM];
    float b[Cfg::KSTEP][Cfg::TN];
};

__device__ __forceinline__ float2 lds64(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// Byte offset, inside a lane's swizzled 128-byte row, of k-step g: the
// 16-byte chunk (k / 4) moves by the XOR key, the 8-byte half (2-k steps)
// stays in place.
template <int KSTEP>
__device__ __forceinline__ uint32_t kstep_offset(int g, uint32_t key)
{
    if (KSTEP == 4) return (static_cast<uint32_t>(g) << 4) ^ key;
    return ((static_cast<uint32_t>(g >> 1) << 4) ^ key) + (static_cast<uint32_t>(g & 1) << 3);
}

// Loads the fragments of k-step g from a stage.  a_base / b_base are this
// lane's base addresses inside the stage (see simt_consumer).
template <class Cfg, bool A_KIN, bool B_KIN>
__device__ __forceinline__ void load_frag(Frag<Cfg> &f, uint32_t a_base, uint32_t b_base,
                                          uint32_t a_key, uint32_t b_key, int g)
{
    constexpr int kKStep = Cfg::KSTEP;
    constexpr int WMITER = Cfg::WMITER, WNITER = Cfg::WNITER;
    if (A_KIN) {
        const uint32_t ag = a_base + kstep_offset<kKStep>(g, a_key);
#pragma unroll
        for (int wm = 0; wm < WMITER; ++wm)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t addr = ag + (wm * 32 + i * 8) * 128;
                if (kKStep == 4) {
                    const float4 v = lds128(addr);
                    f.a[0][wm * 4 + i] = v.x;
                    f.a[1 % kKStep][wm * 4 + i] = v.y;
                    f.a[2 % kKStep][wm * 4 + i] = v.z;
                    f.a[3 % kKStep][wm * 4 + i] = v.w;
                } else {
                    const float2 v = lds64(addr);
                    f.a[0][wm * 4 + i] = v.x;
                    f.a[1][wm * 4 + i] = v.y;
                }
            }
    } else {
#pragma unroll
        for (int kk = 0; kk < kKStep; ++kk)
#pragma unroll
            for (int wm = 0; wm < WMITER; ++wm) {
                const float4 v = lds128(a_base + ((kKStep * g + kk) * Cfg::BM + wm * 32) * 4);
                f.a[kk][wm * 4 + 0] = v.x;
                f.a[kk][wm * 4 + 1] = v.y;
                f.a[kk][wm * 4 + 2] = v.z;
                f.a[kk][wm * 4 + 3] = v.w;
            }
    }
    if (B_KIN) {
        // rows j = 1, 3 of a 4-row group have the swizzle key lc + 4
        const uint32_t bg0 = b_base + kstep_offset<kKStep>(g, b_key);
        const uint32_t bg1 = b_base + kstep_offset<kKStep>(g, b_key ^ (4u << 4));
#pragma unroll
        for (int wn = 0; wn < WNITER; ++wn)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t addr = ((j & 1) ? bg1 : bg0) + (wn * 16 + j * 4) * 128;
                if (kKStep == 4) {
                    const float4 v = lds128(addr);
                    f.b[0][wn * 4 + j] = v.x;
                    f.b[1 % kKStep][wn * 4 + j] = v.y;
                    f.b[2 % kKStep][wn * 4 + j] = v.z;
                    f.b[3 % kKStep][wn * 4 + j] = v.w;
                } else {
                    const float2 v = lds64(addr);
                    f.b[0][wn * 4 + j] = v.x;
                    f.b[1][wn * 4 + j] = v.y;
                }
            }
    } else {
#pragma unroll
        for (int kk = 0; kk < kKStep; ++kk)
#pragma unroll
            for (int wn = 0; wn < WNITER; ++wn) {
                const float4 v = lds128(b_base + ((kKStep * g + kk) * Cfg::BN + wn * 16) * 4);
                f.b[kk][wn * 4 + 0] = v.x;
                f.b[kk][wn * 4 + 1] = v.y;
                f.b[kk][wn * 4 + 2] = v.z;
                f.b[kk][wn * 4 + 3] = v.w;
            }
    }
}

// ------------------------------------------------------- accumulators
//
// sm_100-class SMs execute two fp32 FMAs per lane in one instruction
// (fma.rn.f32x2 on 64-bit register pairs).  Each of the two products is
// rounded exactly as a scalar fmaf would round it, so results are the same
// as with scalar FFMA; what changes is that one issue slot now carries two
// FMAs, leaving room for the shared loads.  Pairs are taken along the
// dimension whose fragment values arrive adjacent in registers (one 128-bit
// shared load gives four consecutive columns of an N-inner B, or four
// consecutive rows of an M-inner A); the other operand is broadcast into
// both halves.  When both operands are K-inner, no dimension pairs for free.
enum PairDim { kPairNone = 0, kPairJ = 1, kPairI = 2 };
#ifndef SG_SIMT_FFMA2
#define SG_SIMT_FFMA2 1
#endif
#ifndef SG_SIMT_NT_PAIR
#define SG_SIMT_NT_PAIR 0
#endif
template <bool A_KIN, bool B_KIN>
constexpr int pair_dim()
{
    return !SG_SIMT_FFMA2 ? kPairNone : !B_KIN ? kPairJ : !A_KIN ? kPairI : SG_SIMT_NT_PAIR;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d.lo = fma(a.lo, b.lo, d.lo), d.hi = fma(a.hi, b.hi, d.hi), each rounded once.
__device__ __forceinline__ void ffma2(uint64_t &d, uint64_t a, uint64_t b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// TM x TN fp32 accumulators of one lane, stored as PD says.
template <class Cfg, int PD>
struct Acc {
    static constexpr int TM = Cfg::TM, TN = Cfg::TN, kKStep = Cfg::KSTEP;
    static constexpr int R = PD == kPairI ? TM / 2 : TM;
    static constexpr int C = PD == kPairJ ? TN / 2 : TN;
    using T = typename std::conditional<PD == kPairNone, float, uint64_t>::type;
    T v[R][C];

    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) v[r][c] = T(0);
    }

    __device__ __forceinline__ void fma(const Frag<Cfg> &f)
    {
#pragma unroll
        for (int kk = 0; kk < kKStep; ++kk) {
            if constexpr (PD == kPairNone) {
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) v[i][j] = fmaf(f.a[kk][i], f.b[kk][j], v[i][j]);
            } else if constexpr (PD == kPairJ) {
                uint64_t bp[C];
#pragma unroll
                for (int c = 0; c < C; ++c) bp[c] = pack2(f.b[kk][2 * c], f.b[kk][2 * c + 1]);
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const uint64_t ab = pack2(f.a[kk][i], f.a[kk][i]);
#pragma unroll
                    for (int c = 0; c < C; ++c) ffma2(v[i][c], ab, bp[c]);
                }
            } else {
                uint64_t ap[R];
#pragma unroll
                for (int r = 0; r < R; ++r) ap[r] = pack2(f.a[kk][2 * r], f.a[kk][2 * r + 1]);
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    const uint64_t bb = pack2(f.b[kk][j], f.b[kk][j]);
#pragma unroll
                    for (int r = 0; r < R; ++r) ffma2(v[r][j], ap[r], bb);
                }
            }
        }
    }

    __device__ __forceinline__ void to_float(float (&out)[TM][TN]) const
    {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) {
                if constexpr (PD == kPairNone) {
                    out[r][c] = v[r][c];
                } else if constexpr (PD == kPairJ) {
                    unpack2(v[r][c], out[r][2 * c], out[r][2 * c + 1]);
                } else {
                    unpack2(v[r][c], out[2 * r][c], out[2 * r + 1][c]);
                }
            }
    }
};

// One consumer warp: WM x WN outputs of the CTA tile; each lane holds
// TM x TN accumulators as (WM/32) x (WN/16) sub-blocks of 4 x 4.
//
// Addressing is resolved once into per-lane base addresses so that every
// shared load is "base + immediate".  For a K-inner (swizzled) operand the
// lane's rows are `base + 8*i` (A) or `base + 4*j` (B) with base = lane row
// (A) or lane column (B), so the row modulo 8 -- the swizzle key -- is lr for
// A and lc + 4*(j odd) for B, and the 16-byte chunk of k-group g sits at
// (g ^ key) * 16: one XOR per k-group.
//
// The k loop is software-pipelined over k-groups: the fragments of the next
// k-group (or of the next stage's first k-group) are loaded into the second
// register set while the current one feeds the FFMAs.  A stage is released
// after the FFMAs of its last k-group, i.e. once every value read from it has
// been consumed.
template <class Cfg, bool A_KIN, bool B_KIN, class Issuer>
__device__ __forceinline__ void simt_consumer(const GemmParams &p, uint8_t *smem, uint64_t *full,
                                              uint64_t *empty, const Abort &ab, int cw, int lane,
                                              Issuer &iss)
{
    constexpr int WMITER = Cfg::WMITER, WNITER = Cfg::WNITER, TM = Cfg::TM, TN = Cfg::TN;
    constexpr int BM = Cfg::BM, BN = Cfg::BN;
    constexpr int GROUPS = kSubK / Cfg::KSTEP;  // k-steps per sub-block
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

    const uint32_t smem0 = smem_u32(smem);
    // Lane-relative byte offsets inside a stage (runtime part only).
    const uint32_t a_lane = A_KIN ? (wm0 + lr) * 128 : (wm0 + lr * 4) * 4;
    const uint32_t b_lane = Cfg::A_BYTES + (B_KIN ? (wn0 + lc) * 128 : (wn0 + lc * 4) * 4);
    const uint32_t a_key = static_cast<uint32_t>(lr) << 4;
    const uint32_t b_key = static_cast<uint32_t>(lc) << 4;
    auto stage_addr = [&](int s) { return smem0 + static_cast<uint32_t>(s) * Cfg::STAGE_BYTES; };
    auto wait_full = [&](int s, uint32_t ph) {
        return warp_wait(&full[s], ph, ab, kStatusWaitFull, lane);
    };
    int cs = 0;         // stage of the current k-block
    uint32_t cph = 0;   // its round parity

    long long it = 0;  // k-blocks consumed so far by this CTA
    for (long long u = blockIdx.x; u < p.num_units; u += gridDim.x) {
        const WorkUnit wu = work_unit(u, p);
        // out = C, or this slice's workspace slot with alpha 1, beta 0
        const OutTile o = out_tile<BM, BN>(p, wu);
        if (o.beta != 0.f) {
            // ask L2 for this lane's lines of C now, so that the epilogue's
            // loads do not wait on DRAM (valid addresses only)
#pragma unroll
            for (int wm = 0; wm < WMITER; ++wm)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = row_of(wm, i);
                    if (r >= o.rows) continue;
#pragma unroll
                    for (int wn = 0; wn < WNITER; ++wn) {
                        const int c = col_of(wn, 0);
                        if (c < o.cols)
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(o.base + r * o.ld + c));
                    }
                }
        }
        Acc<Cfg, pair_dim<A_KIN, B_KIN>()> accp;
        accp.zero();

        for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb, ++it) {
            if (!wait_full(cs, cph)) return;
            const uint32_t stage = stage_addr(cs);
#pragma unroll kGroupUnroll
            for (int g = 0; g < Cfg::SUBS * GROUPS; ++g) {
                const int sub = g / GROUPS;
                Frag<Cfg> f;
                load_frag<Cfg, A_KIN, B_KIN>(f, stage + sub * Cfg::A_SUB + a_lane,
                                             stage + sub * Cfg::B_SUB + b_lane, a_key, b_key,
                                             g % GROUPS);
                accp.fma(f);
            }
            if (!iss.refill(it, ab, cw, lane, cs)) return;
            if (++cs == Cfg::STAGES) {
                cs = 0;
                cph ^= 1u;
            }
        }

        float acc[TM][TN];
        accp.to_float(acc);

        // ---- epilogue: out = alpha * acc + beta * out, masked at the M/N
        // edges.  A row's loads of C are all issued before its stores (the
        // compiler may not move a load of C past a store to C itself).
        const bool use_beta = o.beta != 0.f;
#pragma unroll
        for (int wm = 0; wm < WMITER; ++wm)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = row_of(wm, i);
                if (r >= o.rows) continue;
                float *orow = o.base + r * o.ld;
                if (!B_KIN && o.vec4 && use_beta) {
                    float4 old[WNITER];
#pragma unroll
                    for (int wn = 0; wn < WNITER; ++wn) {
                        const int c0 = col_of(wn, 0);
                        old[wn] = c0 + 3 < o.cols ? *reinterpret_cast<const float4 *>(orow + c0)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int wn = 0; wn < WNITER; ++wn) {
                        const float *av = &acc[wm * 4 + i][wn * 4];
                        const int c0 = col_of(wn, 0);
                        if (c0 + 3 < o.cols) {
                            float4 v;
                            v.x = fmaf(o.beta, old[wn].x, o.alpha * av[0]);
                            v.y = fmaf(o.beta, old[wn].y, o.alpha * av[1]);
                            v.z = fmaf(o.beta, old[wn].z, o.alpha * av[2]);
                            v.w = fmaf(o.beta, old[wn].w, o.alpha * av[3]);
                            *reinterpret_cast<float4 *>(orow + c0) = v;
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int c = c0 + j;
                                if (c < o.cols) orow[c] = fmaf(o.beta, orow[c], o.alpha * av[j]);
                            }
                        }
                    }
                    continue;
                }
#pragma unroll
                for (int wn = 0; wn < WNITER; ++wn) {
                    const float *av = &acc[wm * 4 + i][wn * 4];
                    if (!B_KIN) {
                        const int c0 = col_of(wn, 0);
                        if (o.vec4 && c0 + 3 < o.cols) {
                            float4 v;
                            v.x = o.alpha * av[0];
                            v.y = o.alpha * av[1];
                            v.z = o.alpha * av[2];
                            v.w = o.alpha * av[3];
                            float4 *dst = reinterpret_cast<float4 *>(orow + c0);
                            if (use_beta) {
                                const float4 old = *dst;
                                v.x = fmaf(o.beta, old.x, v.x);
                                v.y = fmaf(o.beta, old.y, v.y);
                                v.z = fmaf(o.beta, old.z, v.z);
                                v.w = fmaf(o.beta, old.w, v.w);
                            }
                            *dst = v;
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int c = c0 + j;
                                if (c < o.cols) {
                                    float v = o.alpha * av[j];
                                    if (use_beta) v = fmaf(o.beta, orow[c], v);
                                    orow[c] = v;
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int c = col_of(wn, j);
                            if (c < o.cols) {
                                float v = o.alpha * av[j];
                                if (use_beta) v = fmaf(o.beta, orow[c], v);
                                orow[c] = v;
                            }
                        }
                    }
                }
            }
    }
}

// ---------------------------------------------------------------- kernel

template <class Cfg, bool A_KIN, bool B_KIN, bool USE_TMA, bool EVEN_K>
__global__ void __launch_bounds__(Cfg::THREADS, kMinBlocks)
    simt_sgemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + Cfg::STAGES);
    unsigned int *released = reinterpret_cast<unsigned int *>(empty + Cfg::STAGES) + 1;
    IssueCursor *cursor = reinterpret_cast<IssueCursor *>(
        (reinterpret_cast<uintptr_t>(released + Cfg::STAGES) + 7) & ~static_cast<uintptr_t>(7));
    static_assert(sizeof(IssueCursor) <= 48, "issue cursor fits the bookkeeping bytes");
    using Issuer = typename std::conditional<USE_TMA, TmaIssuer<Cfg, A_KIN, B_KIN>,
                                             CpAsyncIssuer<Cfg, A_KIN, B_KIN, EVEN_K>>::type;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], Issuer::kFullCount);
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Abort ab{abort_flag, p.status, p.wait_limit};

    // k-blocks this CTA consumes: its units are blockIdx.x + i*gridDim.x
    long long my_kblocks;
    if (p.splits <= 1) {
        my_kblocks = (p.num_units - blockIdx.x + gridDim.x - 1) / static_cast<long long>(gridDim.x) *
                     p.k_blocks;
    } else {
        my_kblocks = 0;
        for (long long u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            const WorkUnit w = work_unit(u, p);
            my_kblocks += w.kb_hi - w.kb_lo;
        }
    }
    Issuer iss;
    if constexpr (USE_TMA) {
        iss.tmA = &tmA;
        iss.tmB = &tmB;
        iss.released = released;
        iss.cur = cursor;
    }
    iss.p = &p;
    iss.smem = smem;
    iss.full = full;
    iss.empty = empty;
    iss.total = my_kblocks;
    iss.prologue(warp, lane, ab);
    __syncthreads();  // the cursor and release counters are set up
    simt_consumer<Cfg, A_KIN, B_KIN>(p, smem, full, empty, ab, warp, lane, iss);
    __syncthreads();  // no copy is issued after this point
    if (*abort_flag) iss.drain(ab.limit, warp, lane);
    __syncthreads();
}

}  // namespace sg
