// tc_ss.cuh -- tensor-core GEMM on CTA pairs with both operands read by the
// MMA from shared memory, fp32 accumulation and output:
// C = alpha * op(A) @ op(B) + beta * C.
//
// TMA stages the operands straight into the layout tcgen05.mma reads:
//   - 16-bit inputs (bf16 or fp16, kind::f16): the contraction the pages
//     point to for tensor cores with narrower inputs ("From 1% to 94% of
//     cuBLAS, one kernel at a time", future work); products of 16-bit values
//     are exact in fp32;
//   - fp32 operands already in TF32 form (kind::tf32), made by a pass over
//     the operands into the caller's workspace: one plane rounded to the
//     nearest TF32 value (TF32), or the hi and lo planes of the 3xTF32 split,
//     multiplied as hi*hi + hi*lo + lo*hi per k step (3xTF32; the first
//     two read A's hi box once, through the collector buffer);
//   - the caller's fp32 matrices themselves (kind::tf32 reads the 19 high
//     bits of each 32-bit value and ignores the 13 low mantissa bits): the
//     single pass of TF32, or the hi planes of 3xTF32 beside lo planes that
//     a pass wrote in the operands' own layout or that the kernel makes
//     itself (below).  An operand whose rows run along M or N (A stored
//     K x M, B stored K x N) is staged M/N-major: TMA boxes of 32 rows-inner
//     values by 32 k in the 128-byte swizzle with 32-byte atoms, read by the
//     MMA through an M/N-major descriptor; the others K-major, boxes of 32 k
//     (128 bytes of fp32, 64 k of 16-bit) by 128 rows, 128-byte swizzle.
//
// Tile 256 x 256 per CTA pair (cta_group::2, M = 256, N = 256): each CTA
// stages its 128 rows of A and its 128 of the tile's 256 rows of B^T.  A
// stage holds, per CTA, two boxes of each operand (128 k of 16-bit values;
// 64 KB, three stages), one box of each plane of 3xTF32 (32 k; 64 KB, three
// stages; with the lo planes made in the kernel, four raw stages of 32 KB
// and two lo stages), or one box of TF32 (32 k; 32 KB, five stages).  Both CTAs' TMA
// loads complete on the even CTA's barrier (cta_group::2 form, which may
// name the peer's barrier); one thread of the even CTA issues every MMA and
// multicasts its commits (stage free, accumulator full) to both CTAs.  TMEM:
// two 256-column fp32 accumulators per CTA (double buffered, so the epilogue
// overlaps the next tile).
//
// Warps: 0 TMA producer, 1 TMEM allocator + MMA issuer (even CTA), 2-5
// epilogue (warp w reads TMEM lanes 32 * (w % 4) .. +31; C by TMA in chunks
// of 32 rows x 16 columns, 32 x 32 for single-plane TF32, when C's rows suit
// TMA), 6-7 converters (in-kernel lo planes only).  Every wait is bounded; the CTAs meet at a cluster barrier
// before freeing TMEM.
//
// In-kernel lo planes (3xTF32 on the caller's matrices, KindTF32 with CONV):
// TMA stages only the raw boxes (the hi planes), in a ring of its own, each
// CTA's loads completing on its own barrier; SG_TCS_CONV_WARPS converter
// warps per CTA then write each stage's lo boxes into a second, shorter ring
// from the raw boxes, value by value at the same offsets (the swizzle is a
// function of the offset, so a lo box has its raw box's layout), make them
// visible to the tensor core (fence.proxy.async) and arrive on the even
// CTA's conv barrier, which the MMA issuer waits on in place of the load
// barrier.  No pass over the operands and no workspace for planes.
#pragma once

#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_pair.cuh"

namespace sg {
namespace tcs {

using tcp::arrive_on;
using tcp::cluster_sync;
using tcp::cta_rank;
using tcp::drain_cl;
using tcp::tmem_alloc_pair;
using tcp::tmem_dealloc_pair;
using tcp::umma_commit_both;
using tcp::wait_cl;
using tcp::warp_wait_cl;

constexpr int BM = 128;      // rows of C per CTA
constexpr int PM = 2 * BM;   // rows per pair tile (the MMA's M)
constexpr int BN = 256;      // columns per pair tile (the MMA's N)
constexpr int HN = BN / 2;   // rows of B^T each CTA holds
constexpr int SUB_A = BM * 128;  // one 128-byte box of A: 16 KB
constexpr int SUB_B = HN * 128;  // one box of B: 16 KB
// Single-plane TF32 stages: one 32-k box per stage (more bytes in flight
// than 64-k stages in the same room; measured on GB300, TF32 planes route,
// TFLOP/s: three 64-k stages 4092^3 nn 635, nt 648, 8192^3 873; six 32-k
// stages 654 / 667 / 898; five 635 / 654), five deep, the sixth stage's
// room given to the epilogue's C lookahead (EPI_NB, EPI_LA below).
#ifndef SG_TCS_TF32_KSUB
#define SG_TCS_TF32_KSUB 1
#endif
#ifndef SG_TCS_TF32_STAGES
#define SG_TCS_TF32_STAGES 5
#define SG_TCS_TF32_EPI_NB 4
#define SG_TCS_TF32_EPI_LA 3
#endif
// In-kernel lo planes: raw (TMA) and lo (converter) ring depths, 32 KB per
// stage each.
#ifndef SG_TCS_CONV_RAW
#define SG_TCS_CONV_RAW 4
#define SG_TCS_CONV_LO 2
#endif
// 3xTF32: the k step's two MMAs on A's hi box share one read of it through
// the collector buffer (1), or read it twice (0).
#ifndef SG_TCS_COLLECT_A
#define SG_TCS_COLLECT_A 1
#endif
constexpr int kEpiWarp0 = 2;
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kConvWarp0 = kEpiWarp0 + 4;  // in-kernel lo planes: converter warps
#ifndef SG_TCS_CONV_WARPS
#define SG_TCS_CONV_WARPS 2
#endif
constexpr int kConvWarps = SG_TCS_CONV_WARPS;
constexpr uint32_t kTmemCols = 512;
// Epilogue through TMA: per epilogue warp EPI_NB buffers (a kind's choice,
// below), each one chunk of 32 rows x EPI_CH columns of C: 16 columns (2 KB)
// in TMA's 64-byte swizzle (16-byte slot j of row r at slot j ^ ((r >> 1) &
// 3)), or 32 columns (4 KB) in its 128-byte swizzle (slot j ^ (r & 7)), so
// that lane r's reads and writes of its row are free of bank conflicts; C's
// loads run EPI_LA chunks ahead.  The other epilogue (split-K partial tiles,
// or a C TMA cannot describe) stages 32 x 32 chunks in the first 4 KB.
static_assert(2 * BN <= static_cast<int>(kTmemCols), "TMEM columns");

// Operand kinds.  ELEM: bytes per value; BOX_K: k per 128-byte box; UK: k
// per MMA (32 bytes); PLANES: 1, or 2 for the hi/lo planes of 3xTF32;
// KSUB: boxes of each plane per stage.  Instruction descriptor: fp32
// accumulate, both operands K-major, M = 256 (two CTAs), N = 256; operand
// format bf16 = 1, fp16 = 0 (kind::f16), tf32 = 2 (kind::tf32).
// A_MN / B_MN: the operand is staged M/N-major (its stored rows run along
// M or N), otherwise K-major.
template <bool BF16>
struct KindHalf {
    static constexpr bool TF32 = false;
    static constexpr int ELEM = 2, BOX_K = 64, UK = 16, PLANES = 1, KSUB = 2, STAGES = 3;
    static constexpr uint32_t FMT = BF16 ? 1u : 0u;
    static constexpr int LO_STAGES = 0;
    static constexpr int EPI_CH = 16, EPI_NB = 4, EPI_LA = 2;
    static constexpr bool A_MN = false, B_MN = false, CONV = false;
};
// CONV (3xTF32 only): the lo planes are made in the kernel from the raw
// operands (which TMA stages as the hi planes); otherwise TMA loads both.
template <int PLANES_, bool A_MN_ = false, bool B_MN_ = false, bool CONV_ = false>
struct KindTF32 {
    static constexpr bool TF32 = true;
    static constexpr int ELEM = 4, BOX_K = 32, UK = 8, PLANES = PLANES_;
    static constexpr int KSUB = PLANES_ == 1 ? SG_TCS_TF32_KSUB : 1;
    // CONV: STAGES raw stages (hi boxes, by TMA) and LO_STAGES lo stages
    // (made by the converters) in the room of three two-plane stages
    static constexpr int STAGES =
        PLANES_ == 1 ? SG_TCS_TF32_STAGES : (CONV_ ? SG_TCS_CONV_RAW : 3);
    static constexpr int LO_STAGES = CONV_ ? SG_TCS_CONV_LO : 0;
    // epilogue chunks, buffers per warp and C's lookahead: single-plane TF32
    // gives a stage's room to the epilogue (its epilogue, a third of
    // 3xTF32's MMA time per tile away, is what short tiles wait on when
    // beta != 0) in 32-column chunks, half the TMA operations of 16-column
    // ones (measured on GB300, interleaved, batched workload beta = 0.25:
    // 406 -> 426 TFLOP/s; 3xTF32 with 32-column chunks, two buffers in its
    // room: 282.7 -> 278.1, so it keeps four 16-column ones)
    static constexpr int EPI_CH = PLANES_ == 1 ? 32 : 16;
    static constexpr int EPI_NB = PLANES_ == 1 ? SG_TCS_TF32_EPI_NB : 4;
    static constexpr int EPI_LA = PLANES_ == 1 ? SG_TCS_TF32_EPI_LA : 2;
    static constexpr uint32_t FMT = 2u;
    static constexpr bool A_MN = A_MN_, B_MN = B_MN_, CONV = CONV_;
    static_assert(!CONV_ || PLANES_ == 2, "in-kernel lo planes are a 3xTF32 form");
};

template <class KD>
struct Shape {
    static constexpr int STAGES = KD::STAGES;
    static constexpr int THREADS = kThreads + (KD::CONV ? kConvWarps * 32 : 0);
    static constexpr int LO_STAGES = KD::LO_STAGES;
    static constexpr int EPI_NB = KD::EPI_NB, EPI_LA = KD::EPI_LA;
    static constexpr int EPI_CH = KD::EPI_CH;              // columns per chunk
    static constexpr int EPI_BUF = 32 * EPI_CH * 4;        // bytes per chunk
    static_assert(EPI_CH == 16 || EPI_CH == 32, "epilogue chunk width");
    static constexpr int EPI_WARP_BYTES = EPI_NB * EPI_BUF;
    static constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;  // 4 epilogue warps
    static_assert(EPI_LA >= 1 && EPI_LA < EPI_NB, "lookahead");
    static_assert(EPI_WARP_BYTES >= tc::kStageFloats * 4, "register-path staging");
    static constexpr int NBAR = 2 * STAGES + 4 + 1 + 2 * LO_STAGES + 4 * EPI_NB;
    static constexpr int STAGE_K = KD::KSUB * KD::BOX_K;
    // boxes per operand per stage TMA fills (CONV: the raw ones only)
    static constexpr int BOXES = KD::KSUB * (KD::CONV ? 1 : KD::PLANES);
    static constexpr int STAGE_BYTES = BOXES * (SUB_A + SUB_B);  // per CTA
    static constexpr int LO_BYTES = SUB_A + SUB_B;               // per CTA, CONV
    static constexpr int RINGS_BYTES = STAGES * STAGE_BYTES + LO_STAGES * LO_BYTES;
    static constexpr int SMEM_BYTES = RINGS_BYTES + EPI_BYTES + NBAR * 8 + 16 + 1024;
    // bits 15 / 16: A / B M/N-major ("transposed") instead of K-major
    static constexpr uint32_t IDESC = (1u << 4) | (KD::FMT << 7) | (KD::FMT << 10) |
                                      (KD::A_MN ? 1u << 15 : 0u) | (KD::B_MN ? 1u << 16 : 0u) |
                                      (static_cast<uint32_t>(BN >> 3) << 17) |
                                      (static_cast<uint32_t>(PM >> 4) << 24);
    // descriptor address step (16-byte units) per MMA's k: K-major rows
    // advance by the MMA's 32 bytes of k; M/N-major boxes by eight 128-byte
    // k rows (one swizzle atom)
    static constexpr uint64_t A_KSTEP = KD::A_MN ? 64 : 2, B_KSTEP = KD::B_MN ? 64 : 2;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// TMA tile load into this CTA's shared memory whose completion is counted on
// the barrier at shared::cluster address `bar` (the even CTA's).
__device__ __forceinline__ void tma_load_pair(void *smem_dst, const CUtensorMap *m, uint32_t bar,
                                              int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Shared-memory descriptor of an M/N-major TF32 operand staged as TMA boxes
// of 32 M/N values (one 128-byte row per k) by 32 k rows, in the 128-byte
// swizzle with 32-byte atoms (TMA's SWIZZLE_128B_ATOM_32B; descriptor
// swizzle mode 1), the M/N-major layout kind::tf32 reads: groups of four k
// rows (512 bytes) are the stride byte offset apart, and consecutive 32-value
// runs of M/N one 4096-byte box apart (leading byte offset).
__device__ __forceinline__ uint64_t mnmajor_sw128a32_desc(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(4096 >> 4) << 16;                // leading byte offset
    d |= static_cast<uint64_t>(512 >> 4) << 32;                 // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                        // descriptor version
    d |= static_cast<uint64_t>(1) << 61;                        // 128-byte swizzle, 32-byte atoms
    return d;
}

// One operand's box of a stage (ROWS rows of M or N by one box of k) into
// this CTA's shared memory: K-major, one TMA load (coordinates k, row,
// entry); M/N-major, ROWS / 32 loads of 32 rows-inner values by 32 k
// (coordinates row, k, entry), 4096 bytes apart.
template <bool MN, int ROWS>
__device__ __forceinline__ void load_box(uint8_t *dst, const CUtensorMap *m, uint32_t bar, int k0,
                                         int r0, int z)
{
    if constexpr (MN) {
#pragma unroll
        for (int c = 0; c < ROWS / 32; ++c) tma_load_pair(dst + c * 4096, m, bar, r0 + 32 * c, k0, z);
    } else {
        tma_load_pair(dst, m, bar, k0, r0, z);
    }
}

// TMA store of a box from this CTA's shared memory (bulk group; the caller
// commits and waits).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *m, const void *smem_src, int c0,
                                             int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(m)),
        "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's committed bulk groups still read
// shared memory (_read) or are still in progress at all.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// load_box with the completion counted on this CTA's own barrier.
template <bool MN, int ROWS>
__device__ __forceinline__ void load_box_own(uint8_t *dst, const CUtensorMap *m, uint64_t *bar,
                                             int k0, int r0, int z)
{
    if constexpr (MN) {
#pragma unroll
        for (int c = 0; c < ROWS / 32; ++c) tma_load_3d(dst + c * 4096, m, bar, r0 + 32 * c, k0, z);
    } else {
        tma_load_3d(dst, m, bar, k0, r0, z);
    }
}

// One stage's lo boxes (A's and B's, 16 KB each: 1024 16-byte groups per
// box, the B box SUB_A bytes after the A box) from the raw boxes at the same
// offsets: lo = (x - hi) with its 13 low mantissa bits cleared, hi = x with
// its 13 low mantissa bits cleared (the value the tensor core reads from
// the raw box).  Thread ct of the NT converter threads takes groups ct,
// ct + NT, ... of both boxes, all its loads in flight before its stores:
// the loads wait on shared memory the tensor core keeps busy, and one round
// of them per stage instead of four shortened a 4092^3 3xTF32 tile from
// 107.2 to 105.4 us on GB300 (the tile takes 101.8 us when the converters
// read nothing).
template <int NT>
__device__ __forceinline__ void lo_stage(uint32_t raw, uint32_t lo, int ct)
{
    static_assert(SUB_A == 16384 && SUB_B == 16384 && 1024 % NT == 0, "converter groups");
    constexpr int G = 1024 / NT;  // groups per thread and box
    float4 v[2 * G];
#pragma unroll
    for (int i = 0; i < 2 * G; ++i) {
        const uint32_t a = raw + (i < G ? 0u : static_cast<uint32_t>(SUB_A)) +
                           16u * static_cast<uint32_t>(ct + NT * (i % G));
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[i].x), "=f"(v[i].y), "=f"(v[i].z), "=f"(v[i].w)
                     : "r"(a));
    }
#pragma unroll
    for (int i = 0; i < 2 * G; ++i) {
        const uint32_t a = lo + (i < G ? 0u : static_cast<uint32_t>(SUB_A)) +
                           16u * static_cast<uint32_t>(ct + NT * (i % G));
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                     "f"(tc::trunc_tf32(v[i].x - tc::trunc_tf32(v[i].x))),
                     "f"(tc::trunc_tf32(v[i].y - tc::trunc_tf32(v[i].y))),
                     "f"(tc::trunc_tf32(v[i].z - tc::trunc_tf32(v[i].z))),
                     "f"(tc::trunc_tf32(v[i].w - tc::trunc_tf32(v[i].w)))
                     : "memory");
    }
}

__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// One pair MMA d (+)= a * b, operands by shared-memory descriptor; it
// overwrites d unless acc.
template <class KD>
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t acc)
{
    if constexpr (KD::TF32)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(Shape<KD>::IDESC), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(Shape<KD>::IDESC), "r"(acc)
            : "memory");
}

// The same MMA (kind::tf32) with A kept in the tensor core's collector
// buffer for the next MMA (fill), or taken from it and then released
// (lastuse): the two MMAs of a k step that share A's hi box read it from
// shared memory once.
__device__ __forceinline__ void mma_tf32_fill(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32.collector::a::fill [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_lastuse(uint32_t d, uint64_t a, uint64_t b,
                                                 uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32.collector::a::lastuse [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// One stage's MMAs into accumulator d: per box, four k steps of 32 bytes
// (+2 in a descriptor's 16-byte address units); with two planes, box
// (j, lo) follows box (j, hi) and each k step is hi*hi + hi*lo + lo*hi.  The
// first MMA overwrites d unless acc0.  Returns whether the next stage's
// barrier (nbar, parity npar) has already completed, tested without
// blocking (see tcp::issue_stage).
// a0 / b0: descriptors of the stage's first hi box, al0 / bl0 of its first
// lo box (3xTF32; the box after the hi one when both come by TMA, a box of
// the lo ring when the kernel makes them).
template <class KD>
__device__ __forceinline__ uint32_t issue_stage_ss(uint32_t d, uint64_t a0, uint64_t al0,
                                                   uint64_t b0, uint64_t bl0, uint32_t acc0,
                                                   uint32_t nbar, uint32_t npar)
{
    constexpr uint64_t AB = SUB_A >> 4, BB = SUB_B >> 4;
#pragma unroll
    for (int j = 0; j < KD::KSUB; ++j) {
        const uint64_t a = a0 + static_cast<uint64_t>(j * KD::PLANES) * AB;
        const uint64_t b = b0 + static_cast<uint64_t>(j * KD::PLANES) * BB;
        const uint64_t al = al0 + static_cast<uint64_t>(j * KD::PLANES) * AB;
        const uint64_t bl = bl0 + static_cast<uint64_t>(j * KD::PLANES) * BB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ah = a + Shape<KD>::A_KSTEP * kk, bh = b + Shape<KD>::B_KSTEP * kk;
            const uint32_t acc = (j == 0 && kk == 0) ? acc0 : 1u;
            if (KD::PLANES == 2) {
#if SG_TCS_COLLECT_A
                // hi * hi, hi * lo (A's hi box from the collector), lo * hi
                mma_tf32_fill(d, ah, bh, Shape<KD>::IDESC, acc);
                mma_tf32_lastuse(d, ah, bl + Shape<KD>::B_KSTEP * kk, Shape<KD>::IDESC, 1u);
                mma_ss<KD>(d, al + Shape<KD>::A_KSTEP * kk, bh, 1u);
#else
                mma_ss<KD>(d, al + Shape<KD>::A_KSTEP * kk, bh, acc);  // lo * hi
                mma_ss<KD>(d, ah, bl + Shape<KD>::B_KSTEP * kk, 1u);   // hi * lo
                mma_ss<KD>(d, ah, bh, 1u);                             // hi * hi
#endif
            } else {
                mma_ss<KD>(d, ah, bh, acc);
            }
        }
    }
    uint32_t ready;
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(ready)
        : "r"(nbar), "r"(npar)
        : "memory");
    return ready;
}

// tmA / tmB: the operands (their hi planes for 3xTF32); tmA_lo / tmB_lo:
// the lo planes, at batch coordinate entry + a_lo_z / b_lo_z (the same map
// with the plane's offset when one map holds both planes); tmC: C in boxes
// of 32 rows x 16 columns (used when p.c_tma).
template <class KD>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Shape<KD>::THREADS, 1)
    tcs_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA_lo,
                    const __grid_constant__ CUtensorMap tmB_lo,
                    const __grid_constant__ CUtensorMap tmC, const GemmParams p, int a_lo_z,
                    int b_lo_z)
{
    using S = Shape<KD>;
    constexpr int STAGE_BYTES = S::STAGE_BYTES;
    constexpr int STAGES = S::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *lo_base = base + STAGES * STAGE_BYTES;  // CONV: the lo ring
    uint8_t *epi = base + S::RINGS_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + S::RINGS_BYTES + S::EPI_BYTES);
    uint64_t *full = bars;                  // even CTA's: both CTAs' bytes
    uint64_t *empty = full + STAGES;        // per CTA: multicast commit
    uint64_t *acc_full = empty + STAGES;    // per CTA: multicast commit
    uint64_t *acc_empty = acc_full + 2;     // even CTA's: both CTAs' epilogues
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *conv_full = mma_done + 1;     // CONV, even CTA's: both CTAs' converters
    uint64_t *lo_empty = conv_full + S::LO_STAGES;  // CONV, per CTA: multicast commit
    uint64_t *cbar = lo_empty + S::LO_STAGES;       // epilogue C loads, per warp x buffer
    uint32_t *tmem_base = reinterpret_cast<uint32_t *>(cbar + 4 * S::EPI_NB);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_base + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cta_rank();
    const long long cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1u);
            mbar_init(&empty[s], 1u);
        }
        for (int s = 0; s < S::LO_STAGES; ++s) {
            mbar_init(&conv_full[s], 2 * kConvWarps);
            mbar_init(&lo_empty[s], 1u);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1u);
            mbar_init(&acc_empty[b], 2 * 4);
        }
        mbar_init(mma_done, 1u);
        for (int b = 0; b < 4 * S::EPI_NB; ++b) mbar_init(&cbar[b], 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_base, kTmemCols);
    tc::tc_fence_before();
    cluster_sync();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_base;
    const Abort ab{abort_flag, p.status, p.wait_limit};

    if (warp == 0) {
        // ------------------------------------------------ producer (own CTA's rows)
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            if (KD::PLANES == 2) {
                tma_prefetch_desc(&tmA_lo);
                tma_prefetch_desc(&tmB_lo);
            }
            // Launched as a programmatic dependent (launch_ss): the set-up
            // above overlapped the previous kernel's tail; its writes (the
            // operands' planes or copies) are visible after this wait.  Every
            // other access to memory (MMAs, epilogue loads and stores of C
            // and of split slots) follows the loads issued below.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            tc::Ring<STAGES> rr;
            long long issued = 0;
            bool ok = true;
            for (long long u = cid; ok && u < p.num_units; u += ncl) {
                const WorkUnit wu = work_unit(u, p);
                const int m0 = wu.tc.tm * PM + static_cast<int>(rank) * BM;
                const int n0 = wu.tc.tn * BN + static_cast<int>(rank) * HN;
                const int qa = wu.tc.q * p.a_q_step, qb = wu.tc.q * p.b_q_step;
                for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                    if (!wait_cl(&empty[rr.s], rr.ph ^ 1u, ab, kStatusWaitEmpty)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = base + rr.s * STAGE_BYTES;
                    uint8_t *sb = sa + S::BOXES * SUB_A;  // CONV: BOXES = 1
                    if (KD::CONV) {
                        // raw boxes only (the hi planes), on this CTA's barrier
                        const int k0 = kb * S::STAGE_K;
                        mbar_arrive_expect_tx(&full[rr.s], SUB_A + SUB_B);
                        load_box_own<KD::A_MN, BM>(sa, &tmA, &full[rr.s], k0, m0, qa);
                        load_box_own<KD::B_MN, HN>(sb, &tmB, &full[rr.s], k0, n0, qb);
                        ++issued;
                        rr.next();
                        continue;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[rr.s], 2 * STAGE_BYTES);
                    const uint32_t fb = cluster_addr(&full[rr.s], 0);
#pragma unroll
                    for (int j = 0; j < KD::KSUB; ++j) {
                        const int k0 = kb * S::STAGE_K + j * KD::BOX_K;
#pragma unroll
                        for (int pl = 0; pl < KD::PLANES; ++pl) {
                            const int x = j * KD::PLANES + pl;
                            load_box<KD::A_MN, BM>(sa + x * SUB_A, pl ? &tmA_lo : &tmA, fb, k0, m0,
                                                   qa + (pl ? a_lo_z : 0));
                            load_box<KD::B_MN, HN>(sb + x * SUB_B, pl ? &tmB_lo : &tmB, fb, k0, n0,
                                                   qb + (pl ? b_lo_z : 0));
                        }
                    }
                    ++issued;
                    rr.next();
                }
            }
            // Both CTAs' loads of a stage complete on the even CTA's barrier:
            // when stopping early, the even CTA waits (bounded) for the last
            // stages' phases, so that after the cluster barrier below no load
            // is still in flight into either CTA's shared memory.  (On the
            // normal path the MMAs consumed every stage.)  An abort in the
            // odd CTA reaches the even one through the waits that then run
            // out there.
            // (With CONV each CTA's loads complete on its own barrier.)
            if ((KD::CONV || rank == 0) && (!ok || *abort_flag)) {
                tc::Ring<STAGES> d;
                for (long long j = 0; j < issued; ++j) {
                    if (j + STAGES >= issued) drain_cl(&full[d.s], d.ph, ab.limit);
                    d.next();
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA only)
        if (rank == 0 && lane == 0) {
            tc::Ring<STAGES> sr;
            tc::Ring<2> acc;
            bool ok = true;
            bool any = false;
            const uint32_t sa0 = smem_u32(base), sb0 = smem_u32(base + S::BOXES * SUB_A);
            const uint64_t adesc0 =
                KD::A_MN ? mnmajor_sw128a32_desc(sa0) : tc::kmajor_sw128_desc(sa0);
            const uint64_t bdesc0 =
                KD::B_MN ? mnmajor_sw128a32_desc(sb0) : tc::kmajor_sw128_desc(sb0);
            // lo boxes: beside the hi ones, or (CONV) in the lo ring
            const uint32_t la0 = smem_u32(lo_base), lb0 = la0 + SUB_A;
            const uint64_t aldesc0 =
                KD::CONV ? (KD::A_MN ? mnmajor_sw128a32_desc(la0) : tc::kmajor_sw128_desc(la0))
                         : adesc0 + (SUB_A >> 4);
            const uint64_t bldesc0 =
                KD::CONV ? (KD::B_MN ? mnmajor_sw128a32_desc(lb0) : tc::kmajor_sw128_desc(lb0))
                         : bdesc0 + (SUB_B >> 4);
            tc::Ring<(S::LO_STAGES > 0 ? S::LO_STAGES : 1)> lr;  // CONV: lo ring position
            for (long long u = cid; ok && u < p.num_units; u += ncl) {
                const WorkUnit wu = work_unit(u, p);
                if (!wait_cl(&acc_empty[acc.s], acc.ph ^ 1u, ab, kStatusWaitAcc)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc.s * BN);
                uint32_t ready = 0;
                // a stage is ready when loaded (CONV: and its lo boxes made,
                // in both CTAs -- the lo ring's barrier)
                for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                    uint64_t *rb = KD::CONV ? &conv_full[lr.s] : &full[sr.s];
                    if (!ready && !wait_cl(rb, KD::CONV ? lr.ph : sr.ph, ab,
                                           KD::CONV ? kStatusWaitConv : kStatusWaitFull)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>(sr.s * (STAGE_BYTES >> 4));
                    const uint64_t loff =
                        KD::CONV ? static_cast<uint64_t>(lr.s * (S::LO_BYTES >> 4)) : soff;
                    tc::Ring<STAGES> nx = sr;
                    nx.next();
                    auto lx = lr;
                    lx.next();
                    ready = issue_stage_ss<KD>(
                        d_tmem, adesc0 + soff, aldesc0 + loff, bdesc0 + soff, bldesc0 + loff,
                        kb > wu.kb_lo ? 1u : 0u,
                        smem_u32(KD::CONV ? &conv_full[lx.s] : &full[nx.s]),
                        KD::CONV ? lx.ph : nx.ph);
                    if (kb + 1 == wu.kb_hi) ready = 0;
                    any = true;
                    umma_commit_both(&empty[sr.s]);
                    if (KD::CONV) umma_commit_both(&lo_empty[lr.s]);
                    sr.next();
                    lr.next();
                }
                if (!ok) break;
                umma_commit_both(&acc_full[acc.s]);
                acc.next();
            }
            if (any) {
                umma_commit_both(mma_done);
                drain_cl(mma_done, 0, ab.limit);
            }
        }
        __syncwarp();
    } else if (KD::CONV && warp >= kConvWarp0) {
        // ------------------------------------------------ converters (own CTA's boxes)
        const int ct = static_cast<int>(threadIdx.x) - kConvWarp0 * 32;
        tc::Ring<STAGES> rr;
        tc::Ring<(S::LO_STAGES > 0 ? S::LO_STAGES : 1)> lr;
        bool ok = true;
        for (long long u = cid; ok && u < p.num_units; u += ncl) {
            const WorkUnit wu = work_unit(u, p);
            for (int kb = wu.kb_lo; kb < wu.kb_hi; ++kb) {
                // the raw stage landed; the lo stage's last reader (the MMAs of
                // the stage LO_STAGES back) is done
                if (!warp_wait(&full[rr.s], rr.ph, ab, kStatusWaitFull, lane) ||
                    !warp_wait_cl(&lo_empty[lr.s], lr.ph ^ 1u, ab, kStatusWaitMma)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = smem_u32(base + rr.s * STAGE_BYTES);
                const uint32_t la = smem_u32(lo_base + lr.s * S::LO_BYTES);
                lo_stage<kConvWarps * 32>(sa, la, ct);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) arrive_on(&conv_full[lr.s], 0);
                rr.next();
                lr.next();
            }
        }
    } else {
        // ------------------------------------------------ epilogue (own CTA's rows)
        const int q = warp & 3;
        const int r0 = static_cast<int>(rank) * BM + q * 32;  // this warp's first row
        uint8_t *wbuf = epi + q * S::EPI_WARP_BYTES;
        float4 *stage = reinterpret_cast<float4 *>(wbuf);   // register path: 32 x 32 staging
        uint64_t *wbar = cbar + q * S::EPI_NB;
        // Launched as a programmatic dependent: C may come from the kernel
        // before, whose writes are visible after this wait.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        tc::Ring<2> acc;
        long long gch = 0;  // TMA chunks this warp has handled: buffer gch % EPI_NB
        bool ok = true;
        for (long long u = cid; ok && u < p.num_units; u += ncl) {
            const WorkUnit wu = work_unit(u, p);
            const OutTile o = out_tile<PM, BN>(p, wu);
            const bool tma = p.c_tma && !wu.split;
            const bool use_beta = o.beta != 0.f;
            const int gm = wu.tc.tm * PM + r0, gn = wu.tc.tn * BN, gz = p.Q > 1 ? wu.tc.q : 0;
            tc::prefetch_c_rows(o, r0, lane);
            // C's first chunk is loaded while the accumulator is made
            float4 ca[8], cb[8];
            constexpr int EPI_CH = S::EPI_CH, EPI_BUF = S::EPI_BUF, NCH = BN / EPI_CH;
            if (tma) {
                if (use_beta && lane == 0) {
                    // chunks gch .. gch + EPI_LA - 1: their buffers' last stores
                    // (chunks gch - EPI_NB ..) have read them
                    bulk_wait_read<S::EPI_NB - S::EPI_LA>();
#pragma unroll
                    for (int i = 0; i < S::EPI_LA; ++i) {
                        const int b = static_cast<int>((gch + i) % S::EPI_NB);
                        mbar_arrive_expect_tx(&wbar[b], EPI_BUF);
                        tma_load_3d(wbuf + b * EPI_BUF, &tmC, &wbar[b], gn + i * EPI_CH, gm, gz);
                    }
                }
            } else {
                if (lane == 0) bulk_wait_read<0>();  // TMA stores have read the staging
                __syncwarp();
                tc::load_c_chunk(o, r0, 0, ca, lane);
            }
            int w = 1;
            if (lane == 0) w = wait_cl(&acc_full[acc.s], acc.ph, ab, kStatusWaitAcc, true);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            drain_cl(&acc_full[acc.s], acc.ph, ab.limit);
            tc::tc_fence_after();
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc.s * BN);
            if (tma) {
                // per chunk: the next chunk's C on its way (beta != 0), this
                // chunk's accumulator from TMEM, alpha * acc + beta * C written
                // in place (lane = row, as TMEM holds it), a TMA store
                const int sw = EPI_CH == 32 ? (lane & 7) : ((lane >> 1) & 3);
#pragma unroll 1
                for (int c = 0; c < NCH; ++c, ++gch) {
                    const int b = static_cast<int>(gch % S::EPI_NB);
                    if (use_beta && c + S::EPI_LA < NCH && lane == 0) {
                        const int nb = static_cast<int>((gch + S::EPI_LA) % S::EPI_NB);
                        // chunk gch + EPI_LA - EPI_NB's store has read buffer nb
                        bulk_wait_read<S::EPI_NB - S::EPI_LA - 1>();
                        mbar_arrive_expect_tx(&wbar[nb], EPI_BUF);
                        tma_load_3d(wbuf + nb * EPI_BUF, &tmC, &wbar[nb],
                                    gn + (c + S::EPI_LA) * EPI_CH, gm, gz);
                    }
                    float v[EPI_CH];
                    if constexpr (EPI_CH == 32)
                        tc::tmem_ld32(tbase + c * EPI_CH, v);
                    else
                        tc::tmem_ld16(tbase + c * EPI_CH, v);
                    if (use_beta) {
                        if (!warp_wait(&wbar[b], static_cast<uint32_t>((gch / S::EPI_NB) & 1), ab,
                                       kStatusWaitAcc, lane)) {
                            // the loads of chunks c .. c + EPI_LA - 1 (those of the
                            // tile) may still be owed: wait (bounded) for them
                            // before the teardown
                            for (int i = 0; i < S::EPI_LA && c + i < NCH; ++i)
                                drain_cl(&wbar[(gch + i) % S::EPI_NB],
                                         static_cast<uint32_t>(((gch + i) / S::EPI_NB) & 1),
                                         ab.limit);
                            ok = false;
                            break;
                        }
                    } else {
                        // chunk gch - EPI_NB's store has read buffer b
                        if (lane == 0) bulk_wait_read<S::EPI_NB - 1>();
                        __syncwarp();
                    }
                    const uint32_t row = smem_u32(wbuf + b * EPI_BUF) + lane * (EPI_CH * 4);
#pragma unroll
                    for (int j = 0; j < EPI_CH / 4; ++j) {
                        const uint32_t a = row + static_cast<uint32_t>((j ^ sw) << 4);
                        float4 x = make_float4(o.alpha * v[4 * j], o.alpha * v[4 * j + 1],
                                               o.alpha * v[4 * j + 2], o.alpha * v[4 * j + 3]);
                        if (use_beta) {
                            float4 cv;
                            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                         : "=f"(cv.x), "=f"(cv.y), "=f"(cv.z), "=f"(cv.w)
                                         : "r"(a));
                            x.x = fmaf(o.beta, cv.x, x.x);
                            x.y = fmaf(o.beta, cv.y, x.y);
                            x.z = fmaf(o.beta, cv.z, x.z);
                            x.w = fmaf(o.beta, cv.w, x.w);
                        }
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                     "f"(x.x), "f"(x.y), "f"(x.z), "f"(x.w)
                                     : "memory");
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmC, wbuf + b * EPI_BUF, gn + c * EPI_CH, gm, gz);
                        bulk_commit();
                    }
                }
                if (!ok) break;
            } else {
                // C's next chunk is loaded before the current one is stored
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 64) {
                    float v[32];
                    tc::load_c_chunk(o, r0, c0 + 32, cb, lane);
                    tc::tmem_ld32(tbase + c0, v);
                    tc::store_chunk_pre(o, r0, c0, v, ca, stage, lane);
                    if (c0 + 64 < BN) tc::load_c_chunk(o, r0, c0 + 64, ca, lane);
                    tc::tmem_ld32(tbase + c0 + 32, v);
                    tc::store_chunk_pre(o, r0, c0 + 32, v, cb, stage, lane);
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_on(&acc_empty[acc.s], 0);
            acc.next();
        }
        if (lane == 0) bulk_wait<0>();  // this warp's stores are done before the CTA exits
        __syncwarp();
    }

    // ---- teardown: free TMEM jointly once both CTAs are done
    tc::tc_fence_before();
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace tcs

// Host side: launches the kernel for `plan` (at most `slots` CTA pairs, each
// looping over work units) and, when the plan splits tiles along K, the
// fix-up kernel after it.
// tmA_lo / tmB_lo and a_lo_z / b_lo_z: the lo planes' maps and batch
// offsets (3xTF32; ignored otherwise).
template <class KD>
int launch_ss(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB,
              const CUtensorMap &tmA_lo, const CUtensorMap &tmB_lo, int a_lo_z, int b_lo_z,
              int slots)
{
    auto kern = tcs::tcs_gemm_kernel<KD>;
    constexpr int smem = tcs::Shape<KD>::SMEM_BYTES;
    if (!smem_attr_once(reinterpret_cast<const void *>(kern), smem)) return SGEMM_ERR_LAUNCH;
    long long pairs = plan.p.num_units;
    if (pairs > slots) pairs = slots;
    // programmatic dependent launch: the CTAs' set-up (barriers, TMEM,
    // descriptor prefetch) overlaps the end of the kernel before
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(tcs::Shape<KD>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = plan.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // C by TMA in the epilogue when its rows and batches suit TMA
    alignas(64) CUtensorMap tmC;
    std::memset(&tmC, 0, sizeof(tmC));
    const GemmParams &p = plan.p;
    plan.p.c_tma = p.c_vec4 && encode_c_tiles(&tmC, p.C, p.M, p.N, p.ldc, p.Q, p.sC,
                                              tcs::Shape<KD>::EPI_CH)
                       ? 1
                       : 0;
    if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmA_lo, tmB_lo, tmC, plan.p, a_lo_z, b_lo_z) !=
        cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    note_launch();
    return plan.p.splits > 1 ? launch_fixup(plan, tcs::PM, tcs::BN) : SGEMM_OK;
}

}  // namespace sg
