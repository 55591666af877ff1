// tc_tf32.cuh -- building blocks of the tcgen05 tensor-core SGEMM kernels
// (3xTF32 and TF32): PTX wrappers (TMEM allocation, MMA, commit, TMEM loads
// and stores), the TF32 split, the A and B converters and the epilogue
// store.  The kernels are tc_pair.cuh (TMA-fed, CTA pairs) and
// tc_direct.cuh (operands TMA cannot describe).
//
// C = alpha * op(A) @ op(B) + beta * C with fp32 inputs and output, the
// contraction on the 5th-generation tensor cores ("Tensor cores" in the
// future-work list of "From 1% to 94% of cuBLAS, one kernel at a time": TF32
// inputs raise peak throughput and turn the problem back into a
// data-movement one).  Accumulators live in tensor memory (TMEM), as the
// "TMEM-friendly block sizes" item of "Triton Optimization Reference (cuTile
// -> Triton)", section 9.4, describes for Blackwell.
//
// FP32 accuracy from TF32 units (3xTF32): every operand value x is split
// into hi = x with the 13 low mantissa bits cleared (a TF32 value) and
// lo = (x - hi) likewise truncated (x - hi is exact in fp32); the product a*b
// is accumulated in fp32 as lo_a*hi_b + hi_a*lo_b + hi_a*hi_b, small terms
// first.  |lo| < 2^-10 |x|, so the dropped lo_a*lo_b and the truncation of
// the two lo terms are each below 2^-20 |a||b|.  Plain TF32 issues
// hi_a*hi_b only, with hi rounded to nearest (ties away) for accuracy
// margin.
//
// Data flow per output tile and 32-wide k-block (both kernels):
//   raw fp32 A and B tiles -> shared memory (TMA, or the direct kernel's
//                      own loads)
//   A converters       raw A rows -> hi/lo planes in TMEM (tcgen05.st); the
//                      MMA reads A from TMEM, so A's split planes never
//                      touch shared memory
//   B converters       raw B tile -> hi/lo planes in shared memory, K-major
//                      with the 128-byte swizzle (N-inner tiles transposed)
//   MMA (one thread)   tcgen05.mma kind::tf32, K=8, A from TMEM, B by
//                      shared-memory descriptor, into one of two TMEM
//                      accumulator buffers
//   epilogue           tcgen05.ld of the other buffer; C = alpha*acc + beta*C
// Warp roles: 0 producer, 1 TMEM allocator + MMA issuer, 2-5 A converters
// (warp w owns TMEM lanes 32*(w%4) .. +31, i.e. those rows of A), 6-9 B
// converters, 10-13 epilogue (lane quarter w%4).
#pragma once

#include <type_traits>

#include "common.cuh"

namespace sg {
namespace tc {

constexpr int BM = 128;   // UMMA M (one CTA)
constexpr int BK = 32;    // k per stage: one 128-byte swizzle row of fp32
constexpr int UK = 8;     // k per tcgen05.mma of kind::tf32
constexpr int kAConvWarp0 = 2;                   // warps 2-5: A -> TMEM
constexpr int kBConvWarp0 = 6, kBConvWarps = 4;  // warps 6-9: B -> shared memory
constexpr int kBConvThreads = kBConvWarps * 32;
constexpr int kEpiWarp0 = kBConvWarp0 + kBConvWarps;  // warps 10-13: epilogue
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kConvWarps = 4 + kBConvWarps;      // arrivals that complete a stage
constexpr uint32_t kTmemCols = 512;

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory writes by threads become visible to the tensor core (async
// proxy) only after this fence.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::tf32, one CTA.  A is M rows (TMEM
// lanes) by K fp32 columns starting at a_tmem.
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier receives one arrival when every tcgen05 operation this
// thread issued before the commit has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one per lane).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Loads 16 consecutive fp32 columns from this warp's 32 TMEM lanes (lane l:
// row l of the warp's quarter) and waits for them.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Stores 16 consecutive fp32 columns into this warp's 32 TMEM lanes (one row
// per lane).  Completion is awaited with tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Round to the nearest TF32 value (10 explicit mantissa bits), ties away.
__device__ __forceinline__ float to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// x with its 13 low mantissa bits cleared: a TF32 value.
__device__ __forceinline__ float trunc_tf32(float x)
{
    return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// The operand planes of one value: 3xTF32 -> (hi, lo) truncated split,
// TF32 -> hi rounded to nearest.
template <bool SPLIT3>
__device__ __forceinline__ void split_value(float x, float &hi, float &lo)
{
    if (SPLIT3) {
        hi = trunc_tf32(x);
        lo = trunc_tf32(x - hi);  // x - hi is exact
    } else {
        hi = to_tf32(x);
        lo = 0.f;
    }
}

// Shared-memory matrix descriptor of a K-major operand tile stored as
// 128-byte rows (32 fp32 of K) with the 128-byte swizzle: 8-row atoms of
// 1024 bytes stacked along M/N (stride byte offset 1024).  The leading byte
// offset is unused for this layout (K of one MMA stays inside one row).
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                        // leading byte offset (16 B)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                        // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                        // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::tf32, fp32 accumulate, both operands K-major,
// M = 128, N = BN.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_tf32()
{
    return (1u << 4)                  // D format: f32
           | (2u << 7)                // A format: tf32
           | (2u << 10)               // B format: tf32
           | (static_cast<uint32_t>(BN >> 3) << 17)   // N / 8
           | (static_cast<uint32_t>(BM >> 4) << 24);  // M / 16
}

// ------------------------------------------------------------ converters

// Ring position walker: stage index and round parity, advanced per use.
template <int N>
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next()
    {
        if (++s == N) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// A converter: this thread's row of the raw A tile (row = TMEM lane) ->
// hi (and lo) planes in TMEM columns [t_hi, t_hi+32) and [t_lo, t_lo+32).
// K-inner raw A is swizzled 128-byte rows (TMA's SWIZZLE_128B layout):
// chunk c of row r sits at chunk c ^ (r mod 8).  M-inner raw A is [32 k][128 m].
template <bool KIN, bool SPLIT3>
__device__ __forceinline__ void convert_a_row(const uint8_t *raw_a, int row, uint32_t t_hi,
                                              uint32_t t_lo)
{
    const uint32_t base = smem_u32(raw_a);
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // 16 k per half
        float x[16];
        if (KIN) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int chunk = half * 4 + c;
                const uint32_t a = base + row * 128 + (((chunk ^ row) & 7) << 4);
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(x[4 * c]), "=f"(x[4 * c + 1]), "=f"(x[4 * c + 2]),
                               "=f"(x[4 * c + 3])
                             : "r"(a));
            }
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t a = base + ((half * 16 + k) * BM + row) * 4;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(x[k]) : "r"(a));
            }
        }
        float h[16], l[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) split_value<SPLIT3>(x[k], h[k], l[k]);
        tmem_st16(t_hi + half * 16, h);
        if (SPLIT3) tmem_st16(t_lo + half * 16, l);
    }
}

// B converter: one raw B tile (R = BN rows of B^T, BK k) -> K-major swizzled
// hi (and lo) planes in shared memory.  K-inner raw tiles already have that
// layout (TMA wrote them with the same swizzle): the split is element-wise.
// N-inner raw tiles ([BK][R], unswizzled) are transposed in 4 x 4 blocks;
// the block assignment (k-block rotated by lane/2) keeps each quarter-warp's
// 16-byte loads and stores on eight distinct bank groups.
template <int R, bool KIN, bool SPLIT3>
__device__ __forceinline__ void convert_b_tile(const uint8_t *raw, uint8_t *hi, uint8_t *lo,
                                               int ct)
{
    const uint32_t raw_a = smem_u32(raw), hi_a = smem_u32(hi), lo_a = smem_u32(lo);
    if constexpr (KIN) {
        constexpr int CHUNKS = R * BK / 4;  // 16-byte chunks
#pragma unroll 4
        for (int c = ct; c < CHUNKS; c += kBConvThreads) {
            float4 x;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                         : "r"(raw_a + c * 16));
            float4 h, l;
            split_value<SPLIT3>(x.x, h.x, l.x);
            split_value<SPLIT3>(x.y, h.y, l.y);
            split_value<SPLIT3>(x.z, h.z, l.z);
            split_value<SPLIT3>(x.w, h.w, l.w);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(hi_a + c * 16),
                         "f"(h.x), "f"(h.y), "f"(h.z), "f"(h.w)
                         : "memory");
            if (SPLIT3) {
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(lo_a + c * 16),
                             "f"(l.x), "f"(l.y), "f"(l.z), "f"(l.w)
                             : "memory");
            }
        }
    } else if constexpr (R == 64) {
        // Half a B tile (the CTA-pair kernel): 16 row blocks x 8 k-blocks of
        // 4, one per thread.  Within each 8-lane phase the row blocks are 8
        // consecutive 16-byte pieces (distinct banks) for the loads, and the
        // k-block rotation by lane/2 puts the stores on 8 distinct chunks.
        static_assert(kBConvThreads == 128, "one 4 x 4 block per converter thread");
        const int warp = ct >> 5, lane = ct & 31;
        const int rb4 = lane & 15;
        const int kb4 = (2 * warp + (lane >> 4) + (lane >> 1)) & 7;
        float v[4][4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a = raw_a + ((4 * kb4 + kk) * R + 4 * rb4) * 4;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v[kk][0]), "=f"(v[kk][1]), "=f"(v[kk][2]), "=f"(v[kk][3])
                         : "r"(a));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * rb4 + i;
            const uint32_t off = sw128_offset(r, 4 * kb4);
            float h[4], l[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) split_value<SPLIT3>(v[kk][i], h[kk], l[kk]);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(hi_a + off), "f"(h[0]),
                         "f"(h[1]), "f"(h[2]), "f"(h[3])
                         : "memory");
            if (SPLIT3)
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(lo_a + off),
                             "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3])
                             : "memory");
        }
    } else {
        // raw: element (k, r) at (k*R + r)*4.  out: element (r, k) at sw128_offset(r, k).
        const int warp = ct >> 5, lane = ct & 31;
        constexpr int RB4 = R / 4;                // 4-row blocks along R
        constexpr int PASSES = RB4 / 32;          // lanes cover 32 row blocks per pass
        constexpr int SHARE = 8 / kBConvWarps;    // k-blocks of 4 per warp and row block
        static_assert(8 % kBConvWarps == 0, "converter warps must divide the 8 k-blocks");
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
            const int rb4 = pass * 32 + lane;
#pragma unroll
            for (int sh = 0; sh < SHARE; ++sh) {
                // the warps x SHARE cover the 8 k-blocks of 4 for every rb4
                const int kb4 = (warp * SHARE + sh + (lane >> 1)) & 7;
                float v[4][4];  // v[kk][i] = raw(k = 4kb4+kk, r = 4rb4+i)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t a = raw_a + ((4 * kb4 + kk) * R + 4 * rb4) * 4;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v[kk][0]), "=f"(v[kk][1]), "=f"(v[kk][2]), "=f"(v[kk][3])
                                 : "r"(a));
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * rb4 + i;
                    const uint32_t off = sw128_offset(r, 4 * kb4);
                    float h[4], l[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) split_value<SPLIT3>(v[kk][i], h[kk], l[kk]);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(hi_a + off),
                                 "f"(h[0]), "f"(h[1]), "f"(h[2]), "f"(h[3])
                                 : "memory");
                    if (SPLIT3)
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(lo_a + off),
                                     "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3])
                                     : "memory");
                }
            }
        }
    }
}

// ---- epilogue through a per-warp staging buffer --------------------------
// A warp's accumulator chunk arrives one row per lane (TMEM lane = row), so a
// direct store covers 32 rows x 16 B per warp instruction: 32 lines, half a
// sector of each, and as many L1 wavefronts, which the converters' shared-
// memory traffic then waits behind.  Transposed through 4 KB of shared
// memory, each group of 8 lanes writes 128 contiguous bytes of one row (a
// warp instruction covers 4 rows x 128 B, whole lines).  The 16-byte slots of
// a staged row are XOR-swizzled by (row & 7), so both the row-per-lane
// writes and the row-per-8-lanes reads are free of bank conflicts.
constexpr int kStageFloats = 32 * 32;  // one warp's chunk

// Asks L2 for the lines of C a warp's epilogue will read (rows [r0, r0 + 32)
// of the tile, lane l row r0 + l), when beta != 0.  Issued as soon as the
// tile is known, before its accumulator is ready, so that the epilogue's
// loads find C in L2 instead of waiting on DRAM twice per chunk.  Only
// addresses inside the tile's valid extent are touched.
__device__ __forceinline__ void prefetch_c_rows(const OutTile &o, int r0, int lane)
{
    const int r = r0 + lane;
    if (o.beta == 0.f || r >= o.rows || o.cols <= 0) return;
    const float *row = o.base + static_cast<long long>(r) * o.ld;
    for (int c = 0; c < o.cols; c += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + c));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + o.cols - 1));
}

// out = alpha * v + beta * out for chunk [c0, c0 + 32) of rows [r0, r0 + 32)
// (lane l holds row r0 + l in v; out is not read when beta == 0), masked at
// the M/N edges; stage is this warp's kStageFloats-float buffer (16-byte
// aligned).  After the transpose, lane l handles slot i = 0..7: row
// r0 + 4 i + l / 8, columns c0 + 4 (l % 8) .. + 3, in two batches of four
// slots whose loads of C are issued together, before their stores.
__device__ __forceinline__ void store_chunk_staged(const OutTile &o, int r0, int c0,
                                                   const float (&v)[32], float4 *stage, int lane)
{
    float4 *mine = stage + lane * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        mine[j ^ (lane & 7)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    const int g = lane & 7, col = c0 + 4 * g;
    const bool full = o.vec4 && col + 4 <= o.cols;
    const bool use_beta = o.beta != 0.f;
    const long long step = 4 * o.ld;  // 4 rows
    const int rl = r0 + (lane >> 3);
    float *row = o.base + static_cast<long long>(rl) * o.ld + col;
#pragma unroll
    for (int h = 0; h < 8; h += 4) {  // two batches of four slots
        float4 old[4];
        if (use_beta) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float *src = row + i * step;
                old[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (rl + 4 * (h + i) >= o.rows) continue;
                if (full) {
                    old[i] = *reinterpret_cast<const float4 *>(src);
                } else {
                    if (col < o.cols) old[i].x = src[0];
                    if (col + 1 < o.cols) old[i].y = src[1];
                    if (col + 2 < o.cols) old[i].z = src[2];
                    if (col + 3 < o.cols) old[i].w = src[3];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = 4 * (h + i) + (lane >> 3);
            const float4 a = stage[rr * 8 + (g ^ (rr & 7))];
            if (rl + 4 * (h + i) >= o.rows) continue;
            float4 x = make_float4(o.alpha * a.x, o.alpha * a.y, o.alpha * a.z, o.alpha * a.w);
            if (use_beta) {
                x.x = fmaf(o.beta, old[i].x, x.x);
                x.y = fmaf(o.beta, old[i].y, x.y);
                x.z = fmaf(o.beta, old[i].z, x.z);
                x.w = fmaf(o.beta, old[i].w, x.w);
            }
            float *dst = row + i * step;
            if (full) {
                *reinterpret_cast<float4 *>(dst) = x;
            } else {
                if (col < o.cols) dst[0] = x.x;
                if (col + 1 < o.cols) dst[1] = x.y;
                if (col + 2 < o.cols) dst[2] = x.z;
                if (col + 3 < o.cols) dst[3] = x.w;
            }
        }
        row += 4 * step;
    }
    __syncwarp();  // the next chunk reuses the buffer
}

// The staged epilogue in two halves, so that the loads of C can run ahead:
// load_c_chunk issues the loads of the C values a lane combines for chunk
// [c0, c0 + 32) of rows [r0, r0 + 32) (slot i = 0..7: row r0 + 4 i + l / 8,
// columns c0 + 4 (l % 8) .. + 3, as in store_chunk_staged; zeros outside the
// tile's valid extent, nothing when beta == 0), and store_chunk_pre writes
// out = alpha * v + beta * old for that chunk.  A caller loads chunk j + 1's
// C before it stores chunk j: eight 16-byte loads per lane stay in flight
// behind the transpose and the stores (store_chunk_staged has four).
__device__ __forceinline__ void load_c_chunk(const OutTile &o, int r0, int c0, float4 (&old)[8],
                                             int lane)
{
    const int col = c0 + 4 * (lane & 7);
    const bool full = o.vec4 && col + 4 <= o.cols;
    const int rl = r0 + (lane >> 3);
    const float *row = o.base + static_cast<long long>(rl) * o.ld + col;
    const long long step = 4 * o.ld;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        old[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (o.beta == 0.f || rl + 4 * i >= o.rows || col >= o.cols) continue;
        const float *src = row + i * step;
        if (full) {
            old[i] = *reinterpret_cast<const float4 *>(src);
        } else {
            old[i].x = src[0];
            if (col + 1 < o.cols) old[i].y = src[1];
            if (col + 2 < o.cols) old[i].z = src[2];
            if (col + 3 < o.cols) old[i].w = src[3];
        }
    }
}

__device__ __forceinline__ void store_chunk_pre(const OutTile &o, int r0, int c0,
                                                const float (&v)[32], const float4 (&old)[8],
                                                float4 *stage, int lane)
{
    float4 *mine = stage + lane * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        mine[j ^ (lane & 7)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    const int g = lane & 7, col = c0 + 4 * g;
    const bool full = o.vec4 && col + 4 <= o.cols;
    const int rl = r0 + (lane >> 3);
    float *row = o.base + static_cast<long long>(rl) * o.ld + col;
    const long long step = 4 * o.ld;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3);
        const float4 a = stage[rr * 8 + (g ^ (rr & 7))];
        if (rl + 4 * i >= o.rows || col >= o.cols) continue;
        float4 x = make_float4(o.alpha * a.x, o.alpha * a.y, o.alpha * a.z, o.alpha * a.w);
        if (o.beta != 0.f) {
            x.x = fmaf(o.beta, old[i].x, x.x);
            x.y = fmaf(o.beta, old[i].y, x.y);
            x.z = fmaf(o.beta, old[i].z, x.z);
            x.w = fmaf(o.beta, old[i].w, x.w);
        }
        float *dst = row + i * step;
        if (full) {
            *reinterpret_cast<float4 *>(dst) = x;
        } else {
            dst[0] = x.x;
            if (col + 1 < o.cols) dst[1] = x.y;
            if (col + 2 < o.cols) dst[2] = x.z;
            if (col + 3 < o.cols) dst[3] = x.w;
        }
    }
    __syncwarp();  // the next chunk reuses the buffer
}

}  // namespace tc
}  // namespace sg
