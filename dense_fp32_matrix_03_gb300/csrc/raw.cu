// raw.cu -- the tensor-core paths on the caller's fp32 matrices as stored.
//
// kind::tf32 reads the 19 high bits of each 32-bit operand value (sign,
// exponent, 10 explicit mantissa bits) and ignores the 13 low mantissa
// bits, so an fp32 matrix is a TF32 operand as it stands: TMA stages it
// straight from the caller's pointer into the MMA's layout -- K-major when
// its rows run along K (A stored M x K, B stored N x K), M/N-major otherwise
// (A stored K x M, B stored K x N).  Then
//   - TF32: one MMA per k step on the raw operands, each value truncated to
//     TF32 by the tensor core; no pass and no workspace beyond split-K;
//   - 3xTF32: the raw operands are the hi planes (hi = x with its 13 low
//     mantissa bits cleared, which is what the tensor core reads); a pass
//     writes each operand's lo plane, lo = (x - hi) with its 13 low mantissa
//     bits cleared, in the operand's own layout (element by element, no
//     transposition), and the product multiplies hi*hi + hi*lo + lo*hi per k
//     step -- the same values and the same order as the planes route
//     (planes.cu), whose pass writes both planes.
// Against the planes route the pass moves two bytes per operand byte
// instead of three (3xTF32) or none instead of two (TF32).  The product is
// tcs_gemm_kernel (tc_ss.cuh): 256 x 256 tiles on CTA pairs.
//
// Lo plane of an operand stored as E entries of `outer` rows of `inner`
// values (inner = K for K-inner operands, else M or N): value (q, r, c) at
// (q * outer + r) * ldl + c, ldl = round_up(inner, 32), so that its rows
// start on 128-byte boundaries (whole L2 lines for TMA, whatever the
// source's pitch).
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_ss.cuh"

namespace sg {

namespace {

constexpr int kGroupM = 8;
constexpr int kColV4 = 64;  // float4 columns per lo-pass block
constexpr int kRowsPB = 4;  // rows per lo-pass block (256 threads)

long long round32(long long x) { return (x + 31) / 32 * 32; }
size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// One operand of the lo pass.
struct LoOperand {
    const float *src;
    long long lds, sstride;  // source row pitch and batch stride (elements)
    float *dst;
    long long ldl;           // lo plane row pitch (elements); entries are outer * ldl apart
    int outer, inner, E;     // stored rows, values per row, stored batch entries
    int zblocks;             // grid z-slices that walk this operand's entries
};

// lo of four values: x - (x with its 13 low mantissa bits cleared) is exact;
// its own 13 low mantissa bits are cleared as well.
__device__ __forceinline__ float lo_tf32(float x)
{
    return tc::trunc_tf32(x - tc::trunc_tf32(x));
}

// One float4 group of a row: 16-byte load when the group lies inside the
// row, value by value (zeros past `inner`) at its ragged end.
__device__ __forceinline__ float4 load_group(const float *sp, int c, int inner)
{
    if (c + 4 <= inner) return __ldg(reinterpret_cast<const float4 *>(sp));
    float4 v;
    v.x = sp[0];
    v.y = c + 1 < inner ? sp[1] : 0.f;
    v.z = c + 2 < inner ? sp[2] : 0.f;
    v.w = 0.f;
    return v;
}

__device__ __forceinline__ float4 lo_group(float4 v)
{
    return make_float4(lo_tf32(v.x), lo_tf32(v.y), lo_tf32(v.z), lo_tf32(v.w));
}

// The lo pass over both operands in one launch.  Block (x, y, z), 256
// threads: thread t takes float4 column x * 64 + t % 64 of rows y * 4 +
// t / 64, strided by the grid's rows (two rows per step, both loads issued
// before either store); z-slices [0, a.zblocks) walk A's entries, the rest
// B's.  A warp reads and writes 512 contiguous bytes of one row.  Sources
// are 16-byte aligned with pitches and batch strides in multiples of four
// values (the raw route's TMA rule); a row's last group of four is read value
// by value when it runs past `inner`, and written with zeros there.
__global__ void __launch_bounds__(256) lo_pass_kernel(LoOperand a, LoOperand b)
{
    const bool is_a = static_cast<int>(blockIdx.z) < a.zblocks;
    const LoOperand &o = is_a ? a : b;
    const int z0 = is_a ? static_cast<int>(blockIdx.z) : static_cast<int>(blockIdx.z) - a.zblocks;
    const int c = (static_cast<int>(blockIdx.x) * kColV4 + (threadIdx.x & (kColV4 - 1))) * 4;
    if (c >= o.inner) return;
    const int ty = threadIdx.x / kColV4;
    const int step = static_cast<int>(gridDim.y) * kRowsPB;
    for (int q = z0; q < o.E; q += o.zblocks) {
        const float *sq = o.src + static_cast<long long>(q) * o.sstride + c;
        float *dq = o.dst + static_cast<long long>(q) * o.outer * o.ldl + c;
        for (int r = static_cast<int>(blockIdx.y) * kRowsPB + ty; r < o.outer; r += 2 * step) {
            const bool two = r + step < o.outer;
            const float4 v0 = load_group(sq + static_cast<long long>(r) * o.lds, c, o.inner);
            float4 v1 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (two) v1 = load_group(sq + static_cast<long long>(r + step) * o.lds, c, o.inner);
            *reinterpret_cast<float4 *>(dq + static_cast<long long>(r) * o.ldl) = lo_group(v0);
            if (two)
                *reinterpret_cast<float4 *>(dq + static_cast<long long>(r + step) * o.ldl) =
                    lo_group(v1);
        }
    }
}

// Stored shape of an operand: `outer` rows of `inner` values.
struct Stored {
    long long outer, inner;
};
Stored stored_a(const Plan &plan)
{
    return plan.transA ? Stored{plan.p.K, plan.p.M} : Stored{plan.p.M, plan.p.K};
}
Stored stored_b(const Plan &plan)
{
    return plan.transB ? Stored{plan.p.N, plan.p.K} : Stored{plan.p.K, plan.p.N};
}

size_t lo_bytes(const Stored &s, int E)
{
    return round256(static_cast<size_t>(E) * s.outer * round32(s.inner) * sizeof(float));
}

LoOperand lo_operand(const float *src, long long lds, long long sstride, const Stored &s, int E,
                     float *dst)
{
    LoOperand o;
    o.src = src;
    o.lds = lds;
    o.sstride = sstride;
    o.dst = dst;
    o.ldl = round32(s.inner);
    o.outer = static_cast<int>(s.outer);
    o.inner = static_cast<int>(s.inner);
    o.E = E;
    o.zblocks = E < 16 ? E : 16;
    return o;
}

int launch_lo_pass(const LoOperand &a, const LoOperand &b, int num_sms, cudaStream_t stream)
{
    const long long cols = (round32(a.inner > b.inner ? a.inner : b.inner) / 4 + kColV4 - 1) / kColV4;
    const long long rows = a.outer > b.outer ? a.outer : b.outer;
    // enough blocks to keep every multiprocessor's loads in flight (8 per
    // multiprocessor), the rows strided beyond that
    long long gy = (rows + kRowsPB - 1) / kRowsPB;
    const long long zs = a.zblocks + b.zblocks;
    const long long want = 8LL * num_sms;
    if (cols * gy * zs > want) {
        gy = (want + cols * zs - 1) / (cols * zs);
        if (gy < 1) gy = 1;
    }
    if (cols > 0x7FFFFFFFLL || gy > 65535 || zs > 65535) return SGEMM_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(cols), static_cast<unsigned>(gy),
                    static_cast<unsigned>(zs));
    lo_pass_kernel<<<grid, 256, 0, stream>>>(a, b);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

// Tensor map of an operand (or of its lo plane) for the shared-memory
// operand kernel: K-major boxes of 32 k by `rows_box` rows, or M/N-major
// boxes of 32 rows-inner values by 32 k.
// Every stored row of the operand starts on a 128-byte boundary.
bool rows_on_lines(const float *base, long long ld, int E, long long stride)
{
    return (reinterpret_cast<uintptr_t>(base) & 127) == 0 && ld % 32 == 0 &&
           (E <= 1 || stride % 32 == 0);
}

bool encode_raw(CUtensorMap *map, const float *base, bool mn, long long rows, long long K,
                long long ld, int E, long long stride, int rows_box)
{
    // 256-byte L2 fills only when every row starts on a 128-byte boundary
    const bool lines = rows_on_lines(base, ld, E, stride);
    return mn ? encode_operand_mn(map, base, rows, K, ld, E, stride, lines)
              : encode_operand(map, base, true, rows, K, ld, E, stride, rows_box, lines);
}

// CONV: 3xTF32 with the lo planes made in the kernel (tmAl / tmBl unused).
template <int PLANES, bool CONV = false>
int launch_raw_product(Plan &plan, bool a_mn, bool b_mn, const CUtensorMap &tmA,
                       const CUtensorMap &tmB, const CUtensorMap &tmAl, const CUtensorMap &tmBl,
                       int slots)
{
    using namespace tcs;
    if (!a_mn && !b_mn)
        return launch_ss<KindTF32<PLANES, false, false, CONV>>(plan, tmA, tmB, tmAl, tmBl, 0, 0, slots);
    if (!a_mn && b_mn)
        return launch_ss<KindTF32<PLANES, false, true, CONV>>(plan, tmA, tmB, tmAl, tmBl, 0, 0, slots);
    if (a_mn && !b_mn)
        return launch_ss<KindTF32<PLANES, true, false, CONV>>(plan, tmA, tmB, tmAl, tmBl, 0, 0, slots);
    return launch_ss<KindTF32<PLANES, true, true, CONV>>(plan, tmA, tmB, tmAl, tmBl, 0, 0, slots);
}

}  // namespace

size_t raw_lo_bytes_max(int mode, long long M, long long N, long long K, int QA, int QB)
{
    if (mode != SGEMM_MODE_3XTF32) return 0;
    const size_t a1 = lo_bytes(Stored{M, K}, QA), a2 = lo_bytes(Stored{K, M}, QA);
    const size_t b1 = lo_bytes(Stored{N, K}, QB), b2 = lo_bytes(Stored{K, N}, QB);
    return (a1 > a2 ? a1 : a2) + (b1 > b2 ? b1 : b2);
}

int raw_choice(int mode, long long M, long long N, long long K, int QA, int QB, int Q,
               int num_sms, bool lines)
{
    if ((mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32) || num_sms <= 0) return kRawNone;
    if (K > 0x7FFFFFFFLL) return kRawNone;
    const int slots = tc_pair_slots(num_sms);
    const size_t any = ~static_cast<size_t>(0);
    int bm = 0, bn = 0;
    tc_tile_dims(mode, static_cast<int>(K), true, bm, bn);
    const long long pair_tiles =
        static_cast<long long>(Q) * ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
    const double t_pair =
        choose_plan(pair_tiles, static_cast<int>(K), slots, mode, bm, bn, kFeedPair, any).seconds;
    const long long ss_tiles =
        static_cast<long long>(Q) * ((M + tcs::PM - 1) / tcs::PM) * ((N + tcs::BN - 1) / tcs::BN);
    auto product = [&](int feed) {
        return choose_plan(ss_tiles, static_cast<int>(K), slots, mode, tcs::PM, tcs::BN, feed, any)
            .seconds;
    };
    const double elems = static_cast<double>(QA * M + QB * N) * K;
    const bool split3 = mode == SGEMM_MODE_3XTF32;
    const double t_planes =
        product(kFeedPlanes) + elems * 4.0 * (split3 ? 3.0 : 2.0) / 6.0e12 + 7e-6;
    const double t_raw = split3 ? product(kFeedInline) * (lines ? 1.0 : 1.06)
                                : product(kFeedPlanes) * (lines ? 1.0 : 1.27);
    if (t_raw < t_pair && t_raw < t_planes) return split3 ? kRawInline : kRawPlain;
    return kRawNone;
}

int run_raw(Plan &plan, bool &taken, bool force, int route)
{
    taken = false;
    GemmParams &p = plan.p;
    if (plan.mode != SGEMM_MODE_3XTF32 && plan.mode != SGEMM_MODE_TF32) return SGEMM_OK;
    if (!plan.a_tma || !plan.b_tma) return SGEMM_OK;
    const int planes = plan.mode == SGEMM_MODE_3XTF32 ? 2 : 1;
    const int QA = (p.Q > 1 && p.sA != 0) ? p.Q : 1, QB = (p.Q > 1 && p.sB != 0) ? p.Q : 1;
    if (!force) {
        const bool lines =
            rows_on_lines(p.A, p.lda, QA, p.sA) && rows_on_lines(p.B, p.ldb, QB, p.sB);
        if (raw_choice(plan.mode, p.M, p.N, p.K, QA, QB, p.Q, plan.num_sms, lines) == kRawNone)
            return SGEMM_OK;
    }
    // 3xTF32: lo planes from a pass into the workspace (forced RAW) or made
    // in the product kernel (INLINE, and the cost models' choice)
    const bool inline_lo = planes == 2 && (!force || route == kRouteTcInline);
    const bool lo_pass = planes == 2 && !inline_lo;
    if (lo_pass && plan.ws == nullptr) return SGEMM_OK;
    const bool a_mn = plan.transA != 0, b_mn = plan.transB == 0;
    const Stored sa = stored_a(plan), sb = stored_b(plan);
    const size_t a_lo = lo_pass ? lo_bytes(sa, QA) : 0;
    const size_t need = lo_pass ? a_lo + lo_bytes(sb, QB) : 0;
    if (need > plan.ws_bytes) return SGEMM_OK;
    if (sa.outer > 0x7FFFFFFFLL || sb.outer > 0x7FFFFFFFLL) return SGEMM_OK;

    alignas(64) CUtensorMap tmA, tmB, tmAl, tmBl;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    std::memset(&tmAl, 0, sizeof(tmAl));
    std::memset(&tmBl, 0, sizeof(tmBl));
    if (!encode_raw(&tmA, p.A, a_mn, p.M, p.K, p.lda, p.Q, p.sA, tcs::BM) ||
        !encode_raw(&tmB, p.B, b_mn, p.N, p.K, p.ldb, p.Q, p.sB, tcs::HN))
        return SGEMM_OK;
    char *w = static_cast<char *>(plan.ws);
    float *la = nullptr, *lb = nullptr;
    if (lo_pass) {
        la = reinterpret_cast<float *>(w);
        lb = reinterpret_cast<float *>(w + a_lo);
        const long long lda_l = round32(sa.inner), ldb_l = round32(sb.inner);
        if (!encode_raw(&tmAl, la, a_mn, p.M, p.K, lda_l, QA, sa.outer * lda_l, tcs::BM) ||
            !encode_raw(&tmBl, lb, b_mn, p.N, p.K, ldb_l, QB, sb.outer * ldb_l, tcs::HN))
            return SGEMM_OK;
    } else {
        tmAl = tmA;
        tmBl = tmB;
    }
    taken = true;

    if (lo_pass) {
        const LoOperand oa = lo_operand(p.A, p.lda, p.sA, sa, QA, la);
        const LoOperand ob = lo_operand(p.B, p.ldb, p.sB, sb, QB, lb);
        const int rc = launch_lo_pass(oa, ob, plan.num_sms, plan.stream);
        if (rc != SGEMM_OK) return rc;
        plan.ws = need < plan.ws_bytes ? static_cast<void *>(w + need) : nullptr;
        plan.ws_bytes = need < plan.ws_bytes ? plan.ws_bytes - need : 0;
    }

    // the batch coordinate of the maps (entries stored; broadcast: 0)
    p.a_q_step = QA > 1 ? 1 : 0;
    p.b_q_step = QB > 1 ? 1 : 0;
    const int stage_k = planes == 2 ? tcs::Shape<tcs::KindTF32<2>>::STAGE_K
                                    : tcs::Shape<tcs::KindTF32<1>>::STAGE_K;
    p.k_blocks = (p.K + stage_k - 1) / stage_k;
    p.group_m = kGroupM;
    p.tiles_m = (p.M + tcs::PM - 1) / tcs::PM;
    p.tiles_n = (p.N + tcs::BN - 1) / tcs::BN;
    p.num_tiles = static_cast<long long>(p.Q) * p.tiles_m * p.tiles_n;
    const int slots = ss_slots(plan.num_sms);
    const int rc = plan_splits(plan, tcs::PM, tcs::BN, inline_lo ? kFeedInline : kFeedPlanes, slots);
    if (rc != SGEMM_OK) return rc;
    if (planes == 1) return launch_raw_product<1>(plan, a_mn, b_mn, tmA, tmB, tmAl, tmBl, slots);
    return inline_lo ? launch_raw_product<2, true>(plan, a_mn, b_mn, tmA, tmB, tmAl, tmBl, slots)
                     : launch_raw_product<2>(plan, a_mn, b_mn, tmA, tmB, tmAl, tmBl, slots);
}

}  // namespace sg
