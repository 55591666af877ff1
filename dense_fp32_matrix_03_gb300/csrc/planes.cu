// planes.cu -- the tensor-core paths with a workspace: operands rewritten
// into TF32 planes, then the product on the shared-memory-operand kernel.
//
// The CTA-pair kernel of tc_pair.cuh converts each stage of fp32 operands
// inside the main loop (rounding or hi/lo split, A into TMEM, B into shared
// memory); that work shares the multiprocessor's shared-memory bandwidth and
// issue slots with the MMAs.  With room in the caller's workspace the
// conversion is done once instead, by a pass over each operand that writes
// it K-major with rows padded to whole 128-byte lines, as
//   - TF32: one plane, each value rounded to the nearest TF32 value;
//   - 3xTF32: two planes, hi = the value with its 13 low mantissa bits
//     cleared and lo = (value - hi) likewise (tc::split_value),
// and the product runs on tcs_gemm_kernel (tc_ss.cuh), which TMA feeds
// with both operands straight into the MMA's layout.  The pass (one launch
// for both operands) reads each operand once and writes its planes once
// (HBM-bound).
//
// Plane layout of an operand with R rows (M for A, N for B) and E stored
// batch entries (1 when broadcast): value (pl, q, r, k) at
// ((pl * E + q) * R + r) * ldp + k, ldp = round_up(K, 32), so that one 3-D
// tensor map covers every plane and entry (entry pl * E + q).
#include <atomic>
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_ss.cuh"

namespace sg {

namespace {

constexpr int kT = 64;         // transpose tile edge
constexpr int kThreads = 256;  // threads per pass block
constexpr int kGroupM = 8;
constexpr int kMaxDevices = 64;
std::atomic<int> g_ss_slots[kMaxDevices];

long long plane_pitch(long long K) { return (K + 31) / 32 * 32; }
size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Writes the planes of four consecutive k of one row (dst 16-byte aligned).
template <int PLANES>
__device__ __forceinline__ void put_planes(float *dst, long long pstride, const float (&v)[4])
{
    float h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) tc::split_value<PLANES == 2>(v[j], h[j], l[j]);
    *reinterpret_cast<float4 *>(dst) = make_float4(h[0], h[1], h[2], h[3]);
    if (PLANES == 2)
        *reinterpret_cast<float4 *>(dst + pstride) = make_float4(l[0], l[1], l[2], l[3]);
}

// One operand of the pass: R rows (M for A, N for B) of K values in E
// stored batch entries; K-inner sources are read row by row, others
// (stored K x R) through a shared-memory transpose.
struct PassOperand {
    const float *src;
    long long lds, sstride;  // source pitch and batch stride (elements)
    float *dst;
    long long pstride;       // elements per plane (E * R * ldp)
    int rows, E;
    int k_inner, vec;        // vec: 16-byte loads allowed
    long long tiles_r, tiles_k, tiles;  // 64 x 64 tiles per entry, and in all
};

// The pass over both operands in one launch: block b converts 64 x 64 tile
// b of A, then of B (tiles numbered entry-major, then row, then k).  256
// threads; thread t reads and writes four consecutive values at slot
// (it, t), it = 0..3: line (it / 2) * 32 + t / 8, values (it % 2) * 32 +
// 4 (t % 8) .. + 3 -- a warp touches four rows of 128 bytes per access.
// K-inner: line = row, values = k.  Transposed: lines are source rows (k)
// on the read and destination rows (r) on the write, through tile[r][k]
// with a 65-float pitch, which these slots access without bank conflicts.
// Values past K in a row's last group of four are written as zeros (the
// pitch leaves room; TMA never reads them).
template <int PLANES>
__global__ void __launch_bounds__(kThreads)
    planes_pass_kernel(PassOperand a, PassOperand b, int K, long long ldp)
{
    __shared__ float tile[kT][kT + 1];
    const int t = threadIdx.x;
    for (long long blk = blockIdx.x; blk < a.tiles + b.tiles; blk += gridDim.x) {
        const bool is_a = blk < a.tiles;
        const PassOperand &o = is_a ? a : b;
        const long long id = is_a ? blk : blk - a.tiles;
        const long long per_entry = o.tiles_r * o.tiles_k;
        const int q = static_cast<int>(id / per_entry);
        const long long rem = id - static_cast<long long>(q) * per_entry;
        const int r0 = static_cast<int>(rem / o.tiles_k) * kT;
        const int k0 = static_cast<int>(rem % o.tiles_k) * kT;
        const float *s = o.src + q * o.sstride;
        float *d = o.dst + static_cast<long long>(q) * o.rows * ldp;
        if (o.k_inner) {
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = r0 + (it >> 1) * 32 + (t >> 3);
                const int k = k0 + (it & 1) * 32 + 4 * (t & 7);
                if (r >= o.rows || k >= K) continue;
                const float *sp = s + static_cast<long long>(r) * o.lds + k;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (o.vec && k + 4 <= K) {
                    const float4 x = *reinterpret_cast<const float4 *>(sp);
                    v[0] = x.x;
                    v[1] = x.y;
                    v[2] = x.z;
                    v[3] = x.w;
                } else {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (k + jj < K) v[jj] = sp[jj];
                }
                put_planes<PLANES>(d + static_cast<long long>(r) * ldp + k, o.pstride, v);
            }
        } else {
            // read: source rows k0 + line, values r0 + ... (stored K x rows)
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int kl = (it >> 1) * 32 + (t >> 3), rl = (it & 1) * 32 + 4 * (t & 7);
                const int kk = k0 + kl, c = r0 + rl;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (kk < K) {
                    const float *sp = s + static_cast<long long>(kk) * o.lds + c;
                    if (o.vec && c + 3 < o.rows) {
                        const float4 x = *reinterpret_cast<const float4 *>(sp);
                        v[0] = x.x;
                        v[1] = x.y;
                        v[2] = x.z;
                        v[3] = x.w;
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            if (c + jj < o.rows) v[jj] = sp[jj];
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) tile[rl + jj][kl] = v[jj];
            }
            __syncthreads();
            // write: destination rows r0 + line, k0 + ...
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int rl = (it >> 1) * 32 + (t >> 3), kl = (it & 1) * 32 + 4 * (t & 7);
                const int r = r0 + rl, k = k0 + kl;
                if (r < o.rows && k < K) {
                    const float v[4] = {tile[rl][kl], tile[rl][kl + 1], tile[rl][kl + 2],
                                        tile[rl][kl + 3]};
                    put_planes<PLANES>(d + static_cast<long long>(r) * ldp + k, o.pstride, v);
                }
            }
            __syncthreads();
        }
    }
}

PassOperand pass_operand(const float *src, long long lds, long long sstride, int rows, int K,
                         int E, bool k_inner, float *dst, long long ldp)
{
    PassOperand o;
    o.src = src;
    o.lds = lds;
    o.sstride = sstride;
    o.dst = dst;
    o.pstride = static_cast<long long>(E) * rows * ldp;
    o.rows = rows;
    o.E = E;
    o.k_inner = k_inner ? 1 : 0;
    o.vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0 && lds % 4 == 0 &&
            (E <= 1 || sstride % 4 == 0);
    o.tiles_r = (rows + kT - 1) / kT;
    o.tiles_k = (K + kT - 1) / kT;
    o.tiles = static_cast<long long>(E) * o.tiles_r * o.tiles_k;
    return o;
}

template <int PLANES>
int launch_planes_pass(const PassOperand &a, const PassOperand &b, int K, long long ldp,
                       int num_sms, cudaStream_t stream)
{
    const long long total = a.tiles + b.tiles;
    if (total <= 0) return SGEMM_OK;
    // one tile per block; past 2^20 tiles the blocks step through the rest
    (void)num_sms;
    const long long cap = 1LL << 20;
    const unsigned grid = static_cast<unsigned>(total < cap ? total : cap);
    planes_pass_kernel<PLANES><<<grid, kThreads, 0, stream>>>(a, b, K, ldp);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

}  // namespace

int ss_slots(int num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return num_sms / 2;
    const int cached = g_ss_slots[dev].load();
    if (cached > 0) return cached;
    using KD = tcs::KindTF32<2>;
    auto kern = tcs::tcs_gemm_kernel<KD>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tcs::Shape<KD>::SMEM_BYTES) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)));
        cfg.blockDim = dim3(tcs::kThreads);
        cfg.dynamicSmemBytes = tcs::Shape<KD>::SMEM_BYTES;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    if (n <= 0 || n > num_sms / 2) n = num_sms / 2;
    if (n < 1) n = 1;
    g_ss_slots[dev].store(n);
    return n;
}

bool planes_pay(int mode, long long M, long long N, long long K, int QA, int QB, int Q,
                int num_sms)
{
    if ((mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32) || num_sms <= 0) return false;
    if (K > 0x7FFFFFFFLL) return false;
    const int planes = mode == SGEMM_MODE_3XTF32 ? 2 : 1;
    const int slots = tc_pair_slots(num_sms);
    const size_t any = ~static_cast<size_t>(0);
    int bm = 0, bn = 0;
    tc_tile_dims(mode, static_cast<int>(K), true, bm, bn);
    const long long pair_tiles = static_cast<long long>(Q) * ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
    const double t_pair =
        choose_plan(pair_tiles, static_cast<int>(K), slots, mode, bm, bn, kFeedPair, any).seconds;
    const long long ss_tiles =
        static_cast<long long>(Q) * ((M + tcs::PM - 1) / tcs::PM) * ((N + tcs::BN - 1) / tcs::BN);
    const double bytes = static_cast<double>(QA * M + QB * N) * K * 4.0 * (1 + planes);
    const double t_planes =
        bytes / 6.0e12 + 7e-6 +
        choose_plan(ss_tiles, static_cast<int>(K), slots, mode, tcs::PM, tcs::BN, kFeedPlanes, any)
            .seconds;
    return t_planes < t_pair;
}

int num_sms_or_zero()
{
    int num_sms = 0;
    unsigned int *status = nullptr;
    return current_sm103(&num_sms, &status) ? num_sms : 0;
}

size_t planes_bytes(int mode, long long M, long long N, long long K, int QA, int QB)
{
    const int planes = mode == SGEMM_MODE_3XTF32 ? 2 : 1;
    const long long ldp = plane_pitch(K);
    return round256(static_cast<size_t>(planes) * QA * M * ldp * sizeof(float)) +
           round256(static_cast<size_t>(planes) * QB * N * ldp * sizeof(float));
}

// The product on planes already written (A's at pa, B's at pb; QA / QB
// stored batch entries per plane): tensor maps, split plan (in plan.ws),
// launch.
static int product_on_planes(Plan &plan, const float *pa, const float *pb, int QA, int QB)
{
    GemmParams &p = plan.p;
    const int planes = plan.mode == SGEMM_MODE_3XTF32 ? 2 : 1;
    const long long ldp = plane_pitch(p.K);
    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    if (!encode_operand(&tmA, pa, true, p.M, p.K, ldp, planes * QA, p.M * ldp, tcs::BM) ||
        !encode_operand(&tmB, pb, true, p.N, p.K, ldp, planes * QB, p.N * ldp, tcs::HN))
        return SGEMM_ERR_UNSUPPORTED;

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
    const int rc = plan_splits(plan, tcs::PM, tcs::BN, kFeedPlanes, slots);
    if (rc != SGEMM_OK) return rc;
    // lo planes: the same maps, entries QA / QB further on
    return planes == 2 ? launch_ss<tcs::KindTF32<2>>(plan, tmA, tmB, tmA, tmB, QA, QB, slots)
                       : launch_ss<tcs::KindTF32<1>>(plan, tmA, tmB, tmA, tmB, 0, 0, slots);
}

int run_planes(Plan &plan, bool &taken, bool force)
{
    taken = false;
    GemmParams &p = plan.p;
    if (plan.mode != SGEMM_MODE_3XTF32 && plan.mode != SGEMM_MODE_TF32) return SGEMM_OK;
    if (plan.ws == nullptr) return SGEMM_OK;
    const int planes = plan.mode == SGEMM_MODE_3XTF32 ? 2 : 1;
    const int QA = (p.Q > 1 && p.sA != 0) ? p.Q : 1, QB = (p.Q > 1 && p.sB != 0) ? p.Q : 1;
    // plane * entries + entry indexes the tensor maps' third dimension (int)
    if (2LL * p.Q > 0x7FFFFFFFLL) return SGEMM_OK;
    const size_t need = planes_bytes(plan.mode, p.M, p.N, p.K, QA, QB);
    if (need > plan.ws_bytes ||
        (!force && !planes_pay(plan.mode, p.M, p.N, p.K, QA, QB, p.Q, plan.num_sms)))
        return SGEMM_OK;
    taken = true;

    const long long ldp = plane_pitch(p.K);
    char *w = static_cast<char *>(plan.ws);
    float *pa = reinterpret_cast<float *>(w);
    const size_t a_bytes = round256(static_cast<size_t>(planes) * QA * p.M * ldp * sizeof(float));
    float *pb = reinterpret_cast<float *>(w + a_bytes);
    // A: K-inner unless stored K x M; B: K-inner when stored N x K
    const PassOperand oa =
        pass_operand(p.A, p.lda, p.sA, p.M, p.K, QA, !plan.transA, pa, ldp);
    const PassOperand ob =
        pass_operand(p.B, p.ldb, p.sB, p.N, p.K, QB, plan.transB != 0, pb, ldp);
    int rc = planes == 2 ? launch_planes_pass<2>(oa, ob, p.K, ldp, plan.num_sms, plan.stream)
                         : launch_planes_pass<1>(oa, ob, p.K, ldp, plan.num_sms, plan.stream);
    if (rc != SGEMM_OK) return rc;

    plan.ws = need < plan.ws_bytes ? static_cast<void *>(w + need) : nullptr;
    plan.ws_bytes = need < plan.ws_bytes ? plan.ws_bytes - need : 0;
    return product_on_planes(plan, pa, pb, QA, QB);
}

}  // namespace sg
