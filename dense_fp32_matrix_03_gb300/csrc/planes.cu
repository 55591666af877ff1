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
// with both operands straight into the MMA's layout.  The pass reads each
// operand once and writes its planes once (HBM-bound).
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

// K-inner source (src[q][r * lds + k]): each thread converts four
// consecutive k of one row (a 16-byte load when VEC).  Block (x, y, z) =
// (chunk of 4 * kThreads values of K, row, entry), y and z stepping by the
// grid.  Values past K in the last group are written as zeros (the pitch
// leaves room; TMA never reads them).
template <int PLANES, bool VEC>
__global__ void __launch_bounds__(kThreads)
    planes_copy_kernel(const float *__restrict__ src, long long lds, long long sstride, int rows,
                       int K, int E, float *__restrict__ dst, long long ldp, long long pstride)
{
    const int k = (blockIdx.x * kThreads + threadIdx.x) * 4;
    if (k >= K) return;
    for (int q = blockIdx.z; q < E; q += gridDim.z) {
        for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
            const float *sp = src + q * sstride + r * lds + k;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            if (VEC && k + 4 <= K) {
                const float4 x = *reinterpret_cast<const float4 *>(sp);
                v[0] = x.x;
                v[1] = x.y;
                v[2] = x.z;
                v[3] = x.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (k + j < K) v[j] = sp[j];
            }
            put_planes<PLANES>(dst + (static_cast<long long>(q) * rows + r) * ldp + k, pstride, v);
        }
    }
}

// Source stored K x rows (src[q][k * lds + r]): through a 64 x 64 shared
// tile, each thread reading four consecutive values of a source row (a
// 16-byte load when VEC) and writing four consecutive k of a destination
// row.  Block (x, y, z) = (64 destination rows, 64 k, entry), y and z
// stepping by the grid.
template <int PLANES, bool VEC>
__global__ void __launch_bounds__(kThreads)
    planes_transpose_kernel(const float *__restrict__ src, long long lds, long long sstride,
                            int rows, int K, int E, float *__restrict__ dst, long long ldp,
                            long long pstride)
{
    __shared__ float tile[kT][kT + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16
    const int r0 = blockIdx.x * kT;
    for (int q = blockIdx.z; q < E; q += gridDim.z) {
        const float *s = src + q * sstride;
        float *d = dst + static_cast<long long>(q) * rows * ldp;
        for (long long k0l = static_cast<long long>(blockIdx.y) * kT; k0l < K;
             k0l += static_cast<long long>(gridDim.y) * kT) {
            const int k0 = static_cast<int>(k0l);
            // source rows k0 + ty + 16 i, columns r0 + 4 tx .. +3
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tk = ty + 16 * i, kk = k0 + tk, c = r0 + 4 * tx;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (kk < K) {
                    const float *sp = s + static_cast<long long>(kk) * lds + c;
                    if (VEC && c + 3 < rows) {
                        const float4 x = *reinterpret_cast<const float4 *>(sp);
                        v[0] = x.x;
                        v[1] = x.y;
                        v[2] = x.z;
                        v[3] = x.w;
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (c + j < rows) v[j] = sp[j];
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) tile[tk][4 * tx + j] = v[j];
            }
            __syncthreads();
            // destination rows r0 + ty + 16 i, k0 + 4 tx .. +3 (zeros past K)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tr = ty + 16 * i, r = r0 + tr, k = k0 + 4 * tx;
                if (r < rows && k < K) {
                    const float v[4] = {tile[4 * tx][tr], tile[4 * tx + 1][tr],
                                        tile[4 * tx + 2][tr], tile[4 * tx + 3][tr]};
                    put_planes<PLANES>(d + static_cast<long long>(r) * ldp + k, pstride, v);
                }
            }
            __syncthreads();
        }
    }
}

template <int PLANES>
int launch_planes_pass(const float *src, long long lds, long long sstride, int rows, int K, int E,
                       bool k_inner, float *dst, long long ldp, long long pstride,
                       cudaStream_t stream)
{
    const unsigned gz = static_cast<unsigned>(E < 65535 ? E : 65535);
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0 && lds % 4 == 0 &&
                     (E <= 1 || sstride % 4 == 0);
    if (k_inner) {
        const long long cb = (K + 4LL * kThreads - 1) / (4LL * kThreads);
        const dim3 grid(static_cast<unsigned>(cb), static_cast<unsigned>(rows < 65535 ? rows : 65535),
                        gz);
        if (vec)
            planes_copy_kernel<PLANES, true><<<grid, kThreads, 0, stream>>>(
                src, lds, sstride, rows, K, E, dst, ldp, pstride);
        else
            planes_copy_kernel<PLANES, false><<<grid, kThreads, 0, stream>>>(
                src, lds, sstride, rows, K, E, dst, ldp, pstride);
    } else {
        const long long tr = (rows + kT - 1) / kT, tk = (K + kT - 1) / kT;
        if (tr > 0x7FFFFFFFLL) return SGEMM_ERR_UNSUPPORTED;
        const dim3 grid(static_cast<unsigned>(tr), static_cast<unsigned>(tk < 65535 ? tk : 65535),
                        gz);
        if (vec)
            planes_transpose_kernel<PLANES, true><<<grid, kThreads, 0, stream>>>(
                src, lds, sstride, rows, K, E, dst, ldp, pstride);
        else
            planes_transpose_kernel<PLANES, false><<<grid, kThreads, 0, stream>>>(
                src, lds, sstride, rows, K, E, dst, ldp, pstride);
    }
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

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

}  // namespace

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
        bytes / 5.5e12 + 10e-6 +
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

int run_planes(Plan &plan, bool &taken)
{
    taken = false;
    GemmParams &p = plan.p;
    if (plan.mode != SGEMM_MODE_3XTF32 && plan.mode != SGEMM_MODE_TF32) return SGEMM_OK;
    if (plan.ws == nullptr) return SGEMM_OK;
    const int planes = plan.mode == SGEMM_MODE_3XTF32 ? 2 : 1;
    const int QA = (p.Q > 1 && p.sA != 0) ? p.Q : 1, QB = (p.Q > 1 && p.sB != 0) ? p.Q : 1;
    const size_t need = planes_bytes(plan.mode, p.M, p.N, p.K, QA, QB);
    if (need > plan.ws_bytes || !planes_pay(plan.mode, p.M, p.N, p.K, QA, QB, p.Q, plan.num_sms))
        return SGEMM_OK;
    taken = true;

    const long long ldp = plane_pitch(p.K);
    char *w = static_cast<char *>(plan.ws);
    float *pa = reinterpret_cast<float *>(w);
    const size_t a_bytes = round256(static_cast<size_t>(planes) * QA * p.M * ldp * sizeof(float));
    float *pb = reinterpret_cast<float *>(w + a_bytes);
    const long long a_pstride = static_cast<long long>(QA) * p.M * ldp;
    const long long b_pstride = static_cast<long long>(QB) * p.N * ldp;
    int rc;
    // A: K-inner unless stored K x M; B: K-inner when stored N x K
    if (planes == 2) {
        rc = launch_planes_pass<2>(p.A, p.lda, p.sA, p.M, p.K, QA, !plan.transA, pa, ldp,
                                   a_pstride, plan.stream);
        if (rc == SGEMM_OK)
            rc = launch_planes_pass<2>(p.B, p.ldb, p.sB, p.N, p.K, QB, plan.transB != 0, pb, ldp,
                                       b_pstride, plan.stream);
    } else {
        rc = launch_planes_pass<1>(p.A, p.lda, p.sA, p.M, p.K, QA, !plan.transA, pa, ldp,
                                   a_pstride, plan.stream);
        if (rc == SGEMM_OK)
            rc = launch_planes_pass<1>(p.B, p.ldb, p.sB, p.N, p.K, QB, plan.transB != 0, pb, ldp,
                                       b_pstride, plan.stream);
    }
    if (rc != SGEMM_OK) return rc;

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
    plan.ws = need < plan.ws_bytes ? static_cast<void *>(w + need) : nullptr;
    plan.ws_bytes = need < plan.ws_bytes ? plan.ws_bytes - need : 0;
    const int slots = ss_slots(plan.num_sms);
    rc = plan_splits(plan, tcs::PM, tcs::BN, kFeedPlanes, slots);
    if (rc != SGEMM_OK) return rc;
    return planes == 2 ? launch_ss<tcs::KindTF32<2>>(plan, tmA, tmB, slots)
                       : launch_ss<tcs::KindTF32<1>>(plan, tmA, tmB, slots);
}

}  // namespace sg
