// half.cu -- host side of the 16-bit-input path (bf16 / fp16 operands, fp32
// accumulation and output): argument checks, copies of operands the kernel
// cannot read directly, the split plan and the launch of the tc_ss.cuh kernel.
#include <atomic>
#include <cstring>

#include "../../include/sgemm.h"
#include "internal.h"
#include "tc_ss.cuh"

namespace sg {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kGroupM = 8;
std::atomic<int> g_half_slots[kMaxDevices];

long long round64(long long x) { return (x + 63) / 64 * 64; }
size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Whether the kernel can read an operand as it is: K-inner, 16-byte
// aligned, row pitch and batch stride multiples of 8 values (16 bytes).
// (Rows of whole 128-byte lines read a little faster -- bf16 A * B^T at
// 4092^3 on GB300: 1366 TFLOP/s with a 4096-value pitch, 1287 with 4128 --
// but not by enough to pay for a copy; copies get such rows for free.)
bool direct_layout(bool k_inner, long long ld, long long rows, long long K)
{
    (void)rows;
    (void)K;
    return k_inner && ld % 8 == 0;
}

bool direct(const void *p, bool k_inner, long long ld, long long rows, long long K, int Q,
            long long stride)
{
    return direct_layout(k_inner, ld, rows, K) && aligned16(p) &&
           (Q <= 1 || stride == 0 || stride % 8 == 0);
}

// Bytes of a K-inner copy of an operand with `rows` rows: round_up(K, 64)
// values per row (whole 128-byte lines), per batch entry (one entry when
// broadcast).
size_t copy_bytes(long long rows, long long K, int Q, bool broadcast)
{
    return round256(static_cast<size_t>(broadcast ? 1 : Q) * static_cast<size_t>(rows) *
                    static_cast<size_t>(round64(K)) * 2);
}

int half_slots(int num_sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return num_sms / 2;
    const int cached = g_half_slots[dev].load();
    if (cached > 0) return cached;
    using KD = tcs::KindHalf<true>;
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
    g_half_slots[dev].store(n);
    return n;
}

template <bool BF16>
int launch_half(Plan &plan, const CUtensorMap &tmA, const CUtensorMap &tmB, int slots)
{
    return launch_ss<tcs::KindHalf<BF16>>(plan, tmA, tmB, tmA, tmB, 0, 0, slots);
}

bool valid_type(int type) { return type == SGEMM_HALF_BF16 || type == SGEMM_HALF_FP16; }

}  // namespace

}  // namespace sg

using namespace sg;

extern "C" {

size_t sgemm_half_workspace_size(int type, int M, int N, int K, int transA, int transB, int lda,
                                 int ldb, int Q)
{
    if (!valid_type(type) || M <= 0 || N <= 0 || K <= 0 || Q <= 0) return 0;
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!current_sm103(&num_sms, &status)) return 0;
    size_t bytes = 0;
    if (!direct_layout(!transA, lda, M, K)) bytes += copy_bytes(M, K, Q, false);
    if (!direct_layout(transB != 0, ldb, N, K)) bytes += copy_bytes(N, K, Q, false);
    const long long tiles = static_cast<long long>(Q) * ((M + tcs::PM - 1) / tcs::PM) *
                            ((N + tcs::BN - 1) / tcs::BN);
    const SplitPlan sp = choose_plan(tiles, K, half_slots(num_sms), kModeHalf, tcs::PM, tcs::BN,
                                     kFeedPair, ~static_cast<size_t>(0));
    return bytes + sp.ws_bytes;
}

int sgemm_half_batched(int type, int M, int N, int K, float alpha, const void *A, int lda,
                       const void *B, int ldb, float beta, float *C, int ldc, int transA,
                       int transB, long long strideA, long long strideB, long long strideC, int Q,
                       void *workspace, size_t workspace_bytes, void *stream)
{
    if (!valid_type(type)) return SGEMM_ERR_INVALID_ARG;
    if (workspace_bytes > 0 &&
        (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return SGEMM_ERR_INVALID_ARG;
    int rc = check_shape(M, N, K, alpha, A, lda, B, ldb, C, ldc, transA, transB, strideA,
                         strideB, strideC, Q);
    if (rc != SGEMM_OK || M == 0 || N == 0 || Q == 0) return rc;
    if (K == 0 || alpha == 0.f)  // C = beta * C; A and B are not read
        return sgemm_batched_ex(SGEMM_MODE_3XTF32, M, N, 0, 0.f, nullptr, 1, nullptr, N, beta, C,
                                ldc, 0, 0, 0, 0, strideC, Q, stream);
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!current_sm103(&num_sms, &status)) return SGEMM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const long long sA = Q > 1 ? strideA : 0, sB = Q > 1 ? strideB : 0;
    const uint16_t *pa = static_cast<const uint16_t *>(A);
    const uint16_t *pb = static_cast<const uint16_t *>(B);
    long long la = lda, lb = ldb, xa = sA, xb = sB;
    char *w = static_cast<char *>(workspace);
    size_t used = 0;
    // operands the kernel cannot read as they are: a K-inner copy in the
    // workspace (transposed when M- or N-inner), rows padded to 64 values
    if (!direct(A, !transA, lda, M, K, Q, sA)) {
        const bool bc = Q > 1 && sA == 0;
        const size_t need = copy_bytes(M, K, Q, bc);
        if (used + need > workspace_bytes) return SGEMM_ERR_INVALID_ARG;
        uint16_t *dst = reinterpret_cast<uint16_t *>(w + used);
        const long long ld = round64(K);
        rc = launch_repack16(pa, lda, sA, M, K, bc ? 1 : Q, transA != 0, dst, ld,
                             static_cast<long long>(M) * ld, st);
        if (rc != SGEMM_OK) return rc;
        pa = dst;
        la = ld;
        xa = bc ? 0 : static_cast<long long>(M) * ld;
        used += need;
    }
    if (!direct(B, transB != 0, ldb, N, K, Q, sB)) {
        const bool bc = Q > 1 && sB == 0;
        const size_t need = copy_bytes(N, K, Q, bc);
        if (used + need > workspace_bytes) return SGEMM_ERR_INVALID_ARG;
        uint16_t *dst = reinterpret_cast<uint16_t *>(w + used);
        const long long ld = round64(K);
        rc = launch_repack16(pb, ldb, sB, N, K, bc ? 1 : Q, transB == 0, dst, ld,
                             static_cast<long long>(N) * ld, st);
        if (rc != SGEMM_OK) return rc;
        pb = dst;
        lb = ld;
        xb = bc ? 0 : static_cast<long long>(N) * ld;
        used += need;
    }

    Plan plan{};
    GemmParams &p = plan.p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Q = Q;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.lda = la;
    p.ldb = lb;
    p.ldc = ldc;
    p.sA = xa;
    p.sB = xb;
    p.sC = Q > 1 ? strideC : 0;
    p.a_q_step = (Q > 1 && xa != 0) ? 1 : 0;
    p.b_q_step = (Q > 1 && xb != 0) ? 1 : 0;
    p.c_vec4 = aligned16(C) && ldc % 4 == 0 && (p.sC % 4) == 0;
    p.status = status;
    p.wait_limit = kWaitLimitCycles;
    constexpr int SK = tcs::Shape<tcs::KindHalf<true>>::STAGE_K;
    p.k_blocks = (K + SK - 1) / SK;
    p.group_m = kGroupM;
    p.tiles_m = (M + tcs::PM - 1) / tcs::PM;
    p.tiles_n = (N + tcs::BN - 1) / tcs::BN;
    p.num_tiles = static_cast<long long>(Q) * p.tiles_m * p.tiles_n;
    plan.mode = kModeHalf;
    plan.num_sms = num_sms;
    plan.stream = st;
    plan.ws = used < workspace_bytes ? static_cast<void *>(w + used) : nullptr;
    plan.ws_bytes = used < workspace_bytes ? workspace_bytes - used : 0;

    alignas(64) CUtensorMap tmA;
    alignas(64) CUtensorMap tmB;
    std::memset(&tmA, 0, sizeof(tmA));
    std::memset(&tmB, 0, sizeof(tmB));
    const bool bf16 = type == SGEMM_HALF_BF16;
    if (!encode_operand16(&tmA, pa, bf16, M, K, la, Q, xa, tcs::BM) ||
        !encode_operand16(&tmB, pb, bf16, N, K, lb, Q, xb, tcs::HN))
        return SGEMM_ERR_UNSUPPORTED;
    const int slots = half_slots(num_sms);
    rc = plan_splits(plan, tcs::PM, tcs::BN, kFeedPair, slots);
    if (rc != SGEMM_OK) return rc;
    return bf16 ? launch_half<true>(plan, tmA, tmB, slots) : launch_half<false>(plan, tmA, tmB, slots);
}

}  // extern "C"
