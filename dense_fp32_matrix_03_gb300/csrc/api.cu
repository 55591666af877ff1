// api.cu -- the C ABI (include/sgemm.h): argument checks, the per-call plan,
// TMA tensor-map encoding, the device status word, and dispatch to the SIMT
// or tcgen05 launchers.  Nothing here allocates device memory.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "common.cuh"
#include "internal.h"

namespace sg {

// Device status word: set by kernels whose bounded waits run out.
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;
// A wait may spin for this many SM clock cycles (about a second at the
// GB300's clocks) before the kernel gives up and reports SGEMM_ERR_TIMEOUT.
constexpr long long kWaitLimitCycles = 1LL << 31;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned int *status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
std::atomic<int> g_default_mode{SGEMM_MODE_FP32};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device facts, queried once with the device current.
const DeviceInfo *device_info(int *dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    *dev_out = dev;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return nullptr;
        d.status = static_cast<unsigned int *>(addr);
        d.ready = true;
    }
    return &d;
}

bool get_encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scales C by beta (or zeroes it when beta == 0): the whole result when
// alpha == 0 or K == 0.  One thread per element, grid-stride.
__global__ void scale_c_kernel(float *C, int M, int N, long long ldc, long long sC, int Q,
                               float beta)
{
    const long long total = static_cast<long long>(Q) * M * N;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long q = e / (static_cast<long long>(M) * N);
        const long long r = e - q * M * N;
        const long long i = r / N, j = r - i * N;
        float *c = C + q * sC + i * ldc + j;
        *c = (beta == 0.f) ? 0.f : beta * *c;
    }
}

// Bounded-wait self test: one thread waits on an mbarrier that nobody arrives
// on, gives up after `limit` cycles, then completes the phase itself so the
// barrier is left in a clean state.
__global__ void wait_timeout_kernel(unsigned int *status, long long limit)
{
    __shared__ uint64_t bar;
    __shared__ int flag;
    mbar_init(&bar, 1);
    flag = 0;
    fence_mbar_init();
    const Abort ab{&flag, status, limit};
    mbar_wait(&bar, 0, ab, kStatusWaitTest);
    mbar_arrive(&bar);
}

int check_args(int mode, int M, int N, int K, float alpha, const float *A, int lda,
               const float *B, int ldb, float beta, float *C, int ldc, int transA, int transB,
               long long sA, long long sB, long long sC, int Q)
{
    (void)beta;
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32)
        return SGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || Q < 0) return SGEMM_ERR_INVALID_ARG;
    if (sA < 0 || sB < 0 || sC < 0) return SGEMM_ERR_INVALID_ARG;
    const long long a_row = transA ? M : K, b_row = transB ? K : N;
    if (lda < (a_row > 1 ? a_row : 1) || ldb < (b_row > 1 ? b_row : 1) || ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || Q == 0) return SGEMM_OK;
    if (C == nullptr) return SGEMM_ERR_INVALID_ARG;
    if (Q > 1 && sC < static_cast<long long>(M - 1) * ldc + N) return SGEMM_ERR_INVALID_ARG;
    const bool reads_ab = (K > 0 && alpha != 0.f);
    if (reads_ab && (A == nullptr || B == nullptr)) return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

}  // namespace

bool encode_operand(CUtensorMap *map, const float *base, bool kin, long long rows, long long K,
                    long long ld, int Q, long long stride, int box_rows)
{
    if (!get_encoder()) return false;
    const bool batched = Q > 1 && stride != 0;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    if (kin) {
        dims[0] = static_cast<cuuint64_t>(K);
        dims[1] = static_cast<cuuint64_t>(rows);
        box[0] = 32;
        box[1] = static_cast<cuuint32_t>(box_rows);
    } else {
        dims[0] = static_cast<cuuint64_t>(rows);
        dims[1] = static_cast<cuuint64_t>(K);
        box[0] = static_cast<cuuint32_t>(box_rows);
        box[1] = 32;
    }
    dims[2] = batched ? static_cast<cuuint64_t>(Q) : 1;
    box[2] = 1;
    strides[0] = static_cast<cuuint64_t>(ld) * 4;
    strides[1] = batched ? static_cast<cuuint64_t>(stride) * 4 : strides[0] * dims[1];
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                kin ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int min_slice_k(int mode) { return mode == SGEMM_MODE_FP32 ? 64 : 256; }

int choose_splits(long long num_tiles, int K, int num_sms, int mode)
{
    // as many slices as keep every unit in one wave (units <= multiprocessors)
    if (num_tiles <= 0 || 2 * num_tiles > num_sms) return 1;
    long long s = num_sms / num_tiles;
    const long long by_k = K / min_slice_k(mode);
    if (s > by_k) s = by_k;
    if (s > kMaxSplits) s = kMaxSplits;
    return s < 2 ? 1 : static_cast<int>(s);
}

size_t splitk_workspace_bytes(long long num_tiles, int splits)
{
    if (splits <= 1) return 0;
    const size_t ctr = (static_cast<size_t>(num_tiles) * kSplitRegions * sizeof(unsigned int) + 255) &
                       ~static_cast<size_t>(255);
    return ctr + static_cast<size_t>(num_tiles) * splits * kSplitTile * kSplitTile * sizeof(float);
}

int plan_splits(Plan &plan)
{
    GemmParams &p = plan.p;
    p.splits = 1;
    p.ws_part = nullptr;
    p.ws_ctr = nullptr;
    const int s = plan.ws ? choose_splits(p.num_tiles, p.K, plan.num_sms, plan.mode) : 1;
    const size_t need = splitk_workspace_bytes(p.num_tiles, s);
    if (s > 1 && need <= plan.ws_bytes) {
        const size_t ctr = (static_cast<size_t>(p.num_tiles) * kSplitRegions * sizeof(unsigned int) +
                            255) & ~static_cast<size_t>(255);
        p.splits = s;
        p.ws_ctr = static_cast<unsigned int *>(plan.ws);
        p.ws_part = reinterpret_cast<float *>(static_cast<char *>(plan.ws) + ctr);
        // counters start at zero (the last slice of every region re-arms its
        // counter, but a call that stopped early may have left one raised)
        if (cudaMemsetAsync(plan.ws, 0, ctr, plan.stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    }
    p.num_units = p.num_tiles * p.splits;
    return SGEMM_OK;
}

}  // namespace sg

using namespace sg;

namespace {

// TMA can describe an operand when its base is 16-byte aligned and its row
// pitch and batch stride are multiples of 16 bytes.
bool tma_eligible(const float *p, long long ld, int Q, long long stride)
{
    if (!aligned16(p) || (ld % 4) != 0) return false;
    if (Q > 1 && stride != 0 && (stride % 4) != 0) return false;
    return true;
}

int run(int mode, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
        int ldb, float beta, float *C, int ldc, int transA, int transB, long long sA,
        long long sB, long long sC, int Q, void *stream, void *ws = nullptr,
        size_t ws_bytes = 0)
{
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    int rc = check_args(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, sA,
                        sB, sC, Q);
    if (rc != SGEMM_OK || M == 0 || N == 0 || Q == 0) return rc;

    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return SGEMM_ERR_UNSUPPORTED;
    if (di->cc_major != 10 || di->cc_minor != 3) return SGEMM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (K == 0 || alpha == 0.f) {
        const long long total = static_cast<long long>(Q) * M * N;
        long long blocks = (total + 255) / 256;
        if (blocks > 8LL * di->num_sms) blocks = 8LL * di->num_sms;
        scale_c_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(C, M, N, ldc, sC, Q, beta);
        return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }

    Plan plan{};
    GemmParams &p = plan.p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.Q = Q;
    p.alpha = alpha;
    p.beta = beta;
    p.A = A;
    p.B = B;
    p.C = C;
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.sA = Q > 1 ? sA : 0;
    p.sB = Q > 1 ? sB : 0;
    p.sC = Q > 1 ? sC : 0;
    p.a_q_step = (Q > 1 && sA != 0) ? 1 : 0;
    p.b_q_step = (Q > 1 && sB != 0) ? 1 : 0;
    p.a_vec4 = aligned16(A) && lda % 4 == 0 && (p.sA % 4) == 0;
    p.b_vec4 = aligned16(B) && ldb % 4 == 0 && (p.sB % 4) == 0;
    p.c_vec4 = aligned16(C) && ldc % 4 == 0 && (p.sC % 4) == 0;
    p.status = di->status;
    p.wait_limit = kWaitLimitCycles;
    plan.transA = transA != 0;
    plan.transB = transB != 0;
    plan.mode = mode;
    plan.a_tma = tma_eligible(A, lda, Q, p.sA);
    plan.b_tma = tma_eligible(B, ldb, Q, p.sB);
    plan.num_sms = di->num_sms;
    plan.device = dev;
    plan.stream = st;
    plan.ws = ws;
    plan.ws_bytes = ws_bytes;

    if (mode == SGEMM_MODE_FP32) return launch_simt(plan);
    return launch_tc(plan);
}

}  // namespace

extern "C" {

int sgemm(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
          float beta, float *C, int ldc, void *stream)
{
    return run(SGEMM_MODE_DEFAULT, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, 0, 0, 0, 0, 0,
               1, stream);
}

int sgemm_batched(int M, int N, int K, float alpha, const float *A, int lda, const float *B,
                  int ldb, float beta, float *C, int ldc, int transA, int transB,
                  long long strideA, long long strideB, long long strideC, int Q, void *stream)
{
    return run(SGEMM_MODE_DEFAULT, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
               strideA, strideB, strideC, Q, stream);
}

int sgemm_batched_ex(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                     const float *B, int ldb, float beta, float *C, int ldc, int transA,
                     int transB, long long strideA, long long strideB, long long strideC, int Q,
                     void *stream)
{
    return run(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, strideA,
               strideB, strideC, Q, stream);
}

int sgemm_batched_ex_ws(int mode, int M, int N, int K, float alpha, const float *A, int lda,
                        const float *B, int ldb, float beta, float *C, int ldc, int transA,
                        int transB, long long strideA, long long strideB, long long strideC,
                        int Q, void *workspace, size_t workspace_bytes, void *stream)
{
    if (workspace_bytes > 0 &&
        (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return SGEMM_ERR_INVALID_ARG;
    return run(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, strideA,
               strideB, strideC, Q, stream, workspace_bytes ? workspace : nullptr,
               workspace_bytes);
}

size_t sgemm_workspace_size(int mode, int M, int N, int K, int Q)
{
    if (mode == SGEMM_MODE_DEFAULT) mode = g_default_mode.load();
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32) return 0;
    if (M <= 0 || N <= 0 || K <= 0 || Q <= 0) return 0;
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return 0;
    const long long tiles = static_cast<long long>(Q) * ((M + kSplitTile - 1) / kSplitTile) *
                            ((N + kSplitTile - 1) / kSplitTile);
    return splitk_workspace_bytes(tiles, choose_splits(tiles, K, di->num_sms, mode));
}

int sgemm_set_default_mode(int mode)
{
    if (mode != SGEMM_MODE_FP32 && mode != SGEMM_MODE_3XTF32 && mode != SGEMM_MODE_TF32)
        return SGEMM_ERR_INVALID_ARG;
    g_default_mode.store(mode);
    return SGEMM_OK;
}

int sgemm_get_default_mode(void) { return g_default_mode.load(); }

const char *sgemm_status_string(int status)
{
    switch (status) {
    case SGEMM_OK: return "success";
    case SGEMM_ERR_INVALID_ARG: return "invalid argument";
    case SGEMM_ERR_UNSUPPORTED: return "unsupported: needs a compute capability 10.3 GPU";
    case SGEMM_ERR_LAUNCH: return "CUDA launch or runtime error";
    case SGEMM_ERR_TIMEOUT: return "a kernel's bounded wait ran out (device status word)";
    case SGEMM_ERR_SCRATCH_LIMIT:
        return "the shape needs more split-K scratch than the built-in array holds";
    default: return "unknown status";
    }
}

int sgemm_poll_error(void *stream)
{
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return SGEMM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        return SGEMM_ERR_TIMEOUT;
    }
    return SGEMM_OK;
}

int sgemm_selftest_wait_timeout(long long wait_cycles, void *stream)
{
    if (wait_cycles < 1 || wait_cycles > (1LL << 31)) return SGEMM_ERR_INVALID_ARG;
    int dev = 0;
    const DeviceInfo *di = device_info(&dev);
    if (di == nullptr) return SGEMM_ERR_UNSUPPORTED;
    wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(di->status,
                                                                          wait_cycles);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

int sgemm_version(void) { return 100; }

}  // extern "C"
