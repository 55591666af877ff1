// noalloc.cu -- the split-K GEMM for callers that cannot allocate device
// memory.
//
// sgemm_batched_ex_ws needs a device workspace for its partial tiles.  Some
// callers cannot provide one: code that runs where cudaMalloc is not allowed
// or not wanted (inside a host callback or another library's critical
// section, under a memory pool that may not grow, in a plugin handed only
// the input and output pointers).  sgemm_batched_ex_noalloc gives them the
// same computation with the scratch taken from a fixed array that is part of
// the library image: every GPU that loads the library holds kScratchBytes
// of it until the process exits, and no call allocates or frees anything.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "internal.h"

namespace {

// Enough for the split-K workspace of this entry point's plan on a GPU with
// up to ~190 multiprocessors (at most one partial tile per multiprocessor,
// 256 x 128 fp32 at the largest).
constexpr size_t kScratchBytes = static_cast<size_t>(24) << 20;

// The scratch: shared by every call on a device; needs no initialisation.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device
bool g_scratch_ready[kMaxDevices];

// Device address of the scratch array on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in; the address a kernel may use is
// obtained once per device, with that device current.
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ready[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return SGEMM_ERR_LAUNCH;
        g_scratch_addr[dev] = p;
        g_scratch_ready[dev] = true;
    }
    *out = g_scratch_addr[dev];
    return SGEMM_OK;
}

}  // namespace

extern "C" int sgemm_batched_ex_noalloc(int mode, int M, int N, int K, float alpha,
                                        const float *A, int lda, const float *B, int ldb,
                                        float beta, float *C, int ldc, int transA, int transB,
                                        long long strideA, long long strideB, long long strideC,
                                        int Q, void *stream)
{
    // This entry point splits only grids of at most half as many tiles as
    // multiprocessors, into one wave of slices; its workspace must fit.
    const sg::SplitPlan sp = sg::one_wave_plan(mode, M, N, K, Q);
    if (sp.ws_bytes > kScratchBytes) return SGEMM_ERR_SCRATCH_LIMIT;
    void *ws = nullptr;
    if (sp.splits > 1) {
        const int rc = scratch_address(&ws);
        if (rc != SGEMM_OK) return rc;
    }
    // The workspace path runs the best plan that fits the bytes it is given
    // (this one, or one at least as good by its model); every slot it reads
    // back was written by the same call, so what an earlier call left in the
    // scratch does not matter.
    return sgemm_batched_ex_ws(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
                               strideA, strideB, strideC, Q, ws, ws ? sp.ws_bytes : 0, stream);
}
