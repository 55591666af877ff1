// peaks.cu -- throughput probes: kernels that run only the arithmetic
// instructions of a path, with no operand traffic, so that a GEMM kernel's
// speed can be set against what the same instructions reach on their own on
// the same GPU at the same moment (the peak a roofline fraction divides by).
//
//   FFMA      scalar fma.rn.f32 chains (the FP32 CUDA-core path's arithmetic)
//   FFMA2     packed fma.rn.f32x2 chains (the instruction that path issues)
//   TF32_SS   tcgen05.mma kind::tf32, M=128 N=256 K=8, both operands in
//             shared memory (the largest single-CTA shape)
//   TF32_TS   tcgen05.mma kind::tf32, M=128 N=128 K=8, A in tensor memory
//             (the instruction shape of the 3xTF32 / TF32 GEMM kernels)
//   BF16_SS   tcgen05.mma kind::f16 with bf16 operands, M=128 N=256 K=16
//             (comparable with a measured cuBLAS bf16 GEMM)
//
// The operands hold arbitrary finite values (a hash of their index): the
// results are discarded, but tensor-core power, and so the clock under a
// power cap, depends on the data, and zeros would flatter the figure.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "common.cuh"
#include "internal.h"
#include "tc_tf32.cuh"

namespace sg {

namespace {

// ------------------------------------------------------------------ FFMA

constexpr int kFfmaThreads = 512;
constexpr int kFfmaChains = 16;  // independent accumulators per thread
constexpr int kFfmaUnroll = 8;   // chain steps per loop trip
constexpr int kFfmaBlocksPerSm = 2;

// Each thread advances kFfmaChains independent chains acc = acc * x + y by
// kFfmaUnroll steps per trip (|x| < 1 keeps the values finite).  The sink
// store never happens for the x the host passes; it keeps the result live.
template <bool PACKED>
__global__ void __launch_bounds__(kFfmaThreads) ffma_probe_kernel(long long trips, float x, float y,
                                                                  float *sink)
{
    float acc[kFfmaChains];
#pragma unroll
    for (int c = 0; c < kFfmaChains; ++c) acc[c] = static_cast<float>(threadIdx.x + c) * 1e-3f;
    if (PACKED) {
        uint64_t v[kFfmaChains / 2], xx, yy;
#pragma unroll
        for (int c = 0; c < kFfmaChains / 2; ++c)
            asm("mov.b64 %0, {%1, %2};" : "=l"(v[c]) : "f"(acc[2 * c]), "f"(acc[2 * c + 1]));
        asm("mov.b64 %0, {%1, %1};" : "=l"(xx) : "f"(x));
        asm("mov.b64 %0, {%1, %1};" : "=l"(yy) : "f"(y));
        for (long long t = 0; t < trips; ++t) {
#pragma unroll
            for (int u = 0; u < kFfmaUnroll; ++u) {
#pragma unroll
                for (int c = 0; c < kFfmaChains / 2; ++c)
                    asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v[c]) : "l"(xx), "l"(yy));
            }
        }
#pragma unroll
        for (int c = 0; c < kFfmaChains / 2; ++c)
            asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2 * c]), "=f"(acc[2 * c + 1]) : "l"(v[c]));
    } else {
        for (long long t = 0; t < trips; ++t) {
#pragma unroll
            for (int u = 0; u < kFfmaUnroll; ++u) {
#pragma unroll
                for (int c = 0; c < kFfmaChains; ++c)
                    asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(acc[c]) : "f"(x), "f"(y));
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kFfmaChains; ++c) s += acc[c];
    if (x > 2.f && sink != nullptr) sink[threadIdx.x] = s;
}

// ------------------------------------------------------------ tensor core

constexpr int kTcThreads = 128;
constexpr int kTcSmemBytes = 120 * 1024;  // > half an SM's shared memory: one CTA per SM
constexpr int kTcA = 0;                   // A tile: 128 rows x 128 bytes
constexpr int kTcB = 128 * 128;           // B tile: 256 rows x 128 bytes
constexpr int kTcBar = kTcB + 256 * 128;

enum TcKind { kTf32SS = 0, kTf32TS = 1, kBf16SS = 2 };

template <int KIND>
struct TcShape {
    static constexpr int N = KIND == kTf32TS ? 128 : 256;
    static constexpr int K = KIND == kBf16SS ? 16 : 8;  // k per instruction
    // Instruction descriptor: f32 accumulate, both operands K-major.
    static constexpr uint32_t idesc = (1u << 4)
                                      | ((KIND == kBf16SS ? 1u : 2u) << 7)   // A format
                                      | ((KIND == kBf16SS ? 1u : 2u) << 10)  // B format
                                      | (static_cast<uint32_t>(N >> 3) << 17)
                                      | (static_cast<uint32_t>(128 >> 4) << 24);
};

__device__ __forceinline__ uint32_t mix32(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}

// A finite value in [-1, 1) from a hash: for bf16 operands, two bf16 halves.
__device__ __forceinline__ uint32_t probe_word(uint32_t i, bool bf16)
{
    const uint32_t h = mix32(i * 2654435761u + 12345u);
    const float f0 = static_cast<float>(h & 0xFFFFu) / 32768.f - 1.f;
    if (!bf16) return __float_as_uint(f0);
    const float f1 = static_cast<float>(h >> 16) / 32768.f - 1.f;
    return (__float_as_uint(f0) >> 16) | (__float_as_uint(f1) & 0xFFFF0000u);
}

__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate, bool f16)
{
    if (f16) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

// One CTA per multiprocessor.  Thread 0 issues `iters` MMAs back to back
// into one accumulator, walking the four 32-byte k steps of the 128-byte
// operand rows, as a GEMM's k loop does; then commits, and the CTA waits
// (bounded) for the tensor core to finish before it frees its TMEM.
template <int KIND>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_probe_kernel(long long iters, unsigned int *status, long long wait_limit)
{
    using S = TcShape<KIND>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *done = reinterpret_cast<uint64_t *>(smem + kTcBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTcBar + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kTcBar + 12);
    const int warp = threadIdx.x >> 5;

    uint32_t *words = reinterpret_cast<uint32_t *>(smem);
    for (int i = threadIdx.x; i < kTcBar / 4; i += kTcThreads)
        words[i] = probe_word(i + 977u * blockIdx.x, KIND == kBf16SS);
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, tc::kTmemCols);
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a_tmem = tmem + 256;  // TF32_TS: A in columns 256..287

    if (KIND == kTf32TS) {
        // Each warp writes its 32 lanes of the 32 A columns.
        float v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = __uint_as_float(probe_word(threadIdx.x * 32 + h * 16 + j, false));
            tc::tmem_st16(a_tmem + (static_cast<uint32_t>(warp * 32) << 16) + h * 16, v);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    }

    if (threadIdx.x == 0) {
        const uint64_t a0 = tc::kmajor_sw128_desc(smem_u32(smem + kTcA));
        const uint64_t b0 = tc::kmajor_sw128_desc(smem_u32(smem + kTcB));
        for (long long i = 0; i < iters; ++i) {
            const uint32_t kk = static_cast<uint32_t>(i & 3);
            const uint32_t acc = i > 0 ? 1u : 0u;
            if (KIND == kTf32TS)
                tc::umma_tf32_ts(tmem, a_tmem + kk * 8, b0 + kk * 2, S::idesc, acc);
            else
                umma_ss(tmem, a0 + kk * 2, b0 + kk * 2, S::idesc, acc, KIND == kBf16SS);
        }
        tc::umma_commit(done);
    }
    Abort ab{abort_flag, status, wait_limit};
    mbar_wait(done, 0, ab, kStatusWaitMma, threadIdx.x != 0);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, tc::kTmemCols);
}

// Bounds that keep one probe launch well under a second (and under the
// bounded wait) on any GPU of this class.
constexpr long long kMaxFfmaTrips = 1LL << 16;
constexpr long long kMaxTcIters = 1LL << 22;

template <int KIND>
int launch_tc_probe(long long iters, int num_sms, unsigned int *status, cudaStream_t st,
                    double *flops)
{
    using S = TcShape<KIND>;
    auto kern = tc_probe_kernel<KIND>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcSmemBytes + 1024) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    kern<<<num_sms, kTcThreads, kTcSmemBytes + 1024, st>>>(iters, status, 1LL << 31);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    *flops = 2.0 * 128 * S::N * S::K * static_cast<double>(iters) * num_sms;
    return SGEMM_OK;
}

}  // namespace

bool probe_args_ok(int kind, long long iters)
{
    if (iters < 1) return false;
    switch (kind) {
    case SGEMM_PROBE_FFMA:
    case SGEMM_PROBE_FFMA2: return iters <= kMaxFfmaTrips;
    case SGEMM_PROBE_TF32_SS:
    case SGEMM_PROBE_TF32_TS:
    case SGEMM_PROBE_BF16_SS: return iters <= kMaxTcIters;
    default: return false;
    }
}

int launch_peak_probe(int kind, long long iters, int num_sms, unsigned int *status,
                      cudaStream_t st, double *flops)
{
    if (!probe_args_ok(kind, iters)) return SGEMM_ERR_INVALID_ARG;
    switch (kind) {
    case SGEMM_PROBE_FFMA:
    case SGEMM_PROBE_FFMA2: {
        const int blocks = num_sms * kFfmaBlocksPerSm;
        // x < 2: the sink is never written.
        if (kind == SGEMM_PROBE_FFMA)
            ffma_probe_kernel<false><<<blocks, kFfmaThreads, 0, st>>>(iters, 0.999f, 1e-3f,
                                                                      nullptr);
        else
            ffma_probe_kernel<true><<<blocks, kFfmaThreads, 0, st>>>(iters, 0.999f, 1e-3f,
                                                                     nullptr);
        if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
        note_launch();
        *flops = 2.0 * kFfmaChains * kFfmaUnroll * static_cast<double>(iters) * blocks *
                 kFfmaThreads;
        return SGEMM_OK;
    }
    case SGEMM_PROBE_TF32_SS:
        return launch_tc_probe<kTf32SS>(iters, num_sms, status, st, flops);
    case SGEMM_PROBE_TF32_TS:
        return launch_tc_probe<kTf32TS>(iters, num_sms, status, st, flops);
    case SGEMM_PROBE_BF16_SS:
        return launch_tc_probe<kBf16SS>(iters, num_sms, status, st, flops);
    default:
        return SGEMM_ERR_INVALID_ARG;
    }
}

}  // namespace sg
