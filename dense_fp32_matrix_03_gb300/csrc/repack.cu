// repack.cu -- operand transposition into the caller's workspace.
//
// The FP32 CUDA-core kernel is fastest with A M-inner (stored K x M) and B
// N-inner (stored K x N): a 128-bit shared load then gives four rows of A,
// or four columns of B, at one k.  With a workspace, a K-inner operand of a
// large enough product is first copied transposed (this kernel, bound by
// memory bandwidth) and the product runs in that layout.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "internal.h"

namespace sg {

namespace {

constexpr int kT = 32;       // tile edge
constexpr int kRowsPer = 8;  // thread rows per block (kT x kRowsPer threads)

// dst[q][c * ldd + r] = src[q][r * lds + c] for r < rows, c < cols.
// One kT x kT tile per block and step; blocks walk the tiles grid-stride.
__global__ void __launch_bounds__(kT * kRowsPer)
    transpose_kernel(const float *__restrict__ src, long long lds, long long sstride, int rows,
                     int cols, int Q, float *__restrict__ dst, long long ldd, long long dstride)
{
    __shared__ float tile[kT][kT + 1];
    const long long tiles_r = (rows + kT - 1) / kT, tiles_c = (cols + kT - 1) / kT;
    const long long total = tiles_r * tiles_c * Q;
    for (long long t = blockIdx.x; t < total; t += gridDim.x) {
        const long long q = t / (tiles_r * tiles_c);
        const long long rem = t - q * tiles_r * tiles_c;
        const int r0 = static_cast<int>(rem / tiles_c) * kT;
        const int c0 = static_cast<int>(rem % tiles_c) * kT;
        const float *s = src + q * sstride;
        float *d = dst + q * dstride;
        // read rows of src (coalesced along c)
#pragma unroll
        for (int i = threadIdx.y; i < kT; i += kRowsPer) {
            const int r = r0 + i, c = c0 + threadIdx.x;
            if (r < rows && c < cols) tile[i][threadIdx.x] = s[static_cast<long long>(r) * lds + c];
        }
        __syncthreads();
        // write rows of dst (coalesced along r)
#pragma unroll
        for (int i = threadIdx.y; i < kT; i += kRowsPer) {
            const int c = c0 + i, r = r0 + threadIdx.x;
            if (r < rows && c < cols) d[static_cast<long long>(c) * ldd + r] = tile[threadIdx.x][i];
        }
        __syncthreads();
    }
}

}  // namespace

int launch_transpose(const float *src, long long lds, long long sstride, int rows, int cols, int Q,
                     float *dst, long long ldd, long long dstride, int num_sms, cudaStream_t stream)
{
    const long long tiles =
        static_cast<long long>((rows + kT - 1) / kT) * ((cols + kT - 1) / kT) * Q;
    if (tiles <= 0) return SGEMM_OK;
    long long blocks = tiles;
    if (blocks > 16LL * num_sms) blocks = 16LL * num_sms;
    transpose_kernel<<<static_cast<unsigned>(blocks), dim3(kT, kRowsPer), 0, stream>>>(
        src, lds, sstride, rows, cols, Q, dst, ldd, dstride);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

}  // namespace sg
