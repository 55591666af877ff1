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
// Block (x, y, z) moves tile (column block x, row block y, batch z); y and z
// step by the grid size when there are more tiles than the grid holds.
__global__ void __launch_bounds__(kT * kRowsPer)
    transpose_kernel(const float *__restrict__ src, long long lds, long long sstride, int rows,
                     int cols, int Q, float *__restrict__ dst, long long ldd, long long dstride)
{
    __shared__ float tile[kT][kT + 1];
    const int c0 = blockIdx.x * kT;
    for (int q = blockIdx.z; q < Q; q += gridDim.z) {
        const float *s = src + q * sstride;
        float *d = dst + q * dstride;
        for (long long r0l = static_cast<long long>(blockIdx.y) * kT; r0l < rows;
             r0l += static_cast<long long>(gridDim.y) * kT) {
            const int r0 = static_cast<int>(r0l);
            // read rows of src (coalesced along c)
#pragma unroll
            for (int i = threadIdx.y; i < kT; i += kRowsPer) {
                const int r = r0 + i, c = c0 + threadIdx.x;
                if (r < rows && c < cols)
                    tile[i][threadIdx.x] = s[static_cast<long long>(r) * lds + c];
            }
            __syncthreads();
            // write rows of dst (coalesced along r)
#pragma unroll
            for (int i = threadIdx.y; i < kT; i += kRowsPer) {
                const int c = c0 + i, r = r0 + threadIdx.x;
                if (r < rows && c < cols)
                    d[static_cast<long long>(c) * ldd + r] = tile[threadIdx.x][i];
            }
            __syncthreads();
        }
    }
}

}  // namespace

int launch_transpose(const float *src, long long lds, long long sstride, int rows, int cols, int Q,
                     float *dst, long long ldd, long long dstride, int, cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0 || Q <= 0) return SGEMM_OK;
    const long long tc = (cols + kT - 1) / kT, tr = (rows + kT - 1) / kT;
    if (tc > 0x7FFFFFFFLL) return SGEMM_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(tc), static_cast<unsigned>(tr < 65535 ? tr : 65535),
                    static_cast<unsigned>(Q < 65535 ? Q : 65535));
    transpose_kernel<<<grid, dim3(kT, kRowsPer), 0, stream>>>(src, lds, sstride, rows, cols, Q,
                                                               dst, ldd, dstride);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

}  // namespace sg
