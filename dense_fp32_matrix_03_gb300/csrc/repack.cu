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

constexpr int kT = 64;        // tile edge
constexpr int kThreads = 256;  // 16 threads per 64-float row segment

// dst[q][c * ldd + r] = src[q][r * lds + c] for r < rows, c < cols.
// Block (x, y, z) moves tile (column block x, row block y, batch z); y and z
// step by the grid size when there are more tiles than the grid holds.
// Each thread reads four 4-float pieces of source rows (16-byte loads when
// VEC: source rows and pieces 16-byte aligned) and writes four 4-float
// pieces of destination rows (16-byte stores when the destination allows),
// so a block keeps 16 KB in flight each way.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    transpose_kernel(const float *__restrict__ src, long long lds, long long sstride, int rows,
                     int cols, int Q, float *__restrict__ dst, long long ldd, long long dstride,
                     bool dvec)
{
    __shared__ float tile[kT][kT + 1];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16
    const int c0 = blockIdx.x * kT;
    for (int q = blockIdx.z; q < Q; q += gridDim.z) {
        const float *s = src + q * sstride;
        float *d = dst + q * dstride;
        for (long long r0l = static_cast<long long>(blockIdx.y) * kT; r0l < rows;
             r0l += static_cast<long long>(gridDim.y) * kT) {
            const int r0 = static_cast<int>(r0l);
            // rows r0 + ty + 16*i, columns c0 + 4*tx .. +3
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tr = ty + 16 * i, r = r0 + tr, c = c0 + 4 * tx;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (r < rows) {
                    const float *sp = s + static_cast<long long>(r) * lds + c;
                    if (VEC && c + 3 < cols) {
                        const float4 x = *reinterpret_cast<const float4 *>(sp);
                        v[0] = x.x;
                        v[1] = x.y;
                        v[2] = x.z;
                        v[3] = x.w;
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (c + j < cols) v[j] = sp[j];
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) tile[tr][4 * tx + j] = v[j];
            }
            __syncthreads();
            // destination rows c0 + ty + 16*i, columns r0 + 4*tx .. +3
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tc = ty + 16 * i, c = c0 + tc, r = r0 + 4 * tx;
                if (c < cols && r < rows) {
                    float *dp = d + static_cast<long long>(c) * ldd + r;
                    if (dvec && r + 3 < rows) {
                        *reinterpret_cast<float4 *>(dp) =
                            make_float4(tile[4 * tx][tc], tile[4 * tx + 1][tc], tile[4 * tx + 2][tc],
                                        tile[4 * tx + 3][tc]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (r + j < rows) dp[j] = tile[4 * tx + j][tc];
                    }
                }
            }
            __syncthreads();
        }
    }
}

// 16-bit values (bf16 / fp16 operands of the half path), moved as raw bits.
// TRANS: dst[r][c] = src[c][r] for r < rows, c < cols (src stored cols x
// rows, pitch lds), through a 64 x 65 shared tile; else dst[r][c] = src[r][c]
// (pitch lds).  Block (x, y, z) = (column block, row block, batch), y and z
// stepping by the grid when there are more blocks.
template <bool TRANS>
__global__ void __launch_bounds__(kThreads)
    repack16_kernel(const uint16_t *__restrict__ src, long long lds, long long sstride, int rows,
                    int cols, int Q, uint16_t *__restrict__ dst, long long ldd, long long dstride)
{
    __shared__ uint16_t tile[kT][kT + 1];
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;  // 64 x 4
    const int c0 = blockIdx.x * kT;
    for (int q = blockIdx.z; q < Q; q += gridDim.z) {
        const uint16_t *s = src + q * sstride;
        uint16_t *d = dst + q * dstride;
        for (long long r0l = static_cast<long long>(blockIdx.y) * kT; r0l < rows;
             r0l += static_cast<long long>(gridDim.y) * kT) {
            const int r0 = static_cast<int>(r0l);
            if (TRANS) {
                // source rows are destination columns c0 .. c0+63, read along r
                for (int i = ty; i < kT; i += 4) {
                    const int c = c0 + i, r = r0 + tx;
                    tile[i][tx] = (c < cols && r < rows)
                                      ? s[static_cast<long long>(c) * lds + r]
                                      : static_cast<uint16_t>(0);
                }
                __syncthreads();
                for (int i = ty; i < kT; i += 4) {
                    const int r = r0 + i, c = c0 + tx;
                    if (r < rows && c < cols) d[static_cast<long long>(r) * ldd + c] = tile[tx][i];
                }
                __syncthreads();
            } else {
                for (int i = ty; i < kT; i += 4) {
                    const int r = r0 + i, c = c0 + tx;
                    if (r < rows && c < cols)
                        d[static_cast<long long>(r) * ldd + c] =
                            s[static_cast<long long>(r) * lds + c];
                }
            }
        }
    }
}

}  // namespace

int launch_repack16(const uint16_t *src, long long lds, long long sstride, int rows, int cols,
                    int Q, bool trans, uint16_t *dst, long long ldd, long long dstride,
                    cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0 || Q <= 0) return SGEMM_OK;
    const long long tc = (cols + kT - 1) / kT, tr = (rows + kT - 1) / kT;
    if (tc > 0x7FFFFFFFLL) return SGEMM_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(tc), static_cast<unsigned>(tr < 65535 ? tr : 65535),
                    static_cast<unsigned>(Q < 65535 ? Q : 65535));
    if (trans)
        repack16_kernel<true><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q, dst,
                                                            ldd, dstride);
    else
        repack16_kernel<false><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q,
                                                             dst, ldd, dstride);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

int launch_transpose(const float *src, long long lds, long long sstride, int rows, int cols, int Q,
                     float *dst, long long ldd, long long dstride, int, cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0 || Q <= 0) return SGEMM_OK;
    const long long tc = (cols + kT - 1) / kT, tr = (rows + kT - 1) / kT;
    if (tc > 0x7FFFFFFFLL) return SGEMM_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(tc), static_cast<unsigned>(tr < 65535 ? tr : 65535),
                    static_cast<unsigned>(Q < 65535 ? Q : 65535));
    const bool svec = (reinterpret_cast<uintptr_t>(src) & 15) == 0 && lds % 4 == 0 &&
                      (Q <= 1 || sstride % 4 == 0);
    const bool dvec = (reinterpret_cast<uintptr_t>(dst) & 15) == 0 && ldd % 4 == 0 &&
                      (Q <= 1 || dstride % 4 == 0);
    if (svec)
        transpose_kernel<true><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q,
                                                              dst, ldd, dstride, dvec);
    else
        transpose_kernel<false><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q,
                                                               dst, ldd, dstride, dvec);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

}  // namespace sg
