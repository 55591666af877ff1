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
//
// Re-pitched copy: dst[r][c] = src[r][c] (src pitch lds, dst pitch ldd a
// multiple of 8).  A thread moves 8 values: one 16-byte store, loaded 16,
// 4 or 2 bytes at a time as the source rows' alignment allows (LW values per
// load).  Block (x, y, z) = (chunk of 2048 values, row, batch), y and z
// stepping by the grid.
template <int LW>
__global__ void __launch_bounds__(kThreads)
    copy16_kernel(const uint16_t *__restrict__ src, long long lds, long long sstride, int rows,
                  int cols, int Q, uint16_t *__restrict__ dst, long long ldd, long long dstride)
{
    const int c = (blockIdx.x * kThreads + threadIdx.x) * 8;
    if (c >= cols) return;
    for (int q = blockIdx.z; q < Q; q += gridDim.z) {
        for (long long r = blockIdx.y; r < rows; r += gridDim.y) {
            const uint16_t *sp = src + q * sstride + r * lds + c;
            uint16_t *dp = dst + q * dstride + r * ldd + c;
            if (c + 8 <= cols) {
                uint4 v;
                if (LW == 8) {
                    v = *reinterpret_cast<const uint4 *>(sp);
                } else if (LW == 2) {
                    const uint32_t *w = reinterpret_cast<const uint32_t *>(sp);
                    v = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        w[j] = static_cast<uint32_t>(sp[2 * j]) |
                               (static_cast<uint32_t>(sp[2 * j + 1]) << 16);
                    v = make_uint4(w[0], w[1], w[2], w[3]);
                }
                *reinterpret_cast<uint4 *>(dp) = v;
            } else {
                for (int j = 0; c + j < cols; ++j) dp[j] = sp[j];
            }
        }
    }
}

// Transposed copy: dst[r][c] = src[c][r] (src stored cols x rows, pitch
// lds), through a 64 x 64 shared tile; each thread reads two values of a
// source row (one 4-byte load when the source allows) and writes two of a
// destination row (one 4-byte store: ldd is even).
template <bool SRC4>
__global__ void __launch_bounds__(kThreads)
    transpose16_kernel(const uint16_t *__restrict__ src, long long lds, long long sstride,
                       int rows, int cols, int Q, uint16_t *__restrict__ dst, long long ldd,
                       long long dstride)
{
    __shared__ uint16_t tile[kT][kT + 2];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int c0 = blockIdx.x * kT;
    for (int q = blockIdx.z; q < Q; q += gridDim.z) {
        const uint16_t *s = src + q * sstride;
        uint16_t *d = dst + q * dstride;
        for (long long r0l = static_cast<long long>(blockIdx.y) * kT; r0l < rows;
             r0l += static_cast<long long>(gridDim.y) * kT) {
            const int r0 = static_cast<int>(r0l);
            // source rows c0 + i, values r0 + 2tx, r0 + 2tx + 1
#pragma unroll
            for (int i = ty; i < kT; i += 8) {
                const int c = c0 + i, r = r0 + 2 * tx;
                uint16_t v0 = 0, v1 = 0;
                if (c < cols) {
                    const uint16_t *sp = s + static_cast<long long>(c) * lds + r;
                    if (SRC4 && r + 1 < rows) {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(sp);
                        v0 = static_cast<uint16_t>(w & 0xFFFFu);
                        v1 = static_cast<uint16_t>(w >> 16);
                    } else {
                        if (r < rows) v0 = sp[0];
                        if (r + 1 < rows) v1 = sp[1];
                    }
                }
                tile[i][2 * tx] = v0;
                tile[i][2 * tx + 1] = v1;
            }
            __syncthreads();
            // destination rows r0 + i, values c0 + 2tx, c0 + 2tx + 1
#pragma unroll
            for (int i = ty; i < kT; i += 8) {
                const int r = r0 + i, c = c0 + 2 * tx;
                if (r < rows && c < cols) {
                    uint16_t *dp = d + static_cast<long long>(r) * ldd + c;
                    if (c + 1 < cols) {
                        *reinterpret_cast<uint32_t *>(dp) =
                            static_cast<uint32_t>(tile[2 * tx][i]) |
                            (static_cast<uint32_t>(tile[2 * tx + 1][i]) << 16);
                    } else {
                        dp[0] = tile[2 * tx][i];
                    }
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace

int launch_repack16(const uint16_t *src, long long lds, long long sstride, int rows, int cols,
                    int Q, bool trans, uint16_t *dst, long long ldd, long long dstride,
                    cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0 || Q <= 0) return SGEMM_OK;
    if (ldd % 8 != 0 || (Q > 1 && dstride % 8 != 0) || (reinterpret_cast<uintptr_t>(dst) & 15))
        return SGEMM_ERR_UNSUPPORTED;
    const unsigned gz = static_cast<unsigned>(Q < 65535 ? Q : 65535);
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
    const bool batch_even = Q <= 1 || sstride % 2 == 0;
    if (trans) {
        const long long tc = (cols + kT - 1) / kT, tr = (rows + kT - 1) / kT;
        if (tc > 0x7FFFFFFFLL) return SGEMM_ERR_UNSUPPORTED;
        const dim3 grid(static_cast<unsigned>(tc), static_cast<unsigned>(tr < 65535 ? tr : 65535),
                        gz);
        const bool src4 = (sa & 3) == 0 && lds % 2 == 0 && batch_even;
        if (src4)
            transpose16_kernel<true><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols,
                                                                   Q, dst, ldd, dstride);
        else
            transpose16_kernel<false><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows,
                                                                    cols, Q, dst, ldd, dstride);
    } else {
        const long long cb = (cols + 8LL * kThreads - 1) / (8LL * kThreads);
        const dim3 grid(static_cast<unsigned>(cb), static_cast<unsigned>(rows < 65535 ? rows : 65535),
                        gz);
        const bool w16 = (sa & 15) == 0 && lds % 8 == 0 && (Q <= 1 || sstride % 8 == 0);
        const bool w4 = (sa & 3) == 0 && lds % 2 == 0 && batch_even;
        if (w16)
            copy16_kernel<8><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q, dst,
                                                           ldd, dstride);
        else if (w4)
            copy16_kernel<2><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q, dst,
                                                           ldd, dstride);
        else
            copy16_kernel<1><<<grid, kThreads, 0, stream>>>(src, lds, sstride, rows, cols, Q, dst,
                                                           ldd, dstride);
    }
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
