// host.cu -- the product on host buffers.  The operands are copied into a
// device buffer the caller provides, the product is computed there, and C
// is copied back.  C is cut into panels of rows and, for large K, K into two
// slices: the copy-in of one (slice, panel), the product of the previous one
// and the copy-out of a finished panel run at the same time on three streams
// (the caller's, for the products, and two of the library's own, one per
// copy direction), ordered by events.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "internal.h"

namespace sg {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPanels = 64;
// K from which the call cuts the product in two K slices (below it, half of
// op(B) arrives too soon for the overlap to pay for a second pass over C).
constexpr int kKSplitMin = 1024;

// Copy streams of a device, made on first use and kept for the process.
struct CopyStreams {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
};
std::mutex g_copy_mu;
CopyStreams g_copy[kMaxDevices];

bool copy_streams(cudaStream_t *in, cudaStream_t *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_copy_mu);
    CopyStreams &c = g_copy[dev];
    if (!c.ready) {
        if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(c.in);
            return false;
        }
        c.ready = true;
    }
    *in = c.in;
    *out = c.out;
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
long long round4(long long x) { return x < 4 ? 4 : (x + 3) & ~3LL; }

// Where everything sits in the caller's device buffer.  Each operand is
// stored with its rows padded to a multiple of four floats, so that the
// kernels' TMA feeds can describe it whatever the host pitch.
struct Layout {
    long long ldA, ldB, ldC;       // device row pitches (elements)
    size_t offA, offB, offC, offW; // byte offsets into the buffer
    size_t ws_bytes, total;
    int panel, panels;             // rows of C per panel, panel count
};

// Rows per panel when the caller leaves it to the library: enough output
// tiles for about one wave of the GPU per panel (measured on GB300 at
// 4092^3: one to two waves per panel beat both fewer, larger panels, whose
// first copy-in and last copy-out overlap nothing, and smaller ones, which
// leave multiprocessors idle in every product), at most kMaxPanels.
int auto_panel_rows(int mode, int M, int N, int K, int num_sms)
{
    int bm = 0, bn = 0, slots = num_sms;
    if (mode == SGEMM_MODE_FP32) {
        simt_tile_dims(false, bm, bn);
    } else {
        tc_tile_dims(mode, K, true, bm, bn);
        slots = tc_pair_slots(num_sms);
    }
    const long long tiles_n = (N + bn - 1) / bn;
    long long rows_tiles = (static_cast<long long>(slots) + tiles_n - 1) / tiles_n;
    if (rows_tiles < 1) rows_tiles = 1;
    long long rows = rows_tiles * bm;
    const long long min_rows = (M + kMaxPanels - 1) / kMaxPanels;
    if (rows < min_rows) rows = min_rows;
    return rows >= M ? M : static_cast<int>(rows);
}

int resolve_mode(int mode)
{
    return mode == SGEMM_MODE_DEFAULT ? sgemm_get_default_mode() : mode;
}

bool make_layout(int mode, int M, int N, int K, int transA, int transB, int panel_rows,
                 int num_sms, Layout *L)
{
    L->ldA = transA ? round4(M) : round4(K);
    L->ldB = transB ? round4(K) : round4(N);
    L->ldC = round4(N);
    const long long rowsA = transA ? K : M, rowsB = transB ? N : K;
    L->panel = panel_rows > 0 ? (panel_rows < M ? panel_rows : M)
                              : auto_panel_rows(mode, M, N, K, num_sms);
    if (L->panel < 1) L->panel = 1;
    L->panels = static_cast<int>((M + L->panel - 1) / L->panel);
    if (L->panels > kMaxPanels) return false;
    const int last = M - (L->panels - 1) * L->panel;
    size_t w1 = workspace_size_no_planes(mode, L->panel, N, K, 1);
    size_t w2 = workspace_size_no_planes(mode, last, N, K, 1);
    L->ws_bytes = w1 > w2 ? w1 : w2;
    L->offA = 0;
    L->offB = align256(L->offA + 4ull * rowsA * L->ldA);
    L->offC = align256(L->offB + 4ull * rowsB * L->ldB);
    L->offW = align256(L->offC + 4ull * M * L->ldC);
    L->total = L->offW + L->ws_bytes;
    return true;
}

}  // namespace

}  // namespace sg

using namespace sg;

extern "C" {

size_t sgemm_host_buffer_size(int mode, int M, int N, int K, int transA, int transB,
                              int panel_rows)
{
    mode = resolve_mode(mode);
    if (mode < SGEMM_MODE_FP32 || mode > SGEMM_MODE_TF32) return 0;
    if (M <= 0 || N <= 0 || K < 0 || panel_rows < 0) return 0;
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!current_sm103(&num_sms, &status)) return 0;
    Layout L;
    if (!make_layout(mode, M, N, K, transA != 0, transB != 0, panel_rows, num_sms, &L)) return 0;
    return L.total;
}

int sgemm_host(int mode, int M, int N, int K, float alpha, const float *A, int lda,
               const float *B, int ldb, float beta, float *C, int ldc, int transA, int transB,
               int panel_rows, void *dev, size_t dev_bytes, void *stream)
{
    mode = resolve_mode(mode);
    if (mode < SGEMM_MODE_FP32 || mode > SGEMM_MODE_TF32) return SGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || panel_rows < 0) return SGEMM_ERR_INVALID_ARG;
    if (transA < 0 || transA > 1 || transB < 0 || transB > 1) return SGEMM_ERR_INVALID_ARG;
    const long long need_lda = transA ? M : K, need_ldb = transB ? K : N;
    if (lda < (need_lda > 1 ? need_lda : 1) || ldb < (need_ldb > 1 ? need_ldb : 1) ||
        ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    const bool reads_ab = K > 0 && alpha != 0.f;
    if (C == nullptr || (reads_ab && (A == nullptr || B == nullptr))) return SGEMM_ERR_INVALID_ARG;
    if (dev == nullptr || (reinterpret_cast<uintptr_t>(dev) & 255) != 0)
        return SGEMM_ERR_INVALID_ARG;

    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!current_sm103(&num_sms, &status)) return SGEMM_ERR_UNSUPPORTED;
    Layout L;
    if (!make_layout(mode, M, N, K, transA, transB, panel_rows, num_sms, &L))
        return SGEMM_ERR_INVALID_ARG;
    if (dev_bytes < L.total) return SGEMM_ERR_INVALID_ARG;

    cudaStream_t st = static_cast<cudaStream_t>(stream), in = nullptr, out = nullptr;
    if (!copy_streams(&in, &out)) return SGEMM_ERR_LAUNCH;
    uint8_t *base = static_cast<uint8_t *>(dev);
    float *dA = reinterpret_cast<float *>(base + L.offA);
    float *dB = reinterpret_cast<float *>(base + L.offB);
    float *dC = reinterpret_cast<float *>(base + L.offC);
    void *ws = L.ws_bytes ? base + L.offW : nullptr;

    // K is cut into kslices slices (two when K is large): the products of
    // the first slice start once half of op(B) has arrived, while the rest
    // of the copy-in is still under way; later slices accumulate (beta = 1).
    // Slice boundaries are multiples of 32 so every slice of the device
    // copies stays 16-byte aligned.
    const int kslices = (reads_ab && K >= kKSplitMin) ? 2 : 1;
    long long kb[3] = {0, K, K};
    if (kslices == 2) kb[1] = (K / 2) / 32 * 32;

    cudaEvent_t fork = nullptr, join = nullptr, ready[2][kMaxPanels] = {}, done[kMaxPanels] = {};
    int rc = SGEMM_OK;
    auto ok = [&rc](cudaError_t e) {
        if (e != cudaSuccess && rc == SGEMM_OK) rc = SGEMM_ERR_LAUNCH;
        return rc == SGEMM_OK;
    };
    const unsigned flags = cudaEventDisableTiming;
    bool made = ok(cudaEventCreateWithFlags(&fork, flags)) &&
                ok(cudaEventCreateWithFlags(&join, flags));
    for (int p = 0; made && p < L.panels; ++p) {
        made = ok(cudaEventCreateWithFlags(&done[p], flags));
        for (int h = 0; made && h < kslices; ++h)
            made = ok(cudaEventCreateWithFlags(&ready[h][p], flags));
    }

    // The copies wait for whatever the caller queued on `stream` before.
    if (made && ok(cudaEventRecord(fork, st)) && ok(cudaStreamWaitEvent(in, fork, 0)) &&
        ok(cudaStreamWaitEvent(out, fork, 0))) {
        const size_t f = sizeof(float);
        for (int h = 0; rc == SGEMM_OK && h < kslices; ++h) {
            const long long k0 = kb[h], kn = kb[h + 1] - kb[h];
            // slice h of op(B): rows k0 .. k0+kn of K x N, or columns of N x K
            float *sB = transB ? dB + k0 : dB + k0 * L.ldB;
            if (reads_ab) {
                if (transB)
                    ok(cudaMemcpy2DAsync(sB, L.ldB * f, B + k0, ldb * f, kn * f, N,
                                         cudaMemcpyHostToDevice, in));
                else
                    ok(cudaMemcpy2DAsync(sB, L.ldB * f, B + k0 * ldb, ldb * f, N * f, kn,
                                         cudaMemcpyHostToDevice, in));
            }
            for (int p = 0; rc == SGEMM_OK && p < L.panels; ++p) {
                const long long m0 = static_cast<long long>(p) * L.panel;
                const int rows = static_cast<int>(M - m0 < L.panel ? M - m0 : L.panel);
                // slice h of this panel's rows of op(A)
                float *pA = transA ? dA + k0 * L.ldA + m0 : dA + m0 * L.ldA + k0;
                float *pC = dC + m0 * L.ldC;
                if (reads_ab) {
                    if (transA)
                        ok(cudaMemcpy2DAsync(pA, L.ldA * f, A + k0 * lda + m0, lda * f, rows * f,
                                             kn, cudaMemcpyHostToDevice, in));
                    else
                        ok(cudaMemcpy2DAsync(pA, L.ldA * f, A + m0 * lda + k0, lda * f, kn * f,
                                             rows, cudaMemcpyHostToDevice, in));
                }
                if (h == 0 && beta != 0.f)
                    ok(cudaMemcpy2DAsync(pC, L.ldC * f, C + m0 * ldc, ldc * f, N * f, rows,
                                         cudaMemcpyHostToDevice, in));
                if (!ok(cudaEventRecord(ready[h][p], in)) ||
                    !ok(cudaStreamWaitEvent(st, ready[h][p], 0)))
                    break;
                const int g = sgemm_batched_ex_ws(
                    mode, rows, N, static_cast<int>(kn), alpha, reads_ab ? pA : nullptr,
                    static_cast<int>(L.ldA), reads_ab ? sB : nullptr, static_cast<int>(L.ldB),
                    h == 0 ? beta : 1.f, pC, static_cast<int>(L.ldC), transA, transB, 0, 0, 0, 1,
                    ws, L.ws_bytes, st);
                if (g != SGEMM_OK) {
                    rc = g;
                    break;
                }
                if (h + 1 < kslices) continue;
                if (!ok(cudaEventRecord(done[p], st)) || !ok(cudaStreamWaitEvent(out, done[p], 0)))
                    break;
                ok(cudaMemcpy2DAsync(C + m0 * ldc, ldc * f, pC, L.ldC * f, N * f, rows,
                                     cudaMemcpyDeviceToHost, out));
            }
        }
    }
    // `stream` reaches its next work only once every copy-out is done (also
    // after a failure part-way, so that nothing the call queued outlives it
    // unordered).
    if (join && cudaEventRecord(join, out) == cudaSuccess) ok(cudaStreamWaitEvent(st, join, 0));
    // Destroying a recorded event is safe: it is released once it completes.
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    for (int p = 0; p < L.panels; ++p) {
        for (int h = 0; h < 2; ++h)
            if (ready[h][p]) cudaEventDestroy(ready[h][p]);
        if (done[p]) cudaEventDestroy(done[p]);
    }
    return rc;
}

}  // extern "C"
