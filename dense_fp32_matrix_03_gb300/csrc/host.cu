// host.cu -- the product on host buffers.  The operands are copied into a
// device buffer the caller provides, the product is computed there, and C
// is copied back.  op(B) is copied first, then C is cut into panels of rows:
// the copy-in of one panel's rows of op(A), the products of earlier panels
// and the copy-out of a finished one run at the same time on four streams,
// ordered by events -- the products of even panels on the caller's stream,
// of odd panels on a library stream (each with its own split-K workspace),
// so that one panel's product fills the multiprocessors the previous one's
// last wave leaves idle, and one library stream per copy direction.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "internal.h"

namespace sg {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPanels = 64;

// Copy streams (and the second product stream) of a device, made on first
// use and kept for the process.
struct CopyStreams {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp = nullptr;
};
std::mutex g_copy_mu;
CopyStreams g_copy[kMaxDevices];

bool copy_streams(cudaStream_t *in, cudaStream_t *out, cudaStream_t *comp)
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
        if (cudaStreamCreateWithFlags(&c.comp, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(c.in);
            cudaStreamDestroy(c.out);
            return false;
        }
        c.ready = true;
    }
    *in = c.in;
    *out = c.out;
    *comp = c.comp;
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A pitched copy; one contiguous copy when both pitches equal the row width
// (measured on GB300, 3xTF32 at 4092^3: a call took 1.084 ms with every
// copy in the 2-D form, 0.992 ms with the contiguous ones issued as 1-D
// copies).
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                      size_t height, cudaMemcpyKind kind, cudaStream_t s)
{
    if (dpitch == width && spitch == width)
        return cudaMemcpyAsync(dst, src, width * height, kind, s);
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, s);
}
long long round4(long long x) { return x < 4 ? 4 : (x + 3) & ~3LL; }

// Where everything sits in the caller's device buffer.  Each operand is
// stored with its rows padded to a multiple of four floats, so that the
// kernels' TMA feeds can describe it whatever the host pitch; then one
// split-K workspace per product stream.
struct Layout {
    long long ldA, ldB, ldC;       // device row pitches (elements)
    size_t offA, offB, offC, offW; // byte offsets into the buffer (offW: two workspaces)
    size_t ws_bytes, total;
    int panel, panels;             // rows of C per panel, panel count
};

// Rows per panel when the caller leaves it to the library: as many whole
// rows of output tiles as fit in one wave of the GPU (at least one), so
// that two panels' products, on the two product streams, together fill it
// (measured on GB300, 3xTF32 at 4092^3 with 1-D copies, ms per call:
// 512-row panels 1.004, 768 1.086, 1024 1.117; on one product stream
// 1.133 / 1.079 / 1.108; the earlier schedule, K cut in two slices with
// 768-row panels on one product stream, 1.076), at most kMaxPanels.
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
    long long rows_tiles = static_cast<long long>(slots) / tiles_n;
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
    L->total = L->offW + 2 * align256(L->ws_bytes);
    // Every panel's product is a workspace-entry call on the device copies,
    // which takes the routes the cost models pick (3xTF32 at 4092^3: the raw
    // route with the lo planes made in the kernel, no pass).  Measured on
    // GB300, 3xTF32 4092^3, ms per call, interleaved: 0.943 with op(B)
    // written as TF32 planes once and each panel's op(A) before its product
    // (the planes route), 0.921 without (the device copies keep the host's
    // row pitch, off 128-byte lines at 4092 floats; 128-byte-pitched copies,
    // pitched rather than contiguous, made the call 1.08-1.15 ms).
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

    cudaStream_t st = static_cast<cudaStream_t>(stream), in = nullptr, out = nullptr,
                 comp = nullptr;
    if (!copy_streams(&in, &out, &comp)) return SGEMM_ERR_LAUNCH;
    uint8_t *base = static_cast<uint8_t *>(dev);
    float *dA = reinterpret_cast<float *>(base + L.offA);
    float *dB = reinterpret_cast<float *>(base + L.offB);
    float *dC = reinterpret_cast<float *>(base + L.offC);
    // panel p's product: stream and split-K workspace of its parity
    void *ws_of[2] = {L.ws_bytes ? base + L.offW : nullptr,
                      L.ws_bytes ? base + L.offW + align256(L.ws_bytes) : nullptr};
    cudaStream_t st_of[2] = {st, comp};

    cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr, ready[kMaxPanels] = {},
                done[kMaxPanels] = {};
    int rc = SGEMM_OK;
    auto ok = [&rc](cudaError_t e) {
        if (e != cudaSuccess && rc == SGEMM_OK) rc = SGEMM_ERR_LAUNCH;
        return rc == SGEMM_OK;
    };
    const unsigned flags = cudaEventDisableTiming;
    bool made = ok(cudaEventCreateWithFlags(&fork, flags)) &&
                ok(cudaEventCreateWithFlags(&join, flags)) &&
                ok(cudaEventCreateWithFlags(&join2, flags));
    for (int p = 0; made && p < L.panels; ++p)
        made = ok(cudaEventCreateWithFlags(&done[p], flags)) &&
               ok(cudaEventCreateWithFlags(&ready[p], flags));

    // Every stream waits for whatever the caller queued on `stream` before.
    if (made && ok(cudaEventRecord(fork, st)) && ok(cudaStreamWaitEvent(in, fork, 0)) &&
        ok(cudaStreamWaitEvent(out, fork, 0)) && ok(cudaStreamWaitEvent(comp, fork, 0))) {
        const size_t f = sizeof(float);
        if (reads_ab)  // op(B) whole: K x N, or N x K when transposed
            ok(transB ? copy_rows(dB, L.ldB * f, B, ldb * f, K * f, N,
                                  cudaMemcpyHostToDevice, in)
                      : copy_rows(dB, L.ldB * f, B, ldb * f, N * f, K,
                                  cudaMemcpyHostToDevice, in));
        for (int p = 0; rc == SGEMM_OK && p < L.panels; ++p) {
            const long long m0 = static_cast<long long>(p) * L.panel;
            const int rows = static_cast<int>(M - m0 < L.panel ? M - m0 : L.panel);
            // this panel's rows of op(A) (columns m0.. of A when transposed)
            float *pA = transA ? dA + m0 : dA + m0 * L.ldA;
            float *pC = dC + m0 * L.ldC;
            if (reads_ab) {
                if (transA)
                    ok(copy_rows(pA, L.ldA * f, A + m0, lda * f, rows * f, K,
                                 cudaMemcpyHostToDevice, in));
                else
                    ok(copy_rows(pA, L.ldA * f, A + m0 * lda, lda * f, K * f, rows,
                                 cudaMemcpyHostToDevice, in));
            }
            if (beta != 0.f)
                ok(copy_rows(pC, L.ldC * f, C + m0 * ldc, ldc * f, N * f, rows,
                             cudaMemcpyHostToDevice, in));
            cudaStream_t ps = st_of[p & 1];
            if (!ok(cudaEventRecord(ready[p], in)) || !ok(cudaStreamWaitEvent(ps, ready[p], 0)))
                break;
            const int g = sgemm_batched_ex_ws(
                mode, rows, N, K, alpha, reads_ab ? pA : nullptr, static_cast<int>(L.ldA),
                reads_ab ? dB : nullptr, static_cast<int>(L.ldB), beta, pC,
                static_cast<int>(L.ldC), transA, transB, 0, 0, 0, 1, ws_of[p & 1], L.ws_bytes,
                ps);
            if (g != SGEMM_OK) {
                rc = g;
                break;
            }
            if (!ok(cudaEventRecord(done[p], ps)) || !ok(cudaStreamWaitEvent(out, done[p], 0)))
                break;
            ok(copy_rows(C + m0 * ldc, ldc * f, pC, L.ldC * f, N * f, rows,
                         cudaMemcpyDeviceToHost, out));
        }
    }
    // `stream` reaches its next work only once every copy-out and every
    // product on the second stream is done (also after a failure part-way,
    // so that nothing the call queued outlives it unordered).
    if (join && cudaEventRecord(join, out) == cudaSuccess) ok(cudaStreamWaitEvent(st, join, 0));
    if (join2 && cudaEventRecord(join2, comp) == cudaSuccess) ok(cudaStreamWaitEvent(st, join2, 0));
    // Destroying a recorded event is safe: it is released once it completes.
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    if (join2) cudaEventDestroy(join2);
    for (int p = 0; p < L.panels; ++p) {
        if (ready[p]) cudaEventDestroy(ready[p]);
        if (done[p]) cudaEventDestroy(done[p]);
    }
    return rc;
}

}  // extern "C"
