// linattn.cu -- chunked linear attention with a decay, fp32 on the CUDA
// cores: the chunk kernels "From 1% to 94% of cuBLAS, one kernel at a time"
// describes in "What FLA builds on top of this" and "Why FLA sits somewhere
// else on the roofline", as building blocks behind include/linear_attention.h.
//
// Per head, the recurrence S_t = exp(g_t) S_{t-1} + k_t^T v_t, o_t = scale
// q_t S_t (S_{-1} = h0) is computed in chunks of BT = 64 tokens.  With G_t the
// running sum of g inside a chunk and h_c the state before chunk c:
//   o_t     = scale (exp(G_t) q_t h_c + sum_{s <= t} exp(G_t - G_s) (q_t . k_s) v_s)
//   h_{c+1} = exp(G_last) h_c + sum_s exp(G_last - G_s) k_s^T v_s
//
// Three kernels, one CTA of 256 threads each:
//   la_state_kernel   grid (DV / 64, BH): the scan over chunks.  A CTA keeps
//                     its K x 64 slice of S in registers (thread (ti, tj):
//                     rows 4 ti + 64 r, columns 4 tj), stores each chunk's
//                     starting state to h, then adds the chunk's decayed
//                     K^T V.  Parallelism: heads x state slices (the scan is
//                     sequential in the chunks, as the pages note).
//   la_output_kernel  grid (NT, BH): one chunk of one head: A = Q K^T in
//                     registers (thread (ti, tj): rows ti + 16 r, columns
//                     tj + 16 c), masked, scaled and decayed into shared
//                     memory, then O = A V + scale exp(G_t) (Q h_c), thread
//                     (ti, tj): rows ti + 16 r, columns 4 tj + 64 c.
//   la_fused_kernel   grid (DV / 64, BH): both in one pass, chunk after
//                     chunk, the state never leaving the CTA (registers for
//                     the update, a shared copy for Q S).
// Operands are staged in shared memory with rows padded by four floats so
// that sixteen lanes reading sixteen consecutive rows' 16-byte words hit
// distinct banks.  Every accumulation is fp32 FMA; exp is the CUDA expf.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/linear_attention.h"
#include "../../include/sgemm.h"
#include "internal.h"

namespace sg {
namespace la {

constexpr int BT = 64;        // tokens per chunk
constexpr int BV = 64;        // state / output columns per CTA (state and fused kernels)
constexpr int kThreads = 256;

struct Args {
    const float *q, *k, *v, *g, *h0;
    float *h, *o, *state_out;
    int T, NT;
    float scale;
};

// Copies rows [0, n) of `cols` floats (global row pitch gp, first column c0)
// into shared memory rows of pitch sp, zero-filling rows n .. BT-1.
template <int COLS>
__device__ __forceinline__ void stage_rows(float *dst, int sp, const float *src, long long gp,
                                           int n, int tid)
{
    constexpr int V4 = COLS / 4;
    for (int i = tid; i < BT * V4; i += kThreads) {
        const int r = i / V4, c = (i - r * V4) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < n) x = *reinterpret_cast<const float4 *>(src + r * gp + c);
        *reinterpret_cast<float4 *>(dst + r * sp + c) = x;
    }
}

// G[t] = g[0] + ... + g[t] over the chunk's n tokens (constant past them;
// zero without a decay), by warp 0: lane l sums tokens 2l, 2l+1, then an
// inclusive scan across the lanes.
__device__ __forceinline__ void chunk_decay(const float *g, int n, float *G, int tid)
{
    if (tid >= 32) return;
    const int l = tid;
    const float a = (g != nullptr && 2 * l < n) ? g[2 * l] : 0.f;
    const float b = (g != nullptr && 2 * l + 1 < n) ? g[2 * l + 1] : 0.f;
    float s = a + b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (l >= off) s += y;
    }
    G[2 * l] = s - b;
    G[2 * l + 1] = s;
}

__device__ __forceinline__ void fma4(float (&acc)[4], float a, const float4 b)
{
    acc[0] = fmaf(a, b.x, acc[0]);
    acc[1] = fmaf(a, b.y, acc[1]);
    acc[2] = fmaf(a, b.z, acc[2]);
    acc[3] = fmaf(a, b.w, acc[3]);
}

// ---------------------------------------------------------------- state pass

// The thread's slice of a K x 64 state tile: rows 4 ti + 64 r + e, columns
// 4 tj + f (ti = tid / 16, tj = tid % 16, r < K / 64, e, f < 4).
template <int DK>
struct StateRegs {
    static constexpr int R = DK / 64;
    float s[R][4][4];
};

// S = a S + sum_s Ks[s]^T Vw[s] (Vw: the chunk's V rows already weighted by
// exp(G_last - G_s)); Ks pitch DK + 4, Vw pitch BV + 4.
template <int DK>
__device__ __forceinline__ void state_update(StateRegs<DK> &S, float a, const float *Ks,
                                             const float *Vw, int ti, int tj)
{
    constexpr int KP = DK + 4, VP = BV + 4;
#pragma unroll
    for (int r = 0; r < StateRegs<DK>::R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int f = 0; f < 4; ++f) S.s[r][e][f] *= a;
#pragma unroll 4
    for (int s = 0; s < BT; ++s) {
        const float4 vv = *reinterpret_cast<const float4 *>(Vw + s * VP + 4 * tj);
#pragma unroll
        for (int r = 0; r < StateRegs<DK>::R; ++r) {
            const float4 kk = *reinterpret_cast<const float4 *>(Ks + s * KP + 4 * ti + 64 * r);
            fma4(S.s[r][0], kk.x, vv);
            fma4(S.s[r][1], kk.y, vv);
            fma4(S.s[r][2], kk.z, vv);
            fma4(S.s[r][3], kk.w, vv);
        }
    }
}

// Stores the thread's slice of S to a K x DV row-major matrix at dst
// (columns v0 ..), or to shared memory rows of pitch `pitch`.
template <int DK>
__device__ __forceinline__ void state_store(const StateRegs<DK> &S, float *dst, long long pitch,
                                            int v0, int ti, int tj)
{
#pragma unroll
    for (int r = 0; r < StateRegs<DK>::R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<float4 *>(dst + (4 * ti + 64 * r + e) * pitch + v0 + 4 * tj) =
                make_float4(S.s[r][e][0], S.s[r][e][1], S.s[r][e][2], S.s[r][e][3]);
}

template <int DK>
__device__ __forceinline__ void state_load(StateRegs<DK> &S, const float *src, long long pitch,
                                           int v0, int ti, int tj)
{
#pragma unroll
    for (int r = 0; r < StateRegs<DK>::R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (src != nullptr)
                x = *reinterpret_cast<const float4 *>(src + (4 * ti + 64 * r + e) * pitch + v0 +
                                                      4 * tj);
            S.s[r][e][0] = x.x;
            S.s[r][e][1] = x.y;
            S.s[r][e][2] = x.z;
            S.s[r][e][3] = x.w;
        }
}

// Stages the chunk's K (all DK columns) and V (columns v0 .. v0 + 63), the
// running decay G and the state update's weights: V rows scaled by
// exp(G_last - G_s) (zero past the chunk's n tokens).  Returns
// exp(G_last).  Ends with a barrier.
template <int DK, int DV>
__device__ __forceinline__ float stage_update_operands(const Args &p, long long head, int t0,
                                                       int n, int v0, float *Ks, float *Vw,
                                                       float *G, int tid)
{
    stage_rows<DK>(Ks, DK + 4, p.k + (head * p.T + t0) * DK, DK, n, tid);
    stage_rows<BV>(Vw, BV + 4, p.v + (head * p.T + t0) * DV + v0, DV, n, tid);
    chunk_decay(p.g != nullptr ? p.g + head * p.T + t0 : nullptr, n, G, tid);
    __syncthreads();
    const float glast = G[n - 1];
    for (int i = tid; i < BT * (BV / 4); i += kThreads) {
        const int s = i / (BV / 4), c = (i - s * (BV / 4)) * 4;
        const float w = s < n ? expf(glast - G[s]) : 0.f;
        float4 *x = reinterpret_cast<float4 *>(Vw + s * (BV + 4) + c);
        float4 y = *x;
        y.x *= w;
        y.y *= w;
        y.z *= w;
        y.w *= w;
        *x = y;
    }
    __syncthreads();
    return expf(glast);
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) la_state_kernel(const Args p)
{
    extern __shared__ float4 smem4[];
    float *Ks = reinterpret_cast<float *>(smem4);  // BT x (DK + 4)
    float *Vw = Ks + BT * (DK + 4);                // BT x (BV + 4)
    float *G = Vw + BT * (BV + 4);                 // BT
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    const int v0 = blockIdx.x * BV;
    const long long head = blockIdx.y;
    StateRegs<DK> S;
    state_load<DK>(S, p.h0 != nullptr ? p.h0 + head * DK * DV : nullptr, DV, v0, ti, tj);
    for (int c = 0; c < p.NT; ++c) {
        const int t0 = c * BT, n = min(BT, p.T - t0);
        state_store<DK>(S, p.h + (head * p.NT + c) * DK * DV, DV, v0, ti, tj);
        const float a = stage_update_operands<DK, DV>(p, head, t0, n, v0, Ks, Vw, G, tid);
        state_update<DK>(S, a, Ks, Vw, ti, tj);
        __syncthreads();  // before the next chunk overwrites Ks, Vw, G
    }
    if (p.state_out != nullptr)
        state_store<DK>(S, p.state_out + head * DK * DV, DV, v0, ti, tj);
}

// --------------------------------------------------------------- output pass

// A = Q K^T for the chunk (Qs, Ks: pitch DK + 4), then masked (s <= t < n),
// scaled and decayed: As[t][s] = scale exp(G_t - G_s) (q_t . k_s) (pitch
// BT + 4).  Thread (ti, tj): rows ti + 16 r, columns tj + 16 c.  Ends with a
// barrier.
template <int DK>
__device__ __forceinline__ void attention_tile(const float *Qs, const float *Ks, const float *G,
                                               int n, float scale, float *As, int ti, int tj)
{
    constexpr int KP = DK + 4;
    float acc[4][4] = {};
#pragma unroll 2
    for (int k = 0; k < DK; k += 4) {
        float4 qa[4], kb[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            qa[r] = *reinterpret_cast<const float4 *>(Qs + (ti + 16 * r) * KP + k);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            kb[c] = *reinterpret_cast<const float4 *>(Ks + (tj + 16 * c) * KP + k);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc[r][c] = fmaf(qa[r].x, kb[c].x, acc[r][c]);
                acc[r][c] = fmaf(qa[r].y, kb[c].y, acc[r][c]);
                acc[r][c] = fmaf(qa[r].z, kb[c].z, acc[r][c]);
                acc[r][c] = fmaf(qa[r].w, kb[c].w, acc[r][c]);
            }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = ti + 16 * r;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int s = tj + 16 * c;
            As[t * (BT + 4) + s] =
                (s <= t && t < n) ? scale * expf(G[t] - G[s]) * acc[r][c] : 0.f;
        }
    }
    __syncthreads();
}

// O rows ti + 16 r, columns cb + 4 tj + 64 c (c < NC): intra = A V (As
// pitch BT + 4, Vs pitch vp), inter = Q X (Qs pitch DK + 4, X: DK rows of
// pitch xp); o = intra + scale exp(G_t) inter, stored for rows t < n to
// dst (row pitch dp).
template <int DK, int NC>
__device__ __forceinline__ void output_tile(const float *As, const float *Vs, int vp,
                                            const float *Qs, const float *X, int xp,
                                            const float *G, int n, float scale, float *dst,
                                            long long dp, int ti, int tj)
{
    constexpr int KP = DK + 4;
    float intra[4][NC][4] = {}, inter[4][NC][4] = {};
#pragma unroll 4
    for (int s = 0; s < BT; ++s) {
        float4 vv[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c)
            vv[c] = *reinterpret_cast<const float4 *>(Vs + s * vp + 4 * tj + 64 * c);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float a = As[(ti + 16 * r) * (BT + 4) + s];
#pragma unroll
            for (int c = 0; c < NC; ++c) fma4(intra[r][c], a, vv[c]);
        }
    }
#pragma unroll 4
    for (int k = 0; k < DK; ++k) {
        float4 xx[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c)
            xx[c] = *reinterpret_cast<const float4 *>(X + k * xp + 4 * tj + 64 * c);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float qv = Qs[(ti + 16 * r) * KP + k];
#pragma unroll
            for (int c = 0; c < NC; ++c) fma4(inter[r][c], qv, xx[c]);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = ti + 16 * r;
        if (t >= n) continue;
        const float e = scale * expf(G[t]);
#pragma unroll
        for (int c = 0; c < NC; ++c)
            *reinterpret_cast<float4 *>(dst + t * dp + 4 * tj + 64 * c) =
                make_float4(fmaf(e, inter[r][c][0], intra[r][c][0]),
                            fmaf(e, inter[r][c][1], intra[r][c][1]),
                            fmaf(e, inter[r][c][2], intra[r][c][2]),
                            fmaf(e, inter[r][c][3], intra[r][c][3]));
    }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) la_output_kernel(const Args p)
{
    extern __shared__ float4 smem4[];
    float *Qs = reinterpret_cast<float *>(smem4);  // BT x (DK + 4)
    float *Ks = Qs + BT * (DK + 4);                // BT x (DK + 4)
    float *Vs = Ks + BT * (DK + 4);                // BT x DV
    float *Hs = Vs + BT * DV;                      // DK x DV
    float *As = Hs + DK * DV;                      // BT x (BT + 4)
    float *G = As + BT * (BT + 4);                 // BT
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    const int c = blockIdx.x;
    const long long head = blockIdx.y;
    const int t0 = c * BT, n = min(BT, p.T - t0);
    stage_rows<DK>(Qs, DK + 4, p.q + (head * p.T + t0) * DK, DK, n, tid);
    stage_rows<DK>(Ks, DK + 4, p.k + (head * p.T + t0) * DK, DK, n, tid);
    stage_rows<DV>(Vs, DV, p.v + (head * p.T + t0) * DV, DV, n, tid);
    {
        const float4 *src = reinterpret_cast<const float4 *>(p.h + (head * p.NT + c) * DK * DV);
        float4 *dst = reinterpret_cast<float4 *>(Hs);
        for (int i = tid; i < DK * DV / 4; i += kThreads) dst[i] = src[i];
    }
    chunk_decay(p.g != nullptr ? p.g + head * p.T + t0 : nullptr, n, G, tid);
    __syncthreads();
    attention_tile<DK>(Qs, Ks, G, n, p.scale, As, ti, tj);
    output_tile<DK, DV / 64>(As, Vs, DV, Qs, Hs, DV, G, n, p.scale,
                             p.o + (head * p.T + t0) * DV, DV, ti, tj);
}

// ---------------------------------------------------------------- fused pass

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads) la_fused_kernel(const Args p)
{
    extern __shared__ float4 smem4[];
    float *Qs = reinterpret_cast<float *>(smem4);  // BT x (DK + 4)
    float *Ks = Qs + BT * (DK + 4);                // BT x (DK + 4)
    float *Vs = Ks + BT * (DK + 4);                // BT x (BV + 4): V, then weighted V
    float *Ss = Vs + BT * (BV + 4);                // DK x BV: the state before the chunk
    float *As = Ss + DK * BV;                      // BT x (BT + 4)
    float *G = As + BT * (BT + 4);                 // BT
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    const int v0 = blockIdx.x * BV;
    const long long head = blockIdx.y;
    StateRegs<DK> S;
    state_load<DK>(S, p.h0 != nullptr ? p.h0 + head * DK * DV : nullptr, DV, v0, ti, tj);
    for (int c = 0; c < p.NT; ++c) {
        const int t0 = c * BT, n = min(BT, p.T - t0);
        state_store<DK>(S, Ss, BV, 0, ti, tj);
        stage_rows<DK>(Qs, DK + 4, p.q + (head * p.T + t0) * DK, DK, n, tid);
        stage_rows<DK>(Ks, DK + 4, p.k + (head * p.T + t0) * DK, DK, n, tid);
        stage_rows<BV>(Vs, BV + 4, p.v + (head * p.T + t0) * DV + v0, DV, n, tid);
        chunk_decay(p.g != nullptr ? p.g + head * p.T + t0 : nullptr, n, G, tid);
        __syncthreads();
        attention_tile<DK>(Qs, Ks, G, n, p.scale, As, ti, tj);
        output_tile<DK, 1>(As, Vs, BV + 4, Qs, Ss, BV, G, n, p.scale,
                           p.o + (head * p.T + t0) * DV + v0, DV, ti, tj);
        // the state update: V rows weighted by exp(G_last - G_s)
        const float glast = G[n - 1];
        __syncthreads();  // every thread is done reading Vs as V
        for (int i = tid; i < BT * (BV / 4); i += kThreads) {
            const int s = i / (BV / 4), cc = (i - s * (BV / 4)) * 4;
            const float w = s < n ? expf(glast - G[s]) : 0.f;
            float4 *x = reinterpret_cast<float4 *>(Vs + s * (BV + 4) + cc);
            float4 y = *x;
            y.x *= w;
            y.y *= w;
            y.z *= w;
            y.w *= w;
            *x = y;
        }
        __syncthreads();
        state_update<DK>(S, expf(glast), Ks, Vs, ti, tj);
        __syncthreads();  // before the next chunk overwrites the staged operands
    }
    if (p.state_out != nullptr)
        state_store<DK>(S, p.state_out + head * DK * DV, DV, v0, ti, tj);
}

template <int DK, int DV>
constexpr size_t state_smem()
{
    return sizeof(float) * (BT * (DK + 4) + BT * (BV + 4) + BT);
}
template <int DK, int DV>
constexpr size_t output_smem()
{
    return sizeof(float) * (2 * BT * (DK + 4) + BT * DV + DK * DV + BT * (BT + 4) + BT);
}
template <int DK, int DV>
constexpr size_t fused_smem()
{
    return sizeof(float) * (2 * BT * (DK + 4) + BT * (BV + 4) + DK * BV + BT * (BT + 4) + BT);
}

enum Which { kState, kOutput, kFused };

template <int DK, int DV>
int launch(Which w, const Args &a, int BH, cudaStream_t st)
{
    void (*kern)(const Args);
    size_t smem;
    dim3 grid;
    if (w == kState) {
        kern = la_state_kernel<DK, DV>;
        smem = state_smem<DK, DV>();
        grid = dim3(DV / BV, static_cast<unsigned>(BH));
    } else if (w == kOutput) {
        kern = la_output_kernel<DK, DV>;
        smem = output_smem<DK, DV>();
        grid = dim3(static_cast<unsigned>(a.NT), static_cast<unsigned>(BH));
    } else {
        kern = la_fused_kernel<DK, DV>;
        smem = fused_smem<DK, DV>();
        grid = dim3(DV / BV, static_cast<unsigned>(BH));
    }
    if (grid.x == 0 || grid.y == 0) return SGEMM_OK;
    if (!smem_attr_once(reinterpret_cast<const void *>(kern), static_cast<int>(smem)))
        return SGEMM_ERR_LAUNCH;
    kern<<<grid, kThreads, smem, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    note_launch();
    return SGEMM_OK;
}

int dispatch(Which w, const Args &a, int BH, int DK, int DV, cudaStream_t st)
{
    if (DK == 64 && DV == 64) return launch<64, 64>(w, a, BH, st);
    if (DK == 64 && DV == 128) return launch<64, 128>(w, a, BH, st);
    if (DK == 128 && DV == 64) return launch<128, 64>(w, a, BH, st);
    return launch<128, 128>(w, a, BH, st);
}

bool aligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dims_ok(int BH, int T, int DK, int DV)
{
    return BH >= 0 && T >= 0 && (DK == 64 || DK == 128) && (DV == 64 || DV == 128) &&
           BH <= 65535 && (T + BT - 1) / BT <= 0x7FFFFFFF;
}

}  // namespace la
}  // namespace sg

using namespace sg::la;

extern "C" {

size_t la_state_bytes(int BH, int T, int DK, int DV)
{
    if (!dims_ok(BH, T, DK, DV)) return 0;
    return static_cast<size_t>(BH) * ((static_cast<size_t>(T) + BT - 1) / BT) * DK * DV *
           sizeof(float);
}

int la_chunk_state(int BH, int T, int DK, int DV, const float *k, const float *v,
                   const float *g, const float *h0, float *h, float *state_out, void *stream)
{
    if (!dims_ok(BH, T, DK, DV)) return SGEMM_ERR_INVALID_ARG;
    if (BH == 0) return SGEMM_OK;
    const bool tokens = T > 0;
    if (tokens && (k == nullptr || v == nullptr || h == nullptr)) return SGEMM_ERR_INVALID_ARG;
    if (!aligned(k) || !aligned(v) || !aligned(h) || !aligned(h0) || !aligned(state_out) ||
        (reinterpret_cast<uintptr_t>(g) & 3u) != 0)
        return SGEMM_ERR_INVALID_ARG;
    if (!tokens && state_out == nullptr) return SGEMM_OK;
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!sg::current_sm103(&num_sms, &status)) return SGEMM_ERR_UNSUPPORTED;
    Args a{nullptr, k, v, g, h0, h, nullptr, state_out, T, (T + BT - 1) / BT, 1.f};
    return dispatch(kState, a, BH, DK, DV, static_cast<cudaStream_t>(stream));
}

int la_chunk_output(int BH, int T, int DK, int DV, float scale, const float *q, const float *k,
                    const float *v, const float *g, const float *h, float *o, void *stream)
{
    if (!dims_ok(BH, T, DK, DV)) return SGEMM_ERR_INVALID_ARG;
    if (BH == 0 || T == 0) return SGEMM_OK;
    if (q == nullptr || k == nullptr || v == nullptr || h == nullptr || o == nullptr)
        return SGEMM_ERR_INVALID_ARG;
    if (!aligned(q) || !aligned(k) || !aligned(v) || !aligned(h) || !aligned(o) ||
        (reinterpret_cast<uintptr_t>(g) & 3u) != 0)
        return SGEMM_ERR_INVALID_ARG;
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!sg::current_sm103(&num_sms, &status)) return SGEMM_ERR_UNSUPPORTED;
    Args a{q, k, v, g, nullptr, const_cast<float *>(h), o, nullptr, T, (T + BT - 1) / BT, scale};
    return dispatch(kOutput, a, BH, DK, DV, static_cast<cudaStream_t>(stream));
}

int la_chunk_fused(int BH, int T, int DK, int DV, float scale, const float *q, const float *k,
                   const float *v, const float *g, const float *h0, float *o, float *state_out,
                   void *stream)
{
    if (!dims_ok(BH, T, DK, DV)) return SGEMM_ERR_INVALID_ARG;
    if (BH == 0) return SGEMM_OK;
    const bool tokens = T > 0;
    if (tokens && (q == nullptr || k == nullptr || v == nullptr || o == nullptr))
        return SGEMM_ERR_INVALID_ARG;
    if (!aligned(q) || !aligned(k) || !aligned(v) || !aligned(o) || !aligned(h0) ||
        !aligned(state_out) || (reinterpret_cast<uintptr_t>(g) & 3u) != 0)
        return SGEMM_ERR_INVALID_ARG;
    if (!tokens && state_out == nullptr) return SGEMM_OK;
    int num_sms = 0;
    unsigned int *status = nullptr;
    if (!sg::current_sm103(&num_sms, &status)) return SGEMM_ERR_UNSUPPORTED;
    Args a{q, k, v, g, h0, nullptr, o, state_out, T, (T + BT - 1) / BT, scale};
    return dispatch(kFused, a, BH, DK, DV, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
