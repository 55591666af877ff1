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
// Three kernels, one CTA of 256 threads each, operands staged in shared
// memory by cp.async with rows padded by four floats (sixteen lanes reading
// sixteen rows' 16-byte words at one column hit distinct banks):
//   la_state_kernel   grid (DV / 64, DK / 64, BH), two CTAs per SM: the scan
//                     over chunks.  A CTA keeps a 64 x 64 slice of S in
//                     registers (thread (ti, tj): rows 4 ti + e, columns
//                     4 tj + f), stores each chunk's starting state to h and
//                     adds the chunk's K^T (w V), w the decay weights; the
//                     next two chunks' slices are in flight meanwhile.
//   la_output_kernel  grid (NT, BH), two CTAs per SM: one chunk of one head.
//                     A = Q K^T (thread (ti, tj): rows ti + 16 r, columns
//                     tj + 16 c), masked, scaled and decayed in shared
//                     memory; then one accumulator takes A V and the
//                     earlier chunks' (scale exp(G_t) q_t) h_c (thread
//                     (ti, tj): rows ti + 16 r, columns 4 tj + 64 c).
//   la_fused_kernel   grid (DV / 64, BH): both in one pass, the state slice
//                     never leaving the CTA, the next chunk's operands in
//                     flight while this one is computed.
// Parallelism: the state and fused passes are sequential in the chunks (the
// scan the pages describe); the output pass is parallel over chunks.  Every
// product and sum is an fp32 FMA; exp is the CUDA expf.
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/linear_attention.h"
#include "../../include/sgemm.h"
#include "common.cuh"
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

// 16-byte asynchronous copy global -> shared; zero-filled when !valid (src
// is then not read, but must be a valid address).
__device__ __forceinline__ void cp16(float *dst, const float *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Issues the copies of rows [0, n) of COLS floats (global pitch gp) into
// shared rows of pitch sp, zero-filling rows n .. BT-1 (no commit).
template <int COLS>
__device__ __forceinline__ void stage_rows_async(float *dst, int sp, const float *src,
                                                 long long gp, int n, int tid)
{
    constexpr int V4 = COLS / 4;
    for (int i = tid; i < BT * V4; i += kThreads) {
        const int r = i / V4, c = (i - r * V4) * 4;
        cp16(dst + r * sp + c, r < n ? src + r * gp + c : src, r < n);
    }
}

// Packed accumulation: two fp32 FMAs per instruction (fma.rn.f32x2 on a
// 64-bit register pair; each half rounded exactly as a scalar fmaf, so the
// results are those of scalar FMAs).  A 16-byte shared load gives two such
// pairs; the scalar factor is broadcast into both halves.
__device__ __forceinline__ unsigned long long dup2(float x)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void fma2(unsigned long long &d, unsigned long long a,
                                     unsigned long long b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ float2 unpack2(unsigned long long r)
{
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
// acc (four values as two pairs) += a * (b.x, b.y, b.z, b.w)
__device__ __forceinline__ void fma4p(unsigned long long (&acc)[2], float a, const ulonglong2 b)
{
    const unsigned long long aa = dup2(a);
    fma2(acc[0], aa, b.x);
    fma2(acc[1], aa, b.y);
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

// The chunk's decay for the state update, by warp 0 into W, from the
// chunk's log-decays (lane l holds tokens 2l, 2l+1 in a, b; zero past the
// chunk's n tokens): W[s] = exp(G_last - G_s) for s < n (0 past them),
// W[BT] = exp(G_last), G the running sum over the chunk.
__device__ __forceinline__ void update_weights(float a, float b, int n, float *W, int l)
{
    float s = a + b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (l >= off) s += y;
    }
    // G[n-1]: the inclusive sum up to token n-1 (lane (n-1)/2 holds it)
    const int src = (n - 1) >> 1;
    const float hi = __shfl_sync(0xffffffffu, s, src);
    const float bb = __shfl_sync(0xffffffffu, b, src);
    const float glast = ((n - 1) & 1) ? hi : hi - bb;
    W[2 * l] = 2 * l < n ? expf(glast - (s - b)) : 0.f;
    W[2 * l + 1] = 2 * l + 1 < n ? expf(glast - s) : 0.f;
    if (l == 0) W[BT] = expf(glast);
}

// Warp 0's pair of a chunk's log-decays (see update_weights).
__device__ __forceinline__ void load_decay_pair(const Args &p, long long head, int c, int l,
                                                float &a, float &b)
{
    a = b = 0.f;
    if (p.g == nullptr || c >= p.NT) return;
    const int t0 = c * BT, n = min(BT, p.T - t0);
    const float *g = p.g + head * p.T + t0;
    if (2 * l < n) a = g[2 * l];
    if (2 * l + 1 < n) b = g[2 * l + 1];
}

// The state pass, grid (DV / 64, DK / 64, BH): a CTA owns a 64 x 64 slice of
// one head's state, rows k0 = 64 blockIdx.y .., columns v0 = 64 blockIdx.x
// .. -- thread (ti, tj) rows k0 + 4 ti + e, columns v0 + 4 tj + f -- and
// walks the chunks in order.  The K and V slices of the next two chunks are
// in flight (cp.async, three buffers) while this one's update runs, and
// warp 0 holds the next chunk's log-decays in registers; the decay weights
// multiply the K values as they are read.
constexpr int kStateBufs = 3;
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2) la_state_kernel(const Args p)
{
    constexpr int P = 64 + 4;  // row pitch of the staged slices
    extern __shared__ float4 smem4[];
    float *Kb = reinterpret_cast<float *>(smem4);  // kStateBufs x BT x P
    float *Vb = Kb + kStateBufs * BT * P;          // kStateBufs x BT x P
    float *W = Vb + kStateBufs * BT * P;           // BT + 1
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    const int v0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
    const long long head = blockIdx.z;
    unsigned long long S[4][2];  // row 4 ti + e, columns (4 tj, +1) and (+2, +3), packed
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        ulonglong2 x = make_ulonglong2(0ull, 0ull);
        if (p.h0 != nullptr)
            x = *reinterpret_cast<const ulonglong2 *>(p.h0 + (head * DK + k0 + 4 * ti + e) * DV +
                                                      v0 + 4 * tj);
        S[e][0] = x.x;
        S[e][1] = x.y;
    }
    // one commit group per chunk (empty past the last chunk), so that
    // "all but the newest kStateBufs - 1 groups done" means "this chunk landed"
    auto issue = [&](int c) {
        if (c < p.NT) {
            const int t0 = c * BT, n = min(BT, p.T - t0), buf = c % kStateBufs;
            stage_rows_async<64>(Kb + buf * BT * P, P, p.k + (head * p.T + t0) * DK + k0, DK, n,
                                 tid);
            stage_rows_async<64>(Vb + buf * BT * P, P, p.v + (head * p.T + t0) * DV + v0, DV, n,
                                 tid);
        }
        cp_commit();
    };
    for (int c = 0; c < kStateBufs - 1; ++c) issue(c);
    float ga = 0.f, gb = 0.f;
    if (tid < 32) load_decay_pair(p, head, 0, tid, ga, gb);
    for (int c = 0; c < p.NT; ++c) {
        const int n = min(BT, p.T - c * BT), buf = c % kStateBufs;
        float *hc = p.h + ((head * p.NT + c) * DK + k0 + 4 * ti) * DV + v0 + 4 * tj;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<ulonglong2 *>(hc + e * DV) = make_ulonglong2(S[e][0], S[e][1]);
        issue(c + kStateBufs - 1);
        float na = 0.f, nb = 0.f;
        if (tid < 32) {
            load_decay_pair(p, head, c + 1, tid, na, nb);
            update_weights(ga, gb, n, W, tid);
        }
        cp_wait<kStateBufs - 1>();
        __syncthreads();
        const float *Ks = Kb + buf * BT * P;
        float *Vs = Vb + buf * BT * P;
        // V rows times their weights (each thread four 16-byte words)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int u = tid + i * kThreads, s = u >> 4, cc = (u & 15) * 4;
            float4 *x = reinterpret_cast<float4 *>(Vs + s * P + cc);
            const float w = W[s];
            float4 y = *x;
            y.x *= w;
            y.y *= w;
            y.z *= w;
            y.w *= w;
            *x = y;
        }
        {
            // S *= exp(G_last): fma with a zero addend rounds like the product
            const unsigned long long a = dup2(W[BT]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int f = 0; f < 2; ++f)
                    asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(S[e][f]) : "l"(a), "l"(0ull));
        }
        __syncthreads();
#pragma unroll 8
        for (int s = 0; s < BT; ++s) {
            const float4 kk = *reinterpret_cast<const float4 *>(Ks + s * P + 4 * ti);
            const ulonglong2 vv = *reinterpret_cast<const ulonglong2 *>(Vs + s * P + 4 * tj);
            fma4p(S[0], kk.x, vv);
            fma4p(S[1], kk.y, vv);
            fma4p(S[2], kk.z, vv);
            fma4p(S[3], kk.w, vv);
        }
        ga = na;
        gb = nb;
        __syncthreads();  // the next issue reuses a buffer read here, the next chunk W
    }
    cp_wait<0>();
    if (p.state_out != nullptr) {
        float *so = p.state_out + (head * DK + k0 + 4 * ti) * DV + v0 + 4 * tj;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<ulonglong2 *>(so + e * DV) = make_ulonglong2(S[e][0], S[e][1]);
    }
}

// --------------------------------------------------------------- output pass

// A = Q K^T for the chunk (Qs, Ks: pitch DK + 4), then masked (s <= t < n),
// scaled and decayed: As[t][s] = scale exp(G_t - G_s) (q_t . k_s) (pitch
// BT + 4).  Thread (ti, tj): rows ti + 16 r, columns tj + 16 c.  Ends with a
// barrier.
template <int DK, int AP = BT + 4>
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
            As[t * AP + s] = (s <= t && t < n) ? scale * expf(G[t] - G[s]) * acc[r][c] : 0.f;
        }
    }
    __syncthreads();
}

// acc[r][c] += sum_{x < X} L[(ti + 16 r) * lp + x] R[x * rp + 4 tj + 64 c ..]:
// thread rows ti + 16 r of L (scalars), columns 4 tj + 64 c of R (16-byte).
template <int X, int NC>
__device__ __forceinline__ void rows_times(unsigned long long (&acc)[4][NC][2], const float *L,
                                           int lp, const float *R, int rp, int ti, int tj)
{
#pragma unroll 4
    for (int x = 0; x < X; ++x) {
        ulonglong2 rr[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c)
            rr[c] = *reinterpret_cast<const ulonglong2 *>(R + x * rp + 4 * tj + 64 * c);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float l = L[(ti + 16 * r) * lp + x];
#pragma unroll
            for (int c = 0; c < NC; ++c) fma4p(acc[r][c], l, rr[c]);
        }
    }
}

// Stores the packed accumulator rows t = ti + 16 r < n, columns 4 tj + 64 c.
template <int NC>
__device__ __forceinline__ void store_rows(const unsigned long long (&acc)[4][NC][2], float *o,
                                           long long op, int n, int ti, int tj)
{
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = ti + 16 * r;
        if (t >= n) continue;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float2 a = unpack2(acc[r][c][0]), b = unpack2(acc[r][c][1]);
            *reinterpret_cast<float4 *>(o + t * op + 4 * tj + 64 * c) =
                make_float4(a.x, a.y, b.x, b.y);
        }
    }
}

// The output pass, grid (NT, BH), two CTAs per multiprocessor: one chunk of
// one head.  Q and K are staged; A = Q K^T is masked, scaled and decayed
// into As; then one buffer holds in turn V and the two 64-row halves of the
// chunk's state h_c (DK = 128; one half for DK = 64), and one accumulator
// takes A V and then (scale exp(G_t) q_t) h_c -- the Q rows rescaled in place
// once A is formed.
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2) la_output_kernel(const Args p)
{
    constexpr int QP = DK + 4, BP = (DK > DV ? DK : DV) + 4, AP = BT + 1;
    constexpr int NC = DV / 64;
    extern __shared__ float4 smem4[];
    float *Qs = reinterpret_cast<float *>(smem4);  // BT x QP
    float *Bs = Qs + BT * QP;                      // BT x BP: K, then V, then h_c halves
    float *As = Bs + BT * BP;                      // BT x AP
    float *G = As + BT * AP;                       // BT
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    const int c = blockIdx.x;
    const long long head = blockIdx.y;
    const int t0 = c * BT, n = min(BT, p.T - t0);
    stage_rows_async<DK>(Qs, QP, p.q + (head * p.T + t0) * DK, DK, n, tid);
    stage_rows_async<DK>(Bs, DK + 4, p.k + (head * p.T + t0) * DK, DK, n, tid);
    cp_commit();
    // V and the chunk's state are staged only after A is formed: ask L2 for
    // their lines now, so that those copies wait on L2 rather than DRAM
    {
        const float *vv = p.v + (head * p.T + t0) * DV;
        const float *hh = p.h + (head * p.NT + c) * DK * DV;
        for (int i = tid; i < n * DV / 32; i += kThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(vv + 32 * i));
        for (int i = tid; i < DK * DV / 32; i += kThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(hh + 32 * i));
    }
    chunk_decay(p.g != nullptr ? p.g + head * p.T + t0 : nullptr, n, G, tid);
    cp_wait<0>();
    __syncthreads();
    attention_tile<DK, AP>(Qs, Bs, G, n, p.scale, As, ti, tj);  // ends with a barrier
    stage_rows_async<DV>(Bs, BP, p.v + (head * p.T + t0) * DV, DV, n, tid);
    cp_commit();
    // Q rows times scale exp(G_t), for the earlier chunks' term
    for (int i = tid; i < BT * (DK / 4); i += kThreads) {
        const int t = i / (DK / 4), k = (i - t * (DK / 4)) * 4;
        const float e = p.scale * expf(G[t]);
        float4 *x = reinterpret_cast<float4 *>(Qs + t * QP + k);
        float4 y = *x;
        y.x *= e;
        y.y *= e;
        y.z *= e;
        y.w *= e;
        *x = y;
    }
    cp_wait<0>();
    __syncthreads();
    unsigned long long acc[4][NC][2] = {};
    rows_times<BT, NC>(acc, As, AP, Bs, BP, ti, tj);
    const float *hc = p.h + (head * p.NT + c) * DK * DV;
#pragma unroll 1
    for (int half = 0; half < DK / 64; ++half) {
        __syncthreads();  // every thread is done with Bs
        stage_rows_async<DV>(Bs, BP, hc + half * 64 * DV, DV, 64, tid);
        cp_commit();
        cp_wait<0>();
        __syncthreads();
        rows_times<64, NC>(acc, Qs + half * 64, QP, Bs, BP, ti, tj);
    }
    store_rows<NC>(acc, p.o + (head * p.T + t0) * DV, DV, n, ti, tj);
}

// ---------------------------------------------------------------- fused pass

// Warp 0: the chunk's running decay G (the output's mask and the earlier
// chunks' factor) and the state update's weights W (update_weights), from
// the chunk's log-decays held in registers.
__device__ __forceinline__ void chunk_decays(float a, float b, int n, float *G, float *W, int l)
{
    float s = a + b;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, off);
        if (l >= off) s += y;
    }
    G[2 * l] = s - b;
    G[2 * l + 1] = s;
    const int src = (n - 1) >> 1;
    const float hi = __shfl_sync(0xffffffffu, s, src);
    const float bb = __shfl_sync(0xffffffffu, b, src);
    const float glast = ((n - 1) & 1) ? hi : hi - bb;
    W[2 * l] = 2 * l < n ? expf(glast - (s - b)) : 0.f;
    W[2 * l + 1] = 2 * l + 1 < n ? expf(glast - s) : 0.f;
    if (l == 0) W[BT] = expf(glast);
}

// The fused pass, grid (DV / 64, BH), one CTA per multiprocessor: a 64-column
// slice of one head's state stays in the CTA (registers for the update, a
// shared copy for Q S) while the CTA walks the chunks; the next chunk's Q, K
// and V are in flight (cp.async, two buffers) while this one is computed,
// and warp 0 holds the next chunk's log-decays.  Per chunk: A = Q K^T
// masked, scaled and decayed; O = A V + (scale exp(G_t) q_t) S (one
// accumulator, the Q rows rescaled in place once A is formed); then
// S = exp(G_last) S + sum_s exp(G_last - G_s) k_s^T v_s.
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) la_fused_kernel(const Args p)
{
    constexpr int QP = DK + 4, VP = BV + 4, AP = BT + 1;
    extern __shared__ float4 smem4[];
    float *Qb = reinterpret_cast<float *>(smem4);  // 2 x BT x QP
    float *Kb = Qb + 2 * BT * QP;                  // 2 x BT x QP
    float *Vb = Kb + 2 * BT * QP;                  // 2 x BT x VP
    float *As = Vb + 2 * BT * VP;                  // BT x AP
    float *Ss = As + BT * AP;                      // DK x VP: the state before the chunk
    float *G = Ss + DK * VP;                       // BT
    float *W = G + BT;                             // BT + 1
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    const int v0 = blockIdx.x * BV;
    const long long head = blockIdx.y;
    StateRegs<DK> S;
    state_load<DK>(S, p.h0 != nullptr ? p.h0 + head * DK * DV : nullptr, DV, v0, ti, tj);
    auto issue = [&](int c) {
        if (c < p.NT) {
            const int t0 = c * BT, n = min(BT, p.T - t0), buf = c & 1;
            stage_rows_async<DK>(Qb + buf * BT * QP, QP, p.q + (head * p.T + t0) * DK, DK, n, tid);
            stage_rows_async<DK>(Kb + buf * BT * QP, QP, p.k + (head * p.T + t0) * DK, DK, n, tid);
            stage_rows_async<BV>(Vb + buf * BT * VP, VP, p.v + (head * p.T + t0) * DV + v0, DV, n,
                                 tid);
        }
        cp_commit();
    };
    issue(0);
    float ga = 0.f, gb = 0.f;
    if (tid < 32) load_decay_pair(p, head, 0, tid, ga, gb);
    for (int c = 0; c < p.NT; ++c) {
        const int t0 = c * BT, n = min(BT, p.T - t0), buf = c & 1;
        float *Qs = Qb + buf * BT * QP;
        const float *Ks = Kb + buf * BT * QP;
        float *Vs = Vb + buf * BT * VP;
        issue(c + 1);
        float na = 0.f, nb = 0.f;
        if (tid < 32) {
            load_decay_pair(p, head, c + 1, tid, na, nb);
            chunk_decays(ga, gb, n, G, W, tid);
        }
        state_store<DK>(S, Ss, VP, 0, ti, tj);
        cp_wait<1>();
        __syncthreads();
        attention_tile<DK, AP>(Qs, Ks, G, n, p.scale, As, ti, tj);  // ends with a barrier
        for (int i = tid; i < BT * (DK / 4); i += kThreads) {
            const int t = i / (DK / 4), k = (i - t * (DK / 4)) * 4;
            const float e = p.scale * expf(G[t]);
            float4 *x = reinterpret_cast<float4 *>(Qs + t * QP + k);
            float4 y = *x;
            y.x *= e;
            y.y *= e;
            y.z *= e;
            y.w *= e;
            *x = y;
        }
        __syncthreads();
        unsigned long long acc[4][1][2] = {};
        rows_times<BT, 1>(acc, As, AP, Vs, VP, ti, tj);
        rows_times<DK, 1>(acc, Qs, QP, Ss, VP, ti, tj);
        store_rows<1>(acc, p.o + (head * p.T + t0) * DV + v0, DV, n, ti, tj);
        __syncthreads();  // V is read as V above; the update reads it weighted
        for (int i = tid; i < BT * (BV / 4); i += kThreads) {
            const int s2 = i / (BV / 4), cc = (i - s2 * (BV / 4)) * 4;
            const float w = W[s2];
            float4 *x = reinterpret_cast<float4 *>(Vs + s2 * VP + cc);
            float4 y = *x;
            y.x *= w;
            y.y *= w;
            y.z *= w;
            y.w *= w;
            *x = y;
        }
        __syncthreads();
        state_update<DK>(S, W[BT], Ks, Vs, ti, tj);
        ga = na;
        gb = nb;
        __syncthreads();  // the next issue reuses this chunk's buffers; G, W, Ss
    }
    cp_wait<0>();
    if (p.state_out != nullptr)
        state_store<DK>(S, p.state_out + head * DK * DV, DV, v0, ti, tj);
}

template <int DK, int DV>
constexpr size_t state_smem()
{
    return sizeof(float) * (2 * kStateBufs * BT * 68 + BT + 4);
}
template <int DK, int DV>
constexpr size_t output_smem()
{
    return sizeof(float) * (BT * (DK + 4) + BT * ((DK > DV ? DK : DV) + 4) + BT * (BT + 1) + BT);
}
template <int DK, int DV>
constexpr size_t fused_smem()
{
    return sizeof(float) *
           (4 * BT * (DK + 4) + 2 * BT * (BV + 4) + BT * (BT + 1) + DK * (BV + 4) + 2 * BT + 4);
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
        grid = dim3(DV / 64, DK / 64, static_cast<unsigned>(BH));
    } else if (w == kOutput) {
        kern = la_output_kernel<DK, DV>;
        smem = output_smem<DK, DV>();
        grid = dim3(static_cast<unsigned>(a.NT), static_cast<unsigned>(BH));
    } else {
        kern = la_fused_kernel<DK, DV>;
        smem = fused_smem<DK, DV>();
        grid = dim3(DV / BV, static_cast<unsigned>(BH));
    }
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return SGEMM_OK;
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
