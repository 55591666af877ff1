/*
 * linear_attention.h -- chunked linear attention with a decay, fp32, on one
 * GB300 (part of libsgemm_gb300.so; status codes as in sgemm.h).
 *
 * The operation ("From 1% to 94% of cuBLAS, one kernel at a time", section
 * "What FLA builds on top of this"): for every head b (0 <= b < BH),
 * independently, a recurrence over the tokens t = 0 .. T-1 with a K x V
 * state S (K = DK, V = DV):
 *
 *     S_t = exp(g_t) S_{t-1} + k_t^T v_t        (S_{-1} = h0, zero when NULL)
 *     o_t = scale * q_t S_t
 *
 * g_t is the token's log-decay (exp(g_t) the factor the state keeps; g NULL
 * means no decay, g = 0).  The library computes it in chunks of BT = 64
 * tokens, the chunked form of the same section: h_c, the state before chunk
 * c (c = 0 .. NT-1, NT = ceil(T / 64)), passes between chunks, and inside a
 * chunk, with G_t the running sum of g over the chunk up to t,
 *
 *     o_t     = scale (exp(G_t) q_t h_c + sum_{s <= t in the chunk} exp(G_t - G_s) (q_t . k_s) v_s)
 *     h_{c+1} = exp(G_last) h_c + sum_{s in the chunk} exp(G_last - G_s) k_s^T v_s
 *
 * ("Why FLA sits somewhere else on the roofline": the state pass is a scan
 * over the chunks; materialising h lets the output pass run every chunk in
 * parallel; the fused pass trades that traffic for a longer serial chain.)
 *
 * Layout (row-major, contiguous, fp32, DEVICE pointers owned by the caller):
 *   q, k   BH x T x DK        v, o   BH x T x DV        g   BH x T
 *   h0, state_out   BH x DK x DV        h   BH x NT x DK x DV (h[b][c] = h_c)
 * DK and DV are 64 or 128; T >= 0 (a last chunk shorter than 64 is fine);
 * BH <= 65535.  q, k, v, o, h, h0 and state_out must be 16-byte aligned, g
 * 4-byte aligned.  g, h0 and state_out may be NULL.  Every call returns once
 * its kernel is enqueued on `stream`; nothing is allocated or synchronised.
 * Arithmetic: fp32 products and sums (FMA), exp by the CUDA expf; the
 * accuracy against the exact result is bounded relative to the sum of the
 * absolute values of the terms, like the SGEMM FP32 path.
 *
 * Errors: SGEMM_ERR_INVALID_ARG (dimensions, NULL where data is read or
 * written, misaligned pointers) before anything is launched;
 * SGEMM_ERR_UNSUPPORTED without a compute capability 10.3 GPU;
 * SGEMM_ERR_LAUNCH if the launch fails.  BH == 0 is a no-op; T == 0 writes
 * state_out = h0 (or zeros) where asked.
 */
#ifndef LINEAR_ATTENTION_GB300_H
#define LINEAR_ATTENTION_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of the chunk-state buffer h: BH * NT * DK * DV floats (0 for
 * invalid dimensions). */
size_t la_state_bytes(int BH, int T, int DK, int DV);

/* The state pass: writes h[b][c] = h_c for every chunk (and S_{T-1} to
 * state_out when not NULL).  Sequential in the chunks; parallel over heads
 * and 64-column slices of the state. */
int la_chunk_state(int BH, int T, int DK, int DV, const float *k, const float *v,
                   const float *g, const float *h0, float *h, float *state_out, void *stream);

/* The output pass: o for every token, from q, k, v, g and the states h the
 * state pass wrote (enqueue it after la_chunk_state on the same stream, or
 * order the two).  Parallel over heads and chunks. */
int la_chunk_output(int BH, int T, int DK, int DV, float scale, const float *q, const float *k,
                    const float *v, const float *g, const float *h, float *o, void *stream);

/* Both passes in one kernel: o (and state_out when not NULL) without
 * writing h.  Sequential in the chunks; parallel over heads and 64-column
 * slices of the state. */
int la_chunk_fused(int BH, int T, int DK, int DV, float scale, const float *q, const float *k,
                   const float *v, const float *g, const float *h0, float *o, float *state_out,
                   void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LINEAR_ATTENTION_GB300_H */
