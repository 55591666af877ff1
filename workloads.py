"""Seeded synthetic inputs for the SGEMM workloads.

This module is shared by the tests, the benchmark and the oracle's callers.  It
holds no GEMM arithmetic: it only draws the input matrices and records the
shapes, seeds, distributions and alpha/beta of each workload.

The workloads follow the single-precision GEMM benchmark of "From 1% to 94% of
cuBLAS, one kernel at a time" (arpit2412.github.io, section "Napkin math for
4092 x 4092": C = alpha*A@B + beta*C, A M x K, B K x N, row-major), widened to
the ragged, swept and batched shapes the library is tested on.

Drawing recipe (the same on every machine, numpy PCG64):
  rng = numpy.random.default_rng(seed)
  A (M x K), then the logical B (K x N), then C0 (M x N), each drawn in C order
  as float64 and rounded to float32.  A batched workload draws all Q copies of
  A at once (shape Q x M x K), then B (Q x K x N), then C0 (Q x M x N).
  "uniform" is rng.uniform(-1, 1); "normal(s)" is rng.normal(0, s).
  A matrix that a workload fixes to zero is not drawn.
"""
from __future__ import annotations

import numpy as np

# name -> recipe.  dist_* is ("uniform",) or ("normal", sigma) or ("zeros",).
RECIPES = {
    # small reference case
    "sgemm_256": dict(M=256, N=256, K=256, Q=1, seed=0, alpha=1.5, betas=(0.5,),
                      dist_ab=("uniform",), dist_c=("uniform",)),
    # ragged edges: no dimension is a multiple of any tile; lda = 777 is not
    # a multiple of 4 floats
    "sgemm_ragged_1000x1500x777": dict(M=1000, N=1500, K=777, Q=1, seed=1, alpha=1.0,
                                       betas=(0.0, -2.0), dist_ab=("uniform",),
                                       dist_c=("uniform",)),
    # the pages' benchmark shape
    "sgemm_4092": dict(M=4092, N=4092, K=4092, Q=1, seed=2, alpha=1.0, betas=(0.0,),
                       dist_ab=("normal", 1.0), dist_c=("normal", 1.0)),
    # batched: B stored both as N x K (transB=1) and K x N (transB=0)
    "bmm_q32_1024x1024x512": dict(M=1024, N=1024, K=512, Q=32, seed=4, alpha=0.75,
                                  betas=(0.25,), dist_ab=("normal", 0.5),
                                  dist_c=("uniform",)),
}
SWEEP_SIZES = (128, 512, 1024, 2048, 4096, 8192)
SWEEP_SEED = 3


def sweep_config(n: int) -> dict:
    """Square size-sweep workload: A, B uniform[-1,1], C zeros, alpha=1, beta=0.
    A fresh generator seeded with 3 is used for every size."""
    return dict(M=n, N=n, K=n, Q=1, seed=SWEEP_SEED, alpha=1.0, betas=(0.0,),
                dist_ab=("uniform",), dist_c=("zeros",))


def config(name: str) -> dict:
    if name.startswith("sweep_"):
        return sweep_config(int(name.split("_", 1)[1]))
    return dict(RECIPES[name])


def _draw(rng: np.random.Generator, dist: tuple, shape: tuple) -> np.ndarray:
    kind = dist[0]
    if kind == "uniform":
        x = rng.uniform(-1.0, 1.0, size=shape)
    elif kind == "normal":
        x = rng.normal(0.0, float(dist[1]), size=shape)
    elif kind == "zeros":
        return np.zeros(shape, dtype=np.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.astype(np.float32)


def make(name_or_cfg, *, draw_c: bool = True) -> dict:
    """Draw the inputs of a workload.

    Returns a dict with A (Q x M x K or M x K), B (Q x K x N or K x N, the
    logical B), C0 (like C, or None when draw_c is False and C is drawn after
    A and B) plus the recipe fields.  Arrays are C-contiguous float32.
    """
    cfg = config(name_or_cfg) if isinstance(name_or_cfg, str) else dict(name_or_cfg)
    M, N, K, Q = cfg["M"], cfg["N"], cfg["K"], cfg["Q"]
    rng = np.random.default_rng(cfg["seed"])
    lead = (Q,) if Q > 1 else ()
    A = _draw(rng, cfg["dist_ab"], lead + (M, K))
    B = _draw(rng, cfg["dist_ab"], lead + (K, N))
    C0 = _draw(rng, cfg["dist_c"], lead + (M, N)) if draw_c else None
    out = dict(cfg)
    out.update(A=A, B=B, C0=C0)
    return out


def integer_inputs(M: int, N: int, K: int, Q: int = 1, seed: int = 0, lo: int = -8,
                   hi: int = 8):
    """Integer-valued float32 matrices in [lo, hi].  Every product and every
    partial sum of a K <= 4096 contraction is an integer of magnitude below
    2**24, so fp32 arithmetic on them is exact in any order."""
    rng = np.random.default_rng(seed)
    lead = (Q,) if Q > 1 else ()
    A = rng.integers(lo, hi + 1, size=lead + (M, K)).astype(np.float32)
    B = rng.integers(lo, hi + 1, size=lead + (K, N)).astype(np.float32)
    C0 = rng.integers(lo, hi + 1, size=lead + (M, N)).astype(np.float32)
    return A, B, C0


def random_inputs(M: int, N: int, K: int, Q: int = 1, seed: int = 0):
    """Uniform[-1,1] float32 matrices for the ragged parity sweeps."""
    rng = np.random.default_rng(seed)
    lead = (Q,) if Q > 1 else ()
    A = rng.uniform(-1, 1, size=lead + (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=lead + (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, size=lead + (M, N)).astype(np.float32)
    return A, B, C0


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16 (ties to even), returned
    as float32 (exactly representable in bf16).  Input generation for the
    16-bit-input path; NaN/Inf are not expected here."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16 << 16
    return bits.astype(np.uint32).view(np.float32)


def half_bits(x: np.ndarray, type_: str) -> np.ndarray:
    """The 16-bit encodings (uint16) of float32 values already representable
    in `type_` ("bf16": the high half of the fp32 bits; "fp16": IEEE half)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if type_ == "bf16":
        return (x.view(np.uint32) >> 16).astype(np.uint16)
    return x.astype(np.float16).view(np.uint16)


def half_inputs(M: int, N: int, K: int, type_: str, Q: int = 1, seed: int = 0):
    """Uniform[-1,1] matrices rounded to bf16 or fp16 (as float32), and C0."""
    A, B, C0 = random_inputs(M, N, K, Q, seed)
    if type_ == "bf16":
        return round_to_bf16(A), round_to_bf16(B), C0
    return A.astype(np.float16).astype(np.float32), B.astype(np.float16).astype(np.float32), C0


# ------------------------------------------------- chunked linear attention
#
# Inputs of the linear-attention workload (the chunk kernels "From 1% to 94%
# of cuBLAS, one kernel at a time" describes in "Why FLA sits somewhere else
# on the roofline": chunks of BT = 64 tokens, head dimension 128).  Recipe,
# numpy PCG64 with the given seed, each array drawn in C order as float64 and
# rounded to float32, in this order:
#   q, k (BH x T x DK) and v (BH x T x DV): rng.normal(0, 1);
#   g (BH x T), the per-token log-decay: log(sigmoid(x)) / 16 with
#     x = rng.normal(0, 1) -- a decay factor exp(g) between ~0.9 and 1, the
#     range gated linear-attention layers run in (omitted when decay=False);
#   h0 (BH x DK x DV), the initial state: rng.normal(0, 1) (only when
#     with_h0 is set).
# The attention scale is 1 / sqrt(DK).
LA_WORKLOADS = {
    # the benchmark's linear-attention case: batch 4 x 16 heads, 4096 tokens
    "la_b4h16_t4096_d128": dict(BH=64, T=4096, DK=128, DV=128, seed=7),
    # the small case the oracle finishes in seconds
    "la_b2h2_t300_d64": dict(BH=4, T=300, DK=64, DV=64, seed=8),
}


def linattn_inputs(BH: int, T: int, DK: int, DV: int, seed: int = 0, decay: bool = True,
                   with_h0: bool = False):
    """(q, k, v, g, h0, scale) of one linear-attention call (see the recipe
    above); g and h0 are None when not drawn."""
    rng = np.random.default_rng(seed)
    q = rng.normal(0.0, 1.0, size=(BH, T, DK)).astype(np.float32)
    k = rng.normal(0.0, 1.0, size=(BH, T, DK)).astype(np.float32)
    v = rng.normal(0.0, 1.0, size=(BH, T, DV)).astype(np.float32)
    g = None
    if decay:
        x = rng.normal(0.0, 1.0, size=(BH, T))
        g = (-np.logaddexp(0.0, -x) / 16.0).astype(np.float32)  # log(sigmoid(x)) / 16
    h0 = rng.normal(0.0, 1.0, size=(BH, DK, DV)).astype(np.float32) if with_h0 else None
    return q, k, v, g, h0, float(1.0 / np.sqrt(DK))


def la_make(name: str, **kw):
    cfg = dict(LA_WORKLOADS[name])
    return linattn_inputs(cfg["BH"], cfg["T"], cfg["DK"], cfg["DV"], cfg["seed"], **kw)
