"""Pins for the CPU oracle (oracle/oracle_sgemm.c), checked against facts that
do not come from the oracle itself.

The definition pinned is the SGEMM of "From 1% to 94% of cuBLAS, one kernel at
a time" (section "Napkin math for 4092 x 4092" and the first kernel):
C = alpha * A @ B + beta * C, row-major, plus transposed operands and a batch
index ("Triton Optimization Reference (cuTile -> Triton)", sections 2-3).

Each pin is chosen so that a plausible slip in the oracle fails it:
  * exact rational brute force on every tiny shape (any wrong index, sign,
    dropped term or swapped operand),
  * identity / permutation / rank-1 / all-ones closed forms,
  * integer-valued inputs against exact integer matmul,
  * the BLAS readings of beta == 0, alpha == 0 and K == 0,
  * storage equivalences for transposes, leading dimensions and batches,
  * the error-metric magnitude D.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def store(logical, trans, ld=None):
    """Store a logical R x Cc matrix row-major (or its transpose when trans),
    with leading dimension ld >= stored row length.  Returns (flat, ld)."""
    mat = logical.T if trans else logical
    rows, cols = mat.shape
    ld = cols if ld is None else ld
    buf = np.full(max(rows * ld, 1), np.float32(7.5), dtype=np.float32)  # junk padding
    for r in range(rows):
        buf[r * ld:r * ld + cols] = mat[r]
    return buf, ld


def exact_gemm(A, B, C0, alpha, beta):
    """Exact rational alpha*A@B + beta*C0 and sum |alpha*a*b| + |beta*c|."""
    M, K = A.shape
    N = B.shape[1]
    al, be = Fraction(float(alpha)), Fraction(float(beta))
    out = [[None] * N for _ in range(M)]
    mag = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            m = Fraction(0)
            for k in range(K):
                p = Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                s += p
                m += abs(p)
            c = be * Fraction(float(C0[i, j])) if beta != 0 else Fraction(0)
            if alpha == 0 or K == 0:
                out[i][j], mag[i][j] = c, abs(c)
            else:
                out[i][j], mag[i][j] = al * s + c, abs(al) * m + abs(c)
    return out, mag


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_brute_force_tiny_shapes_exact_rational(oracle_mod, transA, transB):
    rng = np.random.default_rng(100 + 2 * transA + transB)
    for M, N, K in itertools.product(range(1, 6), repeat=3):
        A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
        B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
        C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
        alpha, beta = np.float32(rng.choice([1.5, -0.75, 3.0])), np.float32(
            rng.choice([0.0, 0.5, -2.0]))
        extra = int(rng.integers(0, 3))
        Ab, lda = store(A, transA, (M if transA else K) + extra)
        Bb, ldb = store(B, transB, (K if transB else N) + extra)
        Cb, ldc = store(C0, 0, N + extra)
        Cref, D = oracle_mod.sgemm_ref(M, N, K, alpha, Ab, lda, Bb, ldb, beta, Cb, ldc,
                                       transA=transA, transB=transB)
        ex, mg = exact_gemm(A, B, C0, alpha, beta)
        for i in range(M):
            for j in range(N):
                # fp64 sum of <= 5 exact products: relative error far below 1e-14
                assert abs(Fraction(Cref[i, j]) - ex[i][j]) <= Fraction(1, 10**14) * (
                    mg[i][j] + Fraction(1, 10**30)), (M, N, K, i, j)
                assert abs(Fraction(D[i, j]) - mg[i][j]) <= Fraction(1, 10**14) * mg[i][j]


def test_identity_gives_alpha_b_plus_beta_c(oracle_mod):
    K = N = 37
    rng = np.random.default_rng(1)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    I = np.eye(K, dtype=np.float32)
    for alpha, beta in [(2.0, 0.5), (-4.0, 0.25), (1.0, 0.0), (0.5, -1.0)]:
        Cref, _ = oracle_mod.sgemm_ref(K, N, K, alpha, I, K, B, N, beta, C0, N)
        want = alpha * B.astype(np.float64) + beta * C0.astype(np.float64)
        assert np.array_equal(Cref, want)  # powers of two: exact


def test_permutation_is_bit_exact_row_and_column_shuffle(oracle_mod):
    rng = np.random.default_rng(2)
    M = K = 23
    N = 31
    perm = rng.permutation(M)
    P = np.zeros((M, K), dtype=np.float32)
    P[np.arange(M), perm] = 1.0
    B = rng.normal(size=(K, N)).astype(np.float32)
    Cref, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, P, K, B, N, 0.0, None, N)
    assert np.array_equal(Cref, B[perm].astype(np.float64))
    # permutation on the right shuffles columns
    A = rng.normal(size=(M, N)).astype(np.float32)
    Q = np.zeros((N, N), dtype=np.float32)
    cperm = rng.permutation(N)
    Q[cperm, np.arange(N)] = 1.0
    Cref, _ = oracle_mod.sgemm_ref(M, N, N, 1.0, A, N, Q, N, 0.0, None, N)
    assert np.array_equal(Cref, A[:, cperm].astype(np.float64))


def test_rank1_k_equals_one(oracle_mod):
    rng = np.random.default_rng(3)
    M, N = 19, 13
    a = rng.uniform(-1, 1, (M, 1)).astype(np.float32)
    b = rng.uniform(-1, 1, (1, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    Cref, D = oracle_mod.sgemm_ref(M, N, 1, 1.5, a, 1, b, N, 0.5, C0, N)
    prod = a.astype(np.float64) * b.astype(np.float64)  # exact in fp64
    assert np.array_equal(Cref, 1.5 * prod + 0.5 * C0.astype(np.float64))
    assert np.array_equal(D, 1.5 * np.abs(prod) + np.abs(0.5 * C0.astype(np.float64)))


def test_outer_product_structure_closed_form(oracle_mod):
    # A = u 1^T, B = 1 v^T  =>  S = K u_i v_j
    rng = np.random.default_rng(4)
    M, N, K = 11, 17, 29
    u = rng.integers(-9, 10, M).astype(np.float32)
    v = rng.integers(-9, 10, N).astype(np.float32)
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    Cref, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert np.array_equal(Cref, K * np.outer(u, v).astype(np.float64))
    ones_a = np.ones((M, K), np.float32)
    ones_b = np.ones((K, N), np.float32)
    Cref, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, ones_a, K, ones_b, N, 0.0, None, N)
    assert np.all(Cref == K)


def test_integer_inputs_match_exact_integer_matmul(oracle_mod):
    from workloads import integer_inputs
    for (M, N, K, alpha, beta) in [(64, 48, 333, 1.0, 0.0), (40, 70, 128, 2.0, -2.0),
                                   (33, 33, 1000, 1.0, 1.0)]:
        A, B, C0 = integer_inputs(M, N, K, seed=M + N)
        want = alpha * (A.astype(np.int64) @ B.astype(np.int64)) + beta * C0.astype(np.int64)
        Cref, _ = oracle_mod.sgemm_ref(M, N, K, alpha, A, K, B, N, beta, C0, N)
        assert np.array_equal(Cref, want.astype(np.float64))


def test_beta_zero_does_not_read_c(oracle_mod):
    rng = np.random.default_rng(5)
    A = rng.uniform(-1, 1, (8, 5)).astype(np.float32)
    B = rng.uniform(-1, 1, (5, 6)).astype(np.float32)
    C0 = np.full((8, 6), np.nan, np.float32)
    C0[0, 0] = np.inf
    Cref, D = oracle_mod.sgemm_ref(8, 6, 5, 1.0, A, 5, B, 6, 0.0, C0, 6)
    assert np.all(np.isfinite(Cref)) and np.all(np.isfinite(D))


def test_alpha_zero_and_k_zero_give_beta_c(oracle_mod):
    rng = np.random.default_rng(6)
    C0 = rng.uniform(-1, 1, (7, 9)).astype(np.float32)
    A = np.full((7, 4), np.inf, np.float32)  # never read when alpha == 0
    B = np.full((4, 9), np.nan, np.float32)
    Cref, D = oracle_mod.sgemm_ref(7, 9, 4, 0.0, A, 4, B, 9, -2.0, C0, 9)
    assert np.array_equal(Cref, -2.0 * C0.astype(np.float64))
    assert np.array_equal(D, np.abs(-2.0 * C0.astype(np.float64)))
    Cref, _ = oracle_mod.sgemm_ref(7, 9, 0, 1.0, A, 1, B, 9, 0.5, C0, 9)
    assert np.array_equal(Cref, 0.5 * C0.astype(np.float64))
    Cref, _ = oracle_mod.sgemm_ref(7, 9, 0, 1.0, A, 1, B, 9, 0.0, None, 9)
    assert np.all(Cref == 0)


def test_transposed_storage_equals_plain_storage(oracle_mod):
    rng = np.random.default_rng(7)
    M, N, K = 45, 38, 51
    A = rng.normal(size=(M, K)).astype(np.float32)
    B = rng.normal(size=(K, N)).astype(np.float32)
    C0 = rng.normal(size=(M, N)).astype(np.float32)
    base, _ = oracle_mod.sgemm_ref(M, N, K, 0.75, A, K, B, N, 0.25, C0, N)
    for tA, tB in [(1, 0), (0, 1), (1, 1)]:
        Ab, lda = store(A, tA)
        Bb, ldb = store(B, tB)
        got, _ = oracle_mod.sgemm_ref(M, N, K, 0.75, Ab, lda, Bb, ldb, 0.25, C0, N,
                                      transA=tA, transB=tB)
        # same k order either way: identical bits
        assert np.array_equal(got, base)
    # and the transpose is a real transpose, not the same storage read twice
    if M != K:
        with pytest.raises(ValueError):
            oracle_mod.sgemm_ref(M, N, K, 1.0, A[:, :M].copy(), M, B, N, 0.0, None, N,
                                 transA=1)


def test_leading_dimension_padding_matches_packed(oracle_mod):
    rng = np.random.default_rng(8)
    M, N, K = 21, 17, 25
    A = rng.normal(size=(M, K)).astype(np.float32)
    B = rng.normal(size=(K, N)).astype(np.float32)
    C0 = rng.normal(size=(M, N)).astype(np.float32)
    packed, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, A, K, B, N, 1.0, C0, N)
    Ab, lda = store(A, 0, K + 7)
    Bb, ldb = store(B, 0, N + 3)
    Cb, ldc = store(C0, 0, N + 11)
    padded, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, Ab, lda, Bb, ldb, 1.0, Cb, ldc)
    assert np.array_equal(padded, packed)


def test_batched_equals_single_calls_and_broadcast(oracle_mod):
    rng = np.random.default_rng(9)
    Q, M, N, K = 4, 9, 7, 13
    A = rng.normal(size=(Q, M, K)).astype(np.float32)
    B = rng.normal(size=(Q, K, N)).astype(np.float32)
    C0 = rng.normal(size=(Q, M, N)).astype(np.float32)
    got, _ = oracle_mod.sgemm_ref(M, N, K, 0.5, A, K, B, N, 2.0, C0, N, strideA=M * K,
                                  strideB=K * N, strideC=M * N, Q=Q)
    for q in range(Q):
        one, _ = oracle_mod.sgemm_ref(M, N, K, 0.5, A[q], K, B[q], N, 2.0, C0[q], N)
        assert np.array_equal(got[q], one)
    # strideA = 0 broadcasts A[0] over the batch
    got, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, A[0], K, B, N, 0.0, None, N, strideA=0,
                                  strideB=K * N, strideC=M * N, Q=Q)
    for q in range(Q):
        one, _ = oracle_mod.sgemm_ref(M, N, K, 1.0, A[0], K, B[q], N, 0.0, None, N)
        assert np.array_equal(got[q], one)


def test_row_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(10)
    Q, M, N, K = 3, 12, 10, 8
    A = rng.normal(size=(Q, M, K)).astype(np.float32)
    B = rng.normal(size=(Q, N, K)).astype(np.float32)  # stored transposed
    full, fullD = oracle_mod.sgemm_ref(M, N, K, 1.0, A, K, B, K, 0.0, None, N, transB=1,
                                       strideA=M * K, strideB=N * K, strideC=M * N, Q=Q)
    rows = [(2, 11), (0, 0), (1, 5), (2, 3)]
    sub, subD = oracle_mod.sgemm_ref(M, N, K, 1.0, A, K, B, K, 0.0, None, N, transB=1,
                                     strideA=M * K, strideB=N * K, strideC=M * N, Q=Q,
                                     rows=rows)
    for r, (q, i) in enumerate(rows):
        assert np.array_equal(sub[r], full[q, i])
        assert np.array_equal(subD[r], fullD[q, i])


def test_error_magnitude_sign_invariance(oracle_mod):
    rng = np.random.default_rng(11)
    M, N, K = 16, 16, 40
    A = np.abs(rng.normal(size=(M, K))).astype(np.float32)
    B = np.abs(rng.normal(size=(K, N))).astype(np.float32)
    Cp, Dp = oracle_mod.sgemm_ref(M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert np.array_equal(Cp, Dp)  # non-negative terms: |sum| == sum of |.|
    Cn, Dn = oracle_mod.sgemm_ref(M, N, K, 1.0, -A, K, B, N, 0.0, None, N)
    assert np.array_equal(Cn, -Cp) and np.array_equal(Dn, Dp)
    # mixed signs: |C_ref| <= D everywhere
    A2 = rng.normal(size=(M, K)).astype(np.float32)
    C2, D2 = oracle_mod.sgemm_ref(M, N, K, -3.0, A2, K, B, N, 0.0, None, N)
    assert np.all(np.abs(C2) <= D2 * (1 + 1e-15))


def test_error_metric(oracle_mod):
    Cref = np.array([1.0, -2.0, 0.0])
    D = np.array([2.0, 4.0, 0.0])
    assert oracle_mod.max_rel_err(np.array([1.0, -2.0, 0.0]), Cref, D) == 0.0
    assert oracle_mod.max_rel_err(np.array([1.5, -2.0, 0.0]), Cref, D) == 0.25
    assert oracle_mod.max_rel_err(np.array([1.0, np.nan, 0.0]), Cref, D) == np.inf


def test_workload_recipes_are_seeded_and_shaped():
    import workloads
    a = workloads.make("sgemm_256")
    b = workloads.make("sgemm_256")
    assert a["A"].shape == (256, 256) and a["A"].dtype == np.float32
    assert np.array_equal(a["A"], b["A"]) and np.array_equal(a["C0"], b["C0"])
    assert a["A"].min() >= -1 and a["A"].max() <= 1
    r = workloads.make("sgemm_ragged_1000x1500x777")
    assert r["A"].shape == (1000, 777) and r["B"].shape == (777, 1500)
    s = workloads.make("sweep_128")
    assert np.all(s["C0"] == 0)
    bm = workloads.config("bmm_q32_1024x1024x512")
    assert (bm["Q"], bm["M"], bm["N"], bm["K"]) == (32, 1024, 1024, 512)
