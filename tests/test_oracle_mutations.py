"""Plant mistakes in a copy of the oracle's C source (on the CPU) and check that
the pins catch each one.  The oracle itself is never modified: each mutant is
compiled from a rewritten temporary copy."""
import os

import numpy as np
import pytest

from test_oracle_pins import exact_gemm, store
from fractions import Fraction

MUTATIONS = {
    "drop_beta_term": ("c = beta * (double)C0row[j];", "c = 0.0;"),
    "wrong_sign": ("acc[j] += p;", "acc[j] -= p;"),
    "transB_index_swapped": ("B[j * ldb + k]", "B[k * ldb + j]"),
    "A_index_transposed": ("(double)A[i * lda + k]", "(double)A[k * lda + i]"),
    "magnitude_without_abs": ("mag[j] += fabs(p);", "mag[j] += p;"),
    "k_loop_skips_first": ("for (k = 0; k < K; ++k) {", "for (k = 1; k < K; ++k) {"),
    "alpha_applied_twice": ("Cref_row[j] = alpha * acc[j] + c;",
                            "Cref_row[j] = alpha * alpha * acc[j] + c;"),
    "batch_stride_ignored": ("B + q * strideB, ldb", "B, ldb"),
}


def pins_pass(oracle_mod, lib) -> bool:
    """A compact battery of the pins: exact rational brute force over small
    shapes, all transpose flags, a batch and a non-trivial alpha/beta."""
    rng = np.random.default_rng(77)
    for (M, N, K) in [(3, 4, 5), (5, 2, 3), (4, 4, 1), (2, 5, 6)]:
        for tA in (0, 1):
            for tB in (0, 1):
                Q = 2
                A = rng.uniform(-1, 1, (Q, M, K)).astype(np.float32)
                B = rng.uniform(-1, 1, (Q, K, N)).astype(np.float32)
                C0 = rng.uniform(-1, 1, (Q, M, N)).astype(np.float32)
                alpha, beta = np.float32(-1.5), np.float32(0.5)
                Ab = np.concatenate([store(A[q], tA)[0] for q in range(Q)])
                Bb = np.concatenate([store(B[q], tB)[0] for q in range(Q)])
                lda = M if tA else K
                ldb = K if tB else N
                Cref, D = oracle_mod.sgemm_ref(M, N, K, alpha, Ab, lda, Bb, ldb, beta, C0, N,
                                               transA=tA, transB=tB, strideA=M * K,
                                               strideB=K * N, strideC=M * N, Q=Q, lib=lib)
                for q in range(Q):
                    ex, mg = exact_gemm(A[q], B[q], C0[q], alpha, beta)
                    for i in range(M):
                        for j in range(N):
                            tol = Fraction(1, 10**14) * (mg[i][j] + Fraction(1, 10**30))
                            if abs(Fraction(Cref[q, i, j]) - ex[i][j]) > tol:
                                return False
                            if abs(Fraction(D[q, i, j]) - mg[i][j]) > tol:
                                return False
    return True


def test_unmutated_oracle_passes_the_battery(oracle_mod):
    assert pins_pass(oracle_mod, None)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "oracle_sgemm.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle_mod.load(oracle_mod.build(force=True, src=str(mutant),
                                           out=str(tmp_path / "libmutant.so")))
    assert not pins_pass(oracle_mod, lib), f"mutation {name} slipped through the pins"
