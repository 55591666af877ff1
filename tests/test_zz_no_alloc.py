"""The allocation-free split-K entry point, sgemm_batched_ex_noalloc.

It serves callers that may not allocate device memory where they multiply
(a host callback, another library's critical section, a plugin handed only
its buffers): its split-K scratch is a fixed array inside the library.  These
tests call it through the C ABI, twice in a row (the second call reuses the
scratch the first one left behind), and check each result against the fp64
oracle within the accuracy bound of the path, and that the call really took
the split route (its plan split, and the product kernel and the split-K
fix-up both launched).
The file is named to be collected last."""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem

pytestmark = pytest.mark.gpu

# Shapes whose grids are small enough for this entry point's one-wave split
# on every path and whose K is long enough for the split to pay (so the
# library's planner takes it), with ragged edges in the second one; every
# operand is TMA-describable, so no operand copy takes the scratch first.
SHAPES = [(1000, 1000, 4096, 1.0, 0.0), (600, 700, 3000, 1.0, -2.0),
          (256, 256, 2048, 1.5, 0.5)]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()


@pytest.mark.parametrize("mode", ["fp32", "3xtf32", "tf32"])
@pytest.mark.parametrize("shape", SHAPES)
def test_noalloc_matches_the_oracle_twice(oracle_mod, mode, shape):
    import dense_fp32_matrix_03_gb300 as lib
    M, N, K, alpha, beta = shape
    A, B, C0 = workloads.random_inputs(M, N, K, seed=M + K)
    prob = Problem(A, B, C0, alpha, beta)
    Cref, D = prob.oracle(oracle_mod)
    C_plain = prob.run_gpu(mode)  # sgemm_batched_ex: the ordinary entry point
    assert oracle_mod.max_rel_err(C_plain, Cref, D) <= TOL[mode]
    for _ in range(2):
        before = lib.sgemm_kernel_launches()
        C = prob.run_gpu(mode, api="noalloc")
        launched = lib.sgemm_kernel_launches() - before
        err = oracle_mod.max_rel_err(C, Cref, D)
        assert err <= TOL[mode], f"{mode} {shape[:3]}: {err:.3e}"
        assert lib.sgemm_last_split_count() > 1, "expected a split plan"
        assert launched == 2, "expected the product kernel and the split-K fix-up"


def test_noalloc_unsplit_shape_and_bad_arguments():
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    a = torch.ones(64, 64, device="cuda")
    c = torch.zeros(64, 64, device="cuda")
    # 64^3 does not split: runs like the ordinary entry point
    assert lib.sgemm_batched_ex_noalloc("fp32", 64, 64, 64, 1.0, a, 64, a, 64, 0.0, c, 64, 0, 0,
                                        0, 0, 0, 1) == lib.SGEMM_OK
    torch.cuda.synchronize()
    assert torch.all(c == 64.0)
    assert lib.sgemm_batched_ex_noalloc("fp32", 64, 64, 64, 1.0, a, 63, a, 64, 0.0, c, 64, 0, 0,
                                        0, 0, 0, 1) == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_status_string(lib.SGEMM_ERR_SCRATCH_LIMIT) != "unknown status"
