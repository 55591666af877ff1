"""The allocation-free split-K entry point, sgemm_batched_ex_noalloc.

It serves callers that may not allocate device memory where they multiply
(a host callback, another library's critical section, a plugin handed only
its buffers): its split-K scratch is a fixed array inside the library.  These
tests call it through the C ABI and check, on two calls in a row (the second
one reuses the scratch the first one left behind), that its output agrees
with the ordinary entry point's within the accuracy bound of every path.
The file is named to be collected last."""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem

pytestmark = pytest.mark.gpu

SHAPES = [(1024, 1024, 1024, 1.0, 0.0), (600, 700, 777, 1.0, -2.0), (256, 256, 600, 1.5, 0.5)]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()


@pytest.mark.parametrize("mode", ["fp32", "3xtf32", "tf32"])
@pytest.mark.parametrize("shape", SHAPES)
def test_noalloc_matches_the_existing_entry_point_twice(oracle_mod, mode, shape):
    import dense_fp32_matrix_03_gb300 as lib
    M, N, K, alpha, beta = shape
    assert lib.sgemm_workspace_size(mode, M, N, K, 1) > 0, "the shape should use split-K"
    A, B, C0 = workloads.random_inputs(M, N, K, seed=M + K)
    prob = Problem(A, B, C0, alpha, beta)
    C_plain = prob.run_gpu(mode)                  # sgemm_batched_ex: no split, no scratch
    _, D = prob.oracle(oracle_mod)                # magnitudes for the accuracy metric
    for _ in range(2):
        C = prob.run_gpu(mode, api="noalloc")
        err = float(np.max(np.abs(C.astype(np.float64) - C_plain) / (D + 1e-30)))
        assert err <= TOL[mode], f"{mode} {shape}: {err:.3e}"


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
