"""Every kernel route the tuning table can pick, forced on every mode, against
the oracle: the table changes which kernel runs, never what it computes.

The FP32 path's 64 x 64 tile (route SMALL) and the tensor-core routes (PAIR,
DIRECT, PLANES, RAW, INLINE) each run ragged, transposed, padded, offset and batched
shapes through the workspace entry and the plain one; integer-valued inputs
must match bit for bit."""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem

pytestmark = pytest.mark.gpu

ROUTES = {"fp32": ["small"], "3xtf32": ["pair", "direct", "planes", "raw", "inline"],
          "tf32": ["pair", "direct", "planes", "raw", "inline"]}
CASES = [(128, 128, 128, 1, 0, 0), (257, 130, 300, 1, 1, 0), (64, 320, 1000, 1, 0, 1),
         (500, 600, 777, 1, 1, 1), (96, 200, 64, 3, 0, 1), (1024, 1024, 512, 2, 0, 0)]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()
    yield
    lib.sgemm_tune_force("auto")


@pytest.fixture
def forced():
    import dense_fp32_matrix_03_gb300 as lib

    def force(route):
        assert lib.sgemm_tune_force(route) == lib.SGEMM_OK
    yield force
    lib.sgemm_tune_force("auto")


@pytest.mark.parametrize("api", ["ws", "ex"])
@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("mode,route", [(m, r) for m, rs in ROUTES.items() for r in rs])
def test_forced_route_matches_the_oracle(oracle_mod, forced, mode, route, case, api):
    import dense_fp32_matrix_03_gb300 as lib
    M, N, K, Q, tA, tB = case
    forced(route)
    assert lib.sgemm_tune_route(mode, M, N, K, Q) == lib.ROUTES[route]
    A, B, C0 = workloads.random_inputs(M, N, K, seed=M + N + K, Q=Q)
    prob = Problem(A, B, C0, 1.25, -0.5, transA=tA, transB=tB, pads=(4, 0, 12),
                   offsets=(4, 0, 4))
    C = prob.run_gpu(mode, api=api)
    Cref, D = prob.oracle(oracle_mod)
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode}/{route} {case}: {err:.3e}"


@pytest.mark.parametrize("mode,route", [(m, r) for m, rs in ROUTES.items() for r in rs])
def test_forced_route_integer_inputs_bit_exact(oracle_mod, forced, mode, route):
    forced(route)
    rng = np.random.default_rng(11)
    M, N, K = 300, 260, 1100
    A = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    B = rng.integers(-8, 9, size=(K, N)).astype(np.float32)
    C0 = rng.integers(-8, 9, size=(M, N)).astype(np.float32)
    prob = Problem(A, B, C0, 2.0, -2.0)
    C = prob.run_gpu(mode, api="ws")
    Cref, _ = prob.oracle(oracle_mod)
    assert np.array_equal(C.astype(np.float64), Cref)


def test_route_of_a_mode_that_cannot_take_it_is_auto(forced):
    import dense_fp32_matrix_03_gb300 as lib
    forced("small")
    assert lib.sgemm_tune_route("3xtf32", 128, 128, 128, 1) == lib.SGEMM_ROUTE_AUTO
    forced("planes")
    assert lib.sgemm_tune_route("fp32", 128, 128, 128, 1) == lib.SGEMM_ROUTE_AUTO


def _launches(fn):
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    torch.cuda.synchronize()
    n0 = lib.sgemm_kernel_launches()
    out = fn()
    return out, lib.sgemm_kernel_launches() - n0


@pytest.mark.parametrize("mode", ["3xtf32", "tf32"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 3), (37, 29, 61)])
def test_tiny_call_on_odd_pitches_keeps_the_direct_kernel(oracle_mod, mode, shape):
    """Operands TMA cannot describe (pitches of 4-byte multiples only) on a
    tiny problem, through the workspace entry: the cost models keep the
    direct kernel on the operands as they are -- one launch -- instead of
    copying them for the pair kernel."""
    M, N, K = shape
    A, B, C0 = workloads.random_inputs(M, N, K, seed=M * N + K)
    prob = Problem(A, B, C0, 1.5, 0.5)
    C, n = _launches(lambda: prob.run_gpu(mode, api="ws"))
    assert n == 1, f"{n} launches"
    Cref, D = prob.oracle(oracle_mod)
    assert oracle_mod.max_rel_err(C, Cref, D) <= TOL[mode]


@pytest.mark.parametrize("mode", ["3xtf32", "tf32"])
def test_ragged_call_on_odd_pitches_copies_its_operand(oracle_mod, mode):
    """The ragged 1000 x 1500 x 777 shape (A's pitch 777 floats): moving A
    into the workspace pays there, so the call launches more than the
    product."""
    A, B, C0 = workloads.random_inputs(1000, 1500, 777, seed=3)
    prob = Problem(A, B, C0, 1.0, -2.0)
    C, n = _launches(lambda: prob.run_gpu(mode, api="ws"))
    assert n >= 2, f"{n} launches"
    rows = [0, 1, 127, 128, 511, 998, 999]
    Cref, D = prob.oracle(oracle_mod, rows=[(0, i) for i in rows])
    got = np.stack([C[0, i] for i in rows])
    assert oracle_mod.max_rel_err(got, Cref, D) <= TOL[mode]
