"""GPU parity of the tensor-core planes route: with a workspace, shapes large
enough for it (the library's cost model: the operand pass must cost less than
the product saves) first rewrite A and B into TF32 planes (3xTF32: hi and
lo; TF32: rounded to nearest) and then multiply on the shared-memory-operand
kernel.  Every layout, padded and unaligned operands, ragged M/N/K, batches
with a broadcast operand, integer data bit for bit; sampled rows against the
oracle.  The workspace shows the route was taken: it starts with op(A)'s
first plane, row 0 of which the test recomputes from the definition (hi:
the 13 low mantissa bits cleared; TF32: rounded to nearest, ties away).

Operands TMA can describe take the raw route under the cost models
(test_gpu_raw.py), so these tests force the planes route; unaligned
operands, which the raw route cannot take, reach it under the cost models."""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem, sample_rows

pytestmark = pytest.mark.gpu

MODES = ["3xtf32", "tf32"]


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
def planes_forced():
    import dense_fp32_matrix_03_gb300 as lib
    assert lib.sgemm_tune_force("planes") == lib.SGEMM_OK
    yield
    lib.sgemm_tune_force("auto")


def first_plane_row(a_row, mode):
    """Row 0 of op(A)'s first plane as the planes route writes it."""
    bits = np.ascontiguousarray(a_row, dtype=np.float32).view(np.uint32)
    if mode == "tf32":
        bits = bits + np.uint32(0x1000)  # half of the dropped range: ties away
    return (bits & np.uint32(0xFFFFE000)).view(np.float32)


def launches_of(fn):
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    torch.cuda.synchronize()
    n0 = lib.sgemm_kernel_launches()
    out = fn()
    return out, lib.sgemm_kernel_launches() - n0


def check(prob, mode, oracle_mod, rows, exact=False, opA0=None):
    """opA0: row 0 of op(A); the workspace must start with its first plane
    (the planes route ran)."""
    C = prob.run_gpu(mode, api="ws")
    if opA0 is not None:
        K = opA0.shape[0]
        got = prob.last_ws[:4 * K].view(__import__("torch").float32).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), first_plane_row(opA0, mode).view(np.uint32)), \
            "planes route not taken"
    Cref, D = prob.oracle(oracle_mod, rows=rows)
    got = np.stack([C[q, i] for q, i in rows])
    if exact:
        assert np.array_equal(got.astype(np.float64), Cref)
    else:
        err = oracle_mod.max_rel_err(got, Cref, D)
        assert err <= TOL[mode], f"{mode}: max rel err {err:.3e}"
    return C


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("mode", MODES)
def test_planes_route_every_layout(oracle_mod, planes_forced, mode, tA, tB):
    """3100 x 3000 x 2333: ragged tiles in M and N, K not a multiple of the
    32-wide box; padded leading dimensions, beta != 0."""
    A, B, C0 = workloads.random_inputs(3100, 3000, 2333, seed=61 + 2 * tA + tB)
    prob = Problem(A, B, C0, 1.25, -0.75, tA, tB, pads=(4, 8, 3))
    check(prob, mode, oracle_mod, sample_rows(1, 3100, 24, seed=tA + 2 * tB, tile=256), opA0=A[0])


@pytest.mark.parametrize("mode", MODES)
def test_planes_route_unaligned_operands(oracle_mod, mode):
    """Odd leading dimensions and bases off 16 bytes: the pass reads them
    value by value; the planes are aligned whatever the source.  Under the
    cost models: TMA cannot describe these operands, so the raw route does
    not apply."""
    A, B, C0 = workloads.random_inputs(3100, 3000, 2333, seed=67)
    for tA, tB in ((0, 0), (1, 1)):
        prob = Problem(A, B, C0, 1.0, 0.5, tA, tB, pads=(1, 3, 1), offsets=(1, 3, 2))
        check(prob, mode, oracle_mod, sample_rows(1, 3100, 16, seed=5, tile=256), opA0=A[0])


@pytest.mark.parametrize("mode", MODES)
def test_planes_route_batched_broadcast(oracle_mod, planes_forced, mode):
    """Q = 3 with A broadcast (stride 0): A's planes hold one entry, B's
    three; batch entries and planes share the tensor map's third dimension."""
    Q = 3
    A, B, C0 = workloads.random_inputs(3100, 3000, 800, Q=Q, seed=71)
    prob = Problem(A[:1].repeat(Q, axis=0), B, C0, 0.5, 1.0, 0, 1, strideA=0)
    check(prob, mode, oracle_mod, sample_rows(Q, 3100, 24, seed=6, tile=256), opA0=A[0, 0])


@pytest.mark.parametrize("mode", MODES)
def test_planes_route_integer_bit_exact(oracle_mod, planes_forced, mode):
    """Small integers: every plane, product and partial sum is exact, so the
    result equals the oracle's bit for bit (the last wave's tiles are also
    split along K)."""
    A, B, C0 = workloads.integer_inputs(3072, 3072, 2000, seed=73)
    for tA, tB in ((0, 0), (1, 1)):
        prob = Problem(A, B, C0, 2.0, -1.0, tA, tB)
        check(prob, mode, oracle_mod, sample_rows(1, 3072, 16, seed=7, tile=256), exact=True,
              opA0=A[0])


@pytest.mark.parametrize("mode", MODES)
def test_planes_route_small_workspace_falls_back(oracle_mod, planes_forced, mode):
    """A workspace too small for the planes: the pair kernel runs instead,
    with the same results within tolerance."""
    import dense_fp32_matrix_03_gb300 as lib
    A, B, C0 = workloads.random_inputs(3100, 3000, 2333, seed=79)
    prob = Problem(A, B, C0, 1.0, 0.0)
    full = lib.sgemm_workspace_size(mode, 3100, 3000, 2333, 1)
    C, n = launches_of(lambda: prob.run_gpu(mode, api="ws", ws_bytes=full // 4))
    assert n <= 2  # the pair kernel and at most a fix-up: no pass
    rows = sample_rows(1, 3100, 16, seed=8, tile=256)
    Cref, D = prob.oracle(oracle_mod, rows=rows)
    got = np.stack([C[q, i] for q, i in rows])
    assert oracle_mod.max_rel_err(got, Cref, D) <= TOL[mode]


@pytest.mark.parametrize("mode", MODES)
def test_planes_route_long_k(oracle_mod, planes_forced, mode):
    """2900 x 3000 x 12001: hundreds of k-blocks, K odd (the pass zero-fills
    the last group of four, TMA the rest of the last box), the last wave's
    tiles split along K into many slices; B stored transposed."""
    A, B, C0 = workloads.random_inputs(2900, 3000, 12001, seed=83)
    prob = Problem(A, B, C0, 1.0, 0.25, 0, 1)
    check(prob, mode, oracle_mod, sample_rows(1, 2900, 12, seed=9, tile=256), opA0=A[0])
