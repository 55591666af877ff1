"""The tensor-core raw route: both operands staged by TMA straight from the
caller's fp32 matrices (K-major or M/N-major as stored), kind::tf32 reading
the 19 high bits of each value.

For 3xTF32 the lo planes come from a pass into the workspace (route RAW) or
are made inside the product kernel from the staged raw operands (route
INLINE).

Pins of what the tensor core does with an fp32 operand:
  - TF32 on the raw route multiplies each value with its 13 low mantissa bits
    cleared: on integer-valued data whose low bits are filled with noise it
    matches the integer product exactly (the noise is dropped, not rounded);
  - 3xTF32 on the raw route (raw values as hi, a pass's lo planes) gives, bit
    for bit, the planes route's result (hi = the value with its 13 low
    mantissa bits cleared, written by that route's pass), in every layout.
And the route against the oracle on ragged, transposed, batched and broadcast
shapes."""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem

pytestmark = pytest.mark.gpu

LAYOUTS = [(0, 1), (0, 0), (1, 1), (1, 0)]


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


def tma_pads(M, N, K, tA, tB):
    """Pads that make both operands' leading dimensions multiples of four
    values (the raw route's TMA rule)."""
    la = M if tA else K
    lb = K if tB else N
    return (-la % 4, -lb % 4, 0)


def noisy_integers(rng, shape):
    """Nonzero integers in [-8, 8] with their 13 low mantissa bits set at
    random: each value is k * (1 + d), 0 <= d < 2^-10, and clearing those
    bits gives k back exactly."""
    k = rng.integers(1, 9, size=shape) * rng.choice([-1, 1], size=shape)
    bits = k.astype(np.float32).view(np.uint32) | rng.integers(0, 0x2000, size=shape,
                                                              dtype=np.uint32)
    return bits.view(np.float32), k.astype(np.float32)


@pytest.mark.parametrize("tA,tB", LAYOUTS)
def test_tf32_raw_drops_the_low_mantissa_bits(oracle_mod, forced, tA, tB):
    forced("raw")
    rng = np.random.default_rng(31 + 2 * tA + tB)
    M, N, K = 300, 260, 333
    A, Ak = noisy_integers(rng, (M, K))
    B, Bk = noisy_integers(rng, (K, N))
    C0 = np.zeros((M, N), np.float32)
    prob = Problem(A, B, C0, 1.0, 0.0, transA=tA, transB=tB, pads=tma_pads(M, N, K, tA, tB))
    C = prob.run_gpu("tf32", api="ws")
    exact = Problem(Ak, Bk, C0, 1.0, 0.0)
    Cref, _ = exact.oracle(oracle_mod)
    assert np.array_equal(C.astype(np.float64), Cref)


@pytest.mark.parametrize("route", ["raw", "inline"])
@pytest.mark.parametrize("tA,tB", LAYOUTS)
def test_3xtf32_raw_matches_planes_bit_for_bit(forced, tA, tB, route):
    """The lo planes from the pass (RAW) or made in the product kernel
    (INLINE): the same values in the same order as the planes route."""
    M, N, K = 520, 390, 700
    A, B, C0 = workloads.random_inputs(M, N, K, seed=41 + 2 * tA + tB)
    pa, pb, _ = tma_pads(M, N, K, tA, tB)
    prob = Problem(A, B, C0, 0.75, 0.25, transA=tA, transB=tB, pads=(pa + 4, pb + 8, 0))
    forced(route)
    C_raw = prob.run_gpu("3xtf32", api="ws")
    forced("planes")
    C_planes = prob.run_gpu("3xtf32", api="ws")
    assert np.array_equal(C_raw, C_planes)


RAW_CASES = [
    # M, N, K, Q, transA, transB, broadcast A, broadcast B
    (1000, 1500, 777, 1, 0, 0, False, False),
    (1000, 1500, 777, 1, 1, 1, False, False),
    (33, 70, 1, 1, 0, 0, False, False),
    (300, 40, 2049, 1, 1, 0, False, False),
    (256, 512, 512, 4, 0, 1, False, False),
    (200, 136, 96, 3, 1, 0, True, False),
    (200, 136, 96, 3, 0, 1, False, True),
]


@pytest.mark.parametrize("mode,route", [("3xtf32", "raw"), ("3xtf32", "inline"), ("tf32", "raw")])
@pytest.mark.parametrize("case", RAW_CASES)
def test_raw_route_matches_the_oracle(oracle_mod, forced, mode, route, case):
    M, N, K, Q, tA, tB, bcA, bcB = case
    forced(route)
    A, B, C0 = workloads.random_inputs(M, N, K, seed=M + 3 * N + K, Q=Q)
    if bcA:
        A = np.broadcast_to(A[:1], A.shape).copy()
    if bcB:
        B = np.broadcast_to(B[:1], B.shape).copy()
    pa, pb, _ = tma_pads(M, N, K, tA, tB)
    prob = Problem(A, B, C0, 1.5, -2.0, transA=tA, transB=tB, pads=(pa, pb + 4, 3),
                   offsets=(4, 8, 1),
                   strideA=0 if bcA else None, strideB=0 if bcB else None)
    C = prob.run_gpu(mode, api="ws")
    Cref, D = prob.oracle(oracle_mod)
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode} {case}: {err:.3e}"


@pytest.mark.parametrize("mode", ["3xtf32", "tf32"])
def test_raw_route_needs_tma_describable_operands(oracle_mod, forced, mode):
    """A leading dimension that is not a multiple of four values cannot go
    through TMA: the forced raw route then runs another kernel, with the same
    result within the mode's bound."""
    forced("raw")
    M, N, K = 130, 200, 301
    A, B, C0 = workloads.random_inputs(M, N, K, seed=7)
    prob = Problem(A, B, C0, 1.0, 0.5, pads=(1, 0, 0))
    C = prob.run_gpu(mode, api="ws")
    Cref, D = prob.oracle(oracle_mod)
    assert oracle_mod.max_rel_err(C, Cref, D) <= TOL[mode]


@pytest.mark.parametrize("mode", ["3xtf32", "tf32"])
def test_one_buffer_many_shapes(oracle_mod, mode):
    """The same device buffers used for calls of different shapes, leading
    dimensions and batch counts in turn (tensor maps are cached by their full
    description: each shape must get its own), each call against the oracle."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    cap = 1 << 22
    dA = torch.empty(cap, device=dev)
    dB = torch.empty(cap, device=dev)
    dC = torch.empty(cap, device=dev)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
    shapes = [(640, 512, 384, 1, 0), (512, 640, 384, 1, 1), (640, 512, 384, 1, 0),
              (256, 384, 512, 3, 0), (384, 256, 640, 1, 1), (640, 512, 384, 1, 0)]
    for i, (M, N, K, Q, tB) in enumerate(shapes):
        A, B, C0 = workloads.random_inputs(M, N, K, seed=200 + i, Q=Q)
        prob = Problem(A, B, C0, 1.0, 0.5, transB=tB)
        assert prob.Abuf.size <= cap and prob.Bbuf.size <= cap and prob.Cbuf.size <= cap
        dA[:prob.Abuf.size].copy_(torch.from_numpy(prob.Abuf))
        dB[:prob.Bbuf.size].copy_(torch.from_numpy(prob.Bbuf))
        dC[:prob.Cbuf.size].copy_(torch.from_numpy(prob.Cbuf))
        wsb = lib.sgemm_workspace_size(mode, M, N, K, Q)
        assert wsb <= ws.numel()
        st = lib.sgemm_batched_ex_ws(mode, M, N, K, 1.0, dA, prob.lda, dB, prob.ldb, 0.5, dC,
                                     prob.ldc, 0, tB, prob.sA, prob.sB, prob.sC, Q, ws, wsb)
        assert st == lib.SGEMM_OK
        assert lib.sgemm_poll_error() == lib.SGEMM_OK
        C = prob.extract(dC[:prob.Cbuf.size].cpu().numpy())
        Cref, D = prob.oracle(oracle_mod)
        assert oracle_mod.max_rel_err(C, Cref, D) <= TOL[mode], (mode, M, N, K, Q, tB)
