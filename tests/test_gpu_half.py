"""GPU parity of the 16-bit-input path (sgemm_half_batched: bf16 or fp16 A
and B, fp32 accumulation and output) against the fp64 oracle run on the
same values: every product of two 16-bit values is exact, so the metric and
tolerance are the FP32 path's (2e-5 of |alpha| |A||B| + |beta C0|), and
integer-valued inputs must match bit for bit."""
import numpy as np
import pytest

import workloads
from _helpers import Problem, sample_rows

pytestmark = pytest.mark.gpu

TYPES = ["bf16", "fp16"]
LAYOUTS = [(0, 1), (0, 0), (1, 0), (1, 1)]   # (transA, transB); (0, 1) is read directly
TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()
    torch.cuda.init()


def run_half(prob, type_, ws_bytes=None, expect=None):
    """C (Q, M, N) from sgemm_half_batched on the problem's buffers, A and B
    encoded as 16-bit values (the problem's float32 values are exact in
    type_, padding included)."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    A = torch.from_numpy(workloads.half_bits(prob.Abuf, type_).view(np.int16)).to(dev)
    B = torch.from_numpy(workloads.half_bits(prob.Bbuf, type_).view(np.int16)).to(dev)
    C = torch.from_numpy(prob.Cbuf).to(dev)
    if ws_bytes is None:
        ws_bytes = lib.sgemm_half_workspace_size(type_, prob.M, prob.N, prob.K, prob.transA,
                                                 prob.transB, prob.lda, prob.ldb, prob.Q)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    st = lib.sgemm_half_batched(type_, prob.M, prob.N, prob.K, prob.alpha,
                                A.data_ptr() + 2 * prob.offA, prob.lda,
                                B.data_ptr() + 2 * prob.offB, prob.ldb, prob.beta,
                                C.data_ptr() + 4 * prob.offC, prob.ldc, prob.transA, prob.transB,
                                prob.sA, prob.sB, prob.sC, prob.Q, ws, ws_bytes)
    if expect is not None:
        assert st == expect, lib.sgemm_status_string(st)
        return None
    assert st == lib.SGEMM_OK, lib.sgemm_status_string(st)
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    return prob.extract(C.cpu().numpy())


def check(prob, type_, oracle_mod, exact=False):
    C = run_half(prob, type_)
    Cref, D = prob.oracle(oracle_mod)
    if exact:
        assert np.array_equal(C.astype(np.float64), Cref), "integer case not bit-exact"
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL, f"{type_}: max rel err {err:.3e}"
    return err


@pytest.mark.parametrize("tA,tB", LAYOUTS)
@pytest.mark.parametrize("type_", TYPES)
@pytest.mark.parametrize("shape", [(256, 256, 128), (300, 500, 200), (1000, 1500, 777),
                                   (64, 900, 2048)])
def test_half_matches_oracle(oracle_mod, type_, tA, tB, shape):
    """Whole tiles, ragged edges on every side, K not a multiple of 8 (the
    operands go through the workspace copy), and a skinny long-K case that
    the planner splits along K."""
    M, N, K = shape
    A, B, C0 = workloads.half_inputs(M, N, K, type_, seed=31)
    check(Problem(A, B, C0, 1.5, -0.5, tA, tB), type_, oracle_mod)


@pytest.mark.parametrize("type_", TYPES)
def test_half_padded_and_offset_operands(oracle_mod, type_):
    """Leading dimensions above the row length and bases off the 16-byte
    grain: the direct layout with ld % 8 != 0 must be copied, not misread."""
    A, B, C0 = workloads.half_inputs(200, 300, 160, type_, seed=32)
    for pads, offs in (((8, 8, 4), (0, 0, 0)), ((3, 5, 1), (1, 3, 1))):
        check(Problem(A, B, C0, 1.0, 0.25, 0, 1, pads=pads, offsets=offs), type_, oracle_mod)


@pytest.mark.parametrize("tB", [1, 0])
@pytest.mark.parametrize("type_", TYPES)
def test_half_batched(oracle_mod, type_, tB):
    A, B, C0 = workloads.half_inputs(513, 260, 136, type_, Q=4, seed=33)
    check(Problem(A, B, C0, 0.75, 0.25, 0, tB), type_, oracle_mod)


@pytest.mark.parametrize("tA,tB", LAYOUTS)
@pytest.mark.parametrize("type_", TYPES)
def test_half_integer_inputs_bit_exact(oracle_mod, type_, tA, tB):
    """Integers in [-8, 8] are exact in bf16 and fp16; every partial sum is an
    integer below 2^24, so any summation order gives the same fp32 bits."""
    A, B, C0 = workloads.integer_inputs(517, 390, 1000, seed=34)
    check(Problem(A, B, C0, 2.0, -2.0, tA, tB), type_, oracle_mod, exact=True)


@pytest.mark.parametrize("tA,tB", [(0, 1), (0, 0)])
@pytest.mark.parametrize("type_", TYPES)
def test_half_4092_sampled_rows(oracle_mod, type_, tA, tB):
    A, B, C0 = workloads.half_inputs(4092, 4092, 4092, type_, seed=35)
    prob = Problem(A, B, C0, 1.0, 0.0, tA, tB)
    C = run_half(prob, type_)
    rows = sample_rows(1, 4092, 24, seed=36, tile=256)
    Cref, D = prob.oracle(oracle_mod, rows=rows)
    got = np.stack([C[q, i] for (q, i) in rows])
    assert oracle_mod.max_rel_err(got, Cref, D) <= TOL


def test_half_beta_zero_ignores_nan_in_c(oracle_mod):
    A, B, _ = workloads.half_inputs(130, 270, 64, "bf16", seed=37)
    C0 = np.full((130, 270), np.nan, dtype=np.float32)
    prob = Problem(A, B, C0, 1.0, 0.0, 0, 1)
    C = run_half(prob, "bf16")
    assert np.isfinite(C).all()
    Cref, D = prob.oracle(oracle_mod)
    assert oracle_mod.max_rel_err(C, Cref, D) <= TOL


def test_half_alpha_zero_and_k_zero(oracle_mod):
    import dense_fp32_matrix_03_gb300 as lib
    A, B, C0 = workloads.half_inputs(100, 120, 48, "fp16", seed=38)
    C = run_half(Problem(A, B, C0, 0.0, -2.0, 0, 1), "fp16")
    assert np.array_equal(C[0], (-2.0 * C0.astype(np.float64)).astype(np.float32))


def test_half_rejects_a_workspace_too_small_for_its_copies():
    import dense_fp32_matrix_03_gb300 as lib
    A, B, C0 = workloads.half_inputs(256, 256, 128, "bf16", seed=39)
    prob = Problem(A, B, C0, 1.0, 0.0, 1, 0)   # both operands need a copy
    run_half(prob, "bf16", ws_bytes=256, expect=lib.SGEMM_ERR_INVALID_ARG)


@pytest.mark.parametrize("type_", TYPES)
def test_half_broadcast_batch_strides(oracle_mod, type_):
    """strideA = 0 (one A for every batch entry, read directly) and strideB =
    0 with B N-inner (copied once, transposed)."""
    A, B, C0 = workloads.half_inputs(96, 80, 64, type_, Q=4, seed=40)
    check(Problem(A, B, C0, 1.0, 0.5, 0, 1, strideA=0), type_, oracle_mod)
    check(Problem(A, B, C0, 1.0, 0.5, 0, 0, strideB=0), type_, oracle_mod)
