"""GPU parity: the library (through the C ABI) against the fp64 CPU oracle,
element by element on the same seeded inputs.

Accuracy metric (per element): |C - C_ref| / (|alpha| (|A||B|)_ij + |beta C0_ij| + 1e-30),
bounded by 2e-5 for the FP32 and 3xTF32 paths and 2e-3 for plain TF32;
integer-valued inputs must match bit for bit on every path.
"""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem, sample_rows

pytestmark = pytest.mark.gpu

MODES = ["fp32", "3xtf32", "tf32"]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()  # fails loudly if the library was not built
    torch.cuda.init()


def supported(mode):
    """Skips the tensor-core modes on a build where they report UNSUPPORTED."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    a = torch.ones(16, 16, device="cuda")
    c = torch.zeros(16, 16, device="cuda")
    st = lib.sgemm_batched_ex(mode, 16, 16, 16, 1.0, a, 16, a, 16, 0.0, c, 16, 0, 0, 0, 0, 0, 1)
    torch.cuda.synchronize()
    if st == lib.SGEMM_ERR_UNSUPPORTED:
        pytest.skip(f"mode {mode} not available on this device")
    assert st == lib.SGEMM_OK


def check_full(prob, mode, oracle_mod, exact=False, api="ex"):
    C = prob.run_gpu(mode, api=api)
    Cref, D = prob.oracle(oracle_mod)
    if exact:
        assert np.array_equal(C.astype(np.float64), Cref), "integer case not bit-exact"
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode}: max rel err {err:.3e}"
    return err


def check_rows(prob, mode, oracle_mod, rows, exact=False, api="ex"):
    C = prob.run_gpu(mode, api=api)
    Cref, D = prob.oracle(oracle_mod, rows=rows)
    got = np.stack([C[q, i] for (q, i) in rows])
    if exact:
        assert np.array_equal(got.astype(np.float64), Cref), "integer case not bit-exact"
    err = oracle_mod.max_rel_err(got, Cref, D)
    assert err <= TOL[mode], f"{mode}: max rel err {err:.3e} on sampled rows"
    return C


# ------------------------------------------------------------- the workloads

@pytest.mark.parametrize("mode", MODES)
def test_sgemm_256(oracle_mod, mode):
    supported(mode)
    w = workloads.make("sgemm_256")
    check_full(Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0]), mode, oracle_mod)


@pytest.mark.parametrize("mode", MODES)
def test_sgemm_ragged_beta_zero_then_minus_two(oracle_mod, mode):
    supported(mode)
    w = workloads.make("sgemm_ragged_1000x1500x777")
    for beta in w["betas"]:
        check_full(Problem(w["A"], w["B"], w["C0"], w["alpha"], beta), mode, oracle_mod)


@pytest.mark.parametrize("mode", MODES)
def test_sgemm_4092_sampled_rows(oracle_mod, mode):
    supported(mode)
    w = workloads.make("sgemm_4092")
    prob = Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0])
    C = check_rows(prob, mode, oracle_mod, sample_rows(1, 4092, 40, seed=2), api="ex")
    assert np.all(np.isfinite(C))


@pytest.fixture(scope="module")
def oracle_4092(oracle_mod):
    """The oracle's whole 4092^3 result (every one of the 16.7 M outputs),
    computed once for the three paths."""
    w = workloads.make("sgemm_4092")
    prob = Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0])
    Cref, D = prob.oracle(oracle_mod)
    return prob, Cref, D


@pytest.mark.parametrize("mode", MODES)
def test_sgemm_4092_every_output_workspace_entry(oracle_4092, oracle_mod, mode):
    """The benchmark's call (sgemm_batched_ex_ws with the workspace the
    library asks for: operand pass, product, split-K fix-up of the last
    wave) against the oracle on every output element, so that every split
    tile of the last wave is checked, not only sampled rows."""
    supported(mode)
    prob, Cref, D = oracle_4092
    C = prob.run_gpu(mode, api="ws")
    assert np.all(np.isfinite(C))
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode}: max rel err {err:.3e} over all outputs"


_SWEEP_ORACLE = {}


def sweep_oracle(oracle_mod, n):
    """The oracle's whole result for sweep size n (computed once for the
    three paths)."""
    if n not in _SWEEP_ORACLE:
        _SWEEP_ORACLE.clear()
        w = workloads.make(f"sweep_{n}")
        prob = Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0])
        _SWEEP_ORACLE[n] = (prob,) + tuple(prob.oracle(oracle_mod))
    return _SWEEP_ORACLE[n]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", workloads.SWEEP_SIZES)
def test_size_sweep(oracle_mod, mode, n):
    """Every output element up to 4096 (the 4096^3 oracle takes a few seconds
    on the host cores and is shared by the three paths); sampled rows at
    8192 (over a minute of oracle time per path otherwise)."""
    supported(mode)
    if n <= 4096:
        prob, Cref, D = sweep_oracle(oracle_mod, n)
        C = prob.run_gpu(mode)
        err = oracle_mod.max_rel_err(C, Cref, D)
        assert err <= TOL[mode], f"{mode} sweep_{n}: max rel err {err:.3e} over all outputs"
    else:
        w = workloads.make(f"sweep_{n}")
        prob = Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0])
        check_rows(prob, mode, oracle_mod, sample_rows(1, n, 24, seed=n))


@pytest.fixture(scope="module")
def oracle_bmm(oracle_mod):
    """The oracle's whole result for the batched workload (32 x 1024 x 1024,
    K = 512; every one of the 33.5 M outputs), computed once: both storages
    of B hold the same logical B."""
    w = workloads.make("bmm_q32_1024x1024x512")
    prob = Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0])
    return w, prob.oracle(oracle_mod)


@pytest.mark.parametrize("api", ["ex", "ws"])
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("transB", [1, 0])
def test_batched_q32(oracle_bmm, oracle_mod, mode, transB, api):
    """The batched workload on both storages of B, through the plain and the
    workspace entry, on every output element."""
    supported(mode)
    w, (Cref, D) = oracle_bmm
    prob = Problem(w["A"], w["B"], w["C0"], w["alpha"], w["betas"][0], transB=transB)
    C = prob.run_gpu(mode, api=api)
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode} transB={transB} {api}: max rel err {err:.3e}"


# -------------------------------------------------------- exactness (integers)

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape,alpha,beta,tA,tB", [
    ((256, 256, 256), 1.0, 0.0, 0, 0),
    ((1000, 1500, 777), 2.0, -2.0, 0, 0),
    ((129, 131, 300), 1.0, 1.0, 1, 0),
    ((200, 96, 4092), 1.0, 0.0, 0, 1),
    ((97, 64, 33), 2.0, 1.0, 1, 1),
])
def test_integer_inputs_bit_exact(oracle_mod, mode, shape, alpha, beta, tA, tB):
    supported(mode)
    M, N, K = shape
    A, B, C0 = workloads.integer_inputs(M, N, K, seed=M + K)
    check_full(Problem(A, B, C0, alpha, beta, transA=tA, transB=tB), mode, oracle_mod, exact=True)


@pytest.fixture(scope="module")
def oracle_4092_integer(oracle_mod):
    """Integer inputs at 4092^3 and the oracle's whole result for them
    (every partial sum an integer below 2^24: exact in fp32 in any order)."""
    A, B, C0 = workloads.integer_inputs(4092, 4092, 4092, seed=42)
    prob = Problem(A, B, C0, 1.0, 0.0)
    Cref, _ = prob.oracle(oracle_mod)
    return prob, Cref


@pytest.mark.parametrize("api", ["ex", "ws"])
@pytest.mark.parametrize("mode", MODES)
def test_integer_4092_bit_exact(oracle_4092_integer, mode, api):
    """Every one of the 16.7 M outputs bit for bit, through the plain entry
    and the benchmark's workspace entry (whose last wave is split along K)."""
    supported(mode)
    prob, Cref = oracle_4092_integer
    C = prob.run_gpu(mode, api=api)
    assert np.array_equal(C.astype(np.float64), Cref), "integer case not bit-exact"


@pytest.mark.parametrize("mode", MODES)
def test_integer_batched_transposed_bit_exact(oracle_mod, mode):
    supported(mode)
    A, B, C0 = workloads.integer_inputs(70, 90, 200, Q=3, seed=9)
    for tA in (0, 1):
        for tB in (0, 1):
            check_full(Problem(A, B, C0, 1.0, 1.0, transA=tA, transB=tB), mode, oracle_mod,
                       exact=True)


@pytest.mark.parametrize("mode", MODES)
def test_integer_unaligned_operands_bit_exact(oracle_mod, mode):
    """Operands TMA cannot describe (odd leading dimensions, unaligned bases)
    take the element-wise producers: still exact on integer data."""
    supported(mode)
    A, B, C0 = workloads.integer_inputs(130, 150, 97, Q=2, seed=13)
    for tA in (0, 1):
        for tB in (0, 1):
            check_full(Problem(A, B, C0, 2.0, -1.0, transA=tA, transB=tB, pads=(3, 5, 7),
                               offsets=(1, 2, 3)), mode, oracle_mod, exact=True)


@pytest.mark.parametrize("mode", MODES)
def test_unaligned_operands_through_the_workspace(oracle_mod, mode):
    """The same unaligned operands with a workspace: the tensor-core paths
    copy them to 128-byte pitches and run the TMA-fed kernel, the FP32 path
    transposes or keeps them; random data within tolerance, integer data
    bit for bit, batched and broadcast."""
    supported(mode)
    A, B, C0 = workloads.random_inputs(300, 260, 197, Q=3, seed=14)
    for tA in (0, 1):
        for tB in (0, 1):
            check_full(Problem(A, B, C0, 1.5, 0.5, transA=tA, transB=tB, pads=(1, 3, 0),
                               offsets=(1, 0, 1)), mode, oracle_mod, api="ws")
    A, B, C0 = workloads.integer_inputs(1000, 1500, 777, seed=15)
    check_full(Problem(A, B, C0, 1.0, 0.0), mode, oracle_mod, exact=True, api="ws")
    A, B, C0 = workloads.integer_inputs(129, 70, 33, Q=4, seed=16)
    check_full(Problem(A, B, C0, 2.0, 1.0, strideA=0, offsets=(1, 0, 0)), mode, oracle_mod,
               exact=True, api="ws")


# ---------------------------------------------------------- ragged sweeps

RAGGED = [1, 7, 31, 127, 128, 129, 777]


@pytest.mark.parametrize("mode", MODES)
def test_ragged_shape_sweep(oracle_mod, mode):
    supported(mode)
    rng = np.random.default_rng(5)
    combos = {(m, n, k) for m in (1, 129) for n in (1, 127) for k in (1, 777)}
    while len(combos) < 40:
        combos.add(tuple(int(x) for x in rng.choice(RAGGED, 3)))
    for i, (M, N, K) in enumerate(sorted(combos)):
        A, B, C0 = workloads.random_inputs(M, N, K, seed=i)
        tA, tB = i % 2, (i // 2) % 2
        check_full(Problem(A, B, C0, 1.25, -0.5, transA=tA, transB=tB), mode, oracle_mod)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("pads,offsets", [
    ((3, 5, 7), (0, 0, 0)),      # leading dimensions not multiples of 4 floats
    ((4, 4, 4), (1, 2, 3)),      # bases not 16-byte aligned
    ((0, 0, 0), (4, 4, 4)),      # 16-byte aligned offsets
    ((64, 0, 32), (0, 0, 1)),    # wide padding, unaligned C only
])
def test_leading_dims_and_alignment(oracle_mod, mode, pads, offsets):
    supported(mode)
    for (tA, tB) in [(0, 0), (1, 1), (0, 1), (1, 0)]:
        A, B, C0 = workloads.random_inputs(150, 170, 97, Q=2, seed=tA * 2 + tB)
        check_full(Problem(A, B, C0, 0.5, 2.0, transA=tA, transB=tB, pads=pads,
                           offsets=offsets), mode, oracle_mod)


@pytest.mark.parametrize("mode", MODES)
def test_broadcast_batch_strides(oracle_mod, mode):
    supported(mode)
    A, B, C0 = workloads.random_inputs(96, 80, 64, Q=4, seed=11)
    check_full(Problem(A, B, C0, 1.0, 0.5, strideA=0), mode, oracle_mod)
    check_full(Problem(A, B, C0, 1.0, 0.5, transB=1, strideB=0), mode, oracle_mod)


# ---------------------------------------------------- BLAS special cases

@pytest.mark.parametrize("mode", MODES)
def test_beta_zero_ignores_nan_in_c(oracle_mod, mode):
    supported(mode)
    A, B, _ = workloads.random_inputs(64, 48, 40, seed=1)
    C0 = np.full((64, 48), np.nan, np.float32)
    prob = Problem(A, B, C0, 1.0, 0.0)
    C = prob.run_gpu(mode)
    assert np.all(np.isfinite(C))
    check_full(prob, mode, oracle_mod)


@pytest.mark.parametrize("mode", MODES)
def test_alpha_zero_and_k_zero(oracle_mod, mode):
    supported(mode)
    rng = np.random.default_rng(2)
    C0 = rng.uniform(-1, 1, (33, 45)).astype(np.float32)
    A = np.full((33, 8), np.nan, np.float32)
    B = np.full((8, 45), np.nan, np.float32)
    C = Problem(A, B, C0, 0.0, -2.0).run_gpu(mode)
    assert np.array_equal(C[0], (-2.0 * C0).astype(np.float32))
    C = Problem(A, B, C0, 0.0, 0.0).run_gpu(mode)
    assert np.all(C == 0)
    A0 = np.zeros((33, 0), np.float32)
    B0 = np.zeros((0, 45), np.float32)
    C = Problem(A0, B0, C0, 1.0, 0.5, pads=(1, 0, 0)).run_gpu(mode)  # lda >= 1
    assert np.array_equal(C[0], (0.5 * C0).astype(np.float32))


@pytest.mark.parametrize("mode", MODES)
def test_empty_dims_leave_c_untouched(mode):
    supported(mode)
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    c = torch.full((8, 8), 3.0, device="cuda")
    a = torch.ones(8, 8, device="cuda")
    for (M, N, Q) in [(0, 8, 1), (8, 0, 1), (8, 8, 0)]:
        st = lib.sgemm_batched_ex(mode, M, N, 8, 1.0, a, 8, a, 8, 0.0, c, 8, 0, 0, 0, 0, 64, Q)
        assert st == lib.SGEMM_OK
    torch.cuda.synchronize()
    assert torch.all(c == 3.0)


def test_default_mode_entry_points(oracle_mod):
    import dense_fp32_matrix_03_gb300 as lib
    old = lib.sgemm_get_default_mode()
    try:
        for mode in MODES:
            if lib.sgemm_set_default_mode(mode) != lib.SGEMM_OK:
                continue
            supported(mode) if mode == "fp32" else None
            A, B, C0 = workloads.random_inputs(200, 136, 72, seed=3)
            prob = Problem(A, B, C0, 1.0, 1.0)
            try:
                C = prob.run_gpu(mode, api="sgemm")
            except AssertionError:
                if mode != "fp32":
                    continue
                raise
            Cref, D = prob.oracle(oracle_mod)
            assert oracle_mod.max_rel_err(C, Cref, D) <= TOL[mode]
    finally:
        lib.sgemm_set_default_mode(old)


@pytest.mark.parametrize("mode", MODES)
def test_single_gemm_explicit_mode_entry(oracle_mod, mode):
    """sgemm_ex: one GEMM, no transposes, the path named by the call."""
    supported(mode)
    A, B, C0 = workloads.random_inputs(333, 517, 258, seed=11)
    prob = Problem(A, B, C0, -0.75, 1.5, pads=(4, 0, 8))
    check_full(prob, mode, oracle_mod, api="sgemm_ex")


def test_runs_on_a_side_stream(oracle_mod):
    import torch
    A, B, C0 = workloads.random_inputs(300, 260, 190, seed=6)
    prob = Problem(A, B, C0, 1.0, 0.25)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = prob.run_gpu("fp32", stream=s)
    Cref, D = prob.oracle(oracle_mod)
    assert oracle_mod.max_rel_err(C, Cref, D) <= TOL["fp32"]


# ---------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_context_survives(oracle_mod):
    """A kernel whose mbarrier is never satisfied gives up after its bound,
    records the timeout in the status word, and exits; the next poll reports
    it once; later GEMMs still run correctly."""
    import dense_fp32_matrix_03_gb300 as lib
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    assert lib.sgemm_selftest_wait_timeout(1 << 20) == lib.SGEMM_OK
    assert lib.sgemm_poll_error() == lib.SGEMM_ERR_TIMEOUT
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    A, B, C0 = workloads.random_inputs(130, 140, 150, seed=7)
    prob = Problem(A, B, C0, 1.0, 1.0)
    C = prob.run_gpu("fp32")
    Cref, D = prob.oracle(oracle_mod)
    assert oracle_mod.max_rel_err(C, Cref, D) <= TOL["fp32"]
