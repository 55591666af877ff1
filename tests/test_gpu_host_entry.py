"""GPU parity of the host-buffer entry point (sgemm_host): the operands start
in host memory, the call copies them in panel by panel, computes and copies C
back, and C on the host must agree with the fp64 oracle on the same host
buffers -- within the path's tolerance on random data, bit for bit on integer
data.  Also checks the throughput probes launch, finish and report plausible
rates."""
import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem

pytestmark = pytest.mark.gpu

MODES = ["fp32", "3xtf32", "tf32"]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()
    torch.cuda.init()


def run_host(prob, mode, panel_rows=0, pinned=True, stream=None):
    """C (Q=1, M, N) from sgemm_host on the problem's host buffers."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    assert prob.Q == 1
    bufs = []
    for arr in (prob.Abuf, prob.Bbuf, prob.Cbuf):
        t = torch.from_numpy(arr.copy())
        bufs.append(t.pin_memory() if pinned else t)
    hA, hB, hC = bufs
    size = lib.sgemm_host_buffer_size(mode, prob.M, prob.N, prob.K, prob.transA, prob.transB,
                                      panel_rows)
    assert size > 0
    dev = torch.empty(size, dtype=torch.uint8, device="cuda")
    st = lib.sgemm_host(mode, prob.M, prob.N, prob.K, prob.alpha,
                        hA.data_ptr() + 4 * prob.offA, prob.lda,
                        hB.data_ptr() + 4 * prob.offB, prob.ldb, prob.beta,
                        hC.data_ptr() + 4 * prob.offC, prob.ldc, prob.transA, prob.transB,
                        panel_rows, dev, size, stream)
    assert st == lib.SGEMM_OK, lib.sgemm_status_string(st)
    assert lib.sgemm_poll_error(stream) == lib.SGEMM_OK  # synchronises the stream
    return prob.extract(hC.numpy())


@pytest.mark.parametrize("panel_rows", [0, 128, 333])
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("mode", MODES)
def test_host_entry_matches_oracle(oracle_mod, mode, tA, tB, panel_rows):
    """1000 x 700 x 300 with padded host pitches (no multiple of four), beta
    != 0 (C is copied in too); panel_rows 128 and 333 give 8 and 4 panels,
    the last one ragged."""
    A, B, C0 = workloads.random_inputs(1000, 700, 300, seed=11)
    prob = Problem(A, B, C0, 1.5, -2.0, tA, tB, pads=(3, 1, 2))
    C = run_host(prob, mode, panel_rows)
    Cref, D = prob.oracle(oracle_mod)
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode}: max rel err {err:.3e}"


@pytest.mark.parametrize("beta", [0.0, 1.0])
@pytest.mark.parametrize("mode", MODES)
def test_host_entry_integer_bit_exact_pageable(oracle_mod, mode, beta):
    """Integer data from pageable host memory, 5 panels of 100 rows + 17."""
    A, B, C0 = workloads.integer_inputs(517, 260, 129, seed=12)
    prob = Problem(A, B, C0, 2.0, beta, 0, 1, pads=(1, 0, 5))
    C = run_host(prob, mode, panel_rows=100, pinned=False)
    Cref, _ = prob.oracle(oracle_mod)
    assert np.array_equal(C.astype(np.float64), Cref)


@pytest.mark.parametrize("mode", MODES)
def test_host_entry_k_zero_and_alpha_zero(oracle_mod, mode):
    """K == 0 or alpha == 0: C = beta * C0 and A, B are never read (NULL)."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    M, N = 300, 200
    rng = np.random.default_rng(13)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    for K, alpha in ((0, 1.0), (64, 0.0)):
        hC = torch.from_numpy(C0.copy()).pin_memory()
        size = lib.sgemm_host_buffer_size(mode, M, N, K, 0, 0, 0)
        dev = torch.empty(size, dtype=torch.uint8, device="cuda")
        st = lib.sgemm_host(mode, M, N, K, alpha, None, max(K, 1), None, N, 2.0, hC, N, 0, 0, 0,
                            dev, size)
        assert st == lib.SGEMM_OK
        assert lib.sgemm_poll_error() == lib.SGEMM_OK
        assert np.array_equal(hC.numpy(), (2 * C0.astype(np.float64)).astype(np.float32))


def test_host_entry_rejects_a_small_buffer():
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    size = lib.sgemm_host_buffer_size("fp32", 256, 256, 256)
    dev = torch.empty(size, dtype=torch.uint8, device="cuda")
    h = torch.zeros(256 * 256).pin_memory()
    st = lib.sgemm_host("fp32", 256, 256, 256, 1.0, h, 256, h, 256, 0.0, h, 256, 0, 0, 0, dev,
                        size - 256)
    assert st == lib.SGEMM_ERR_INVALID_ARG


def test_host_entry_orders_with_the_callers_stream(oracle_mod):
    """Two calls back to back on a side stream reuse one device buffer; the
    second must not overwrite the first's operands before it is done."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    s = torch.cuda.Stream()
    M = N = K = 512
    outs = []
    size = lib.sgemm_host_buffer_size("3xtf32", M, N, K, 0, 0, 128)
    dev = torch.empty(size, dtype=torch.uint8, device="cuda")
    probs = []
    for seed in (21, 22):
        A, B, C0 = workloads.integer_inputs(M, N, K, seed=seed)
        probs.append(Problem(A, B, C0, 1.0, 0.0))
    hosts = [[torch.from_numpy(a.copy()).pin_memory() for a in (p.Abuf, p.Bbuf, p.Cbuf)]
             for p in probs]
    for p, (hA, hB, hC) in zip(probs, hosts):
        st = lib.sgemm_host("3xtf32", M, N, K, 1.0, hA, p.lda, hB, p.ldb, 0.0, hC, p.ldc, 0, 0,
                            128, dev, size, s)
        assert st == lib.SGEMM_OK
    assert lib.sgemm_poll_error(s) == lib.SGEMM_OK
    for p, (_, _, hC) in zip(probs, hosts):
        Cref, _ = p.oracle(oracle_mod)
        assert np.array_equal(p.extract(hC.numpy()).astype(np.float64), Cref)


# ------------------------------------------------------------------ probes

PROBE_RANGES = {  # TFLOP/s a GB300 can plausibly show (nominal peaks inside)
    "ffma": (20, 110), "ffma2": (20, 110), "tf32_ss": (200, 1600),
    "tf32_ts": (200, 1600), "bf16_ss": (400, 3200),
}


@pytest.mark.parametrize("kind", sorted(PROBE_RANGES))
def test_peak_probe_runs_and_is_plausible(kind):
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    iters = 512 if kind.startswith("ffma") else 4096
    st, flops = lib.sgemm_peak_probe(kind, iters)
    assert st == lib.SGEMM_OK and flops > 0
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    st, flops = lib.sgemm_peak_probe(kind, iters)
    e1.record()
    assert st == lib.SGEMM_OK
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    lo, hi = PROBE_RANGES[kind]
    assert lo <= tflops <= hi, f"{kind}: {tflops:.1f} TFLOP/s"


@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("mode", MODES)
def test_host_entry_long_k(oracle_mod, mode, tA, tB):
    """Long K (1500, 1100) with 256- and 128-row panels, products of even
    and odd panels on two streams: random data within tolerance, integer
    data bit for bit."""
    A, B, C0 = workloads.random_inputs(600, 500, 1500, seed=41)
    prob = Problem(A, B, C0, 1.5, -0.5, tA, tB, pads=(2, 1, 3))
    C = run_host(prob, mode, panel_rows=256)
    Cref, D = prob.oracle(oracle_mod)
    assert oracle_mod.max_rel_err(C, Cref, D) <= TOL[mode]
    A, B, C0 = workloads.integer_inputs(300, 260, 1100, seed=42)
    prob = Problem(A, B, C0, 2.0, -1.0, tA, tB)
    C = run_host(prob, mode, panel_rows=128)
    Cref, _ = prob.oracle(oracle_mod)
    assert np.array_equal(C.astype(np.float64), Cref)


@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_host_entry_large_panels(oracle_mod, tA, tB):
    """3xTF32 at 3072 x 3072 x 2000 with 512-row panels: each of the six
    panels' products is one workspace-entry call on the device copies (the
    raw route, no pass over the operands), so the call launches one product
    and at most one split-K fix-up per panel.  Random data on sampled rows
    within tolerance, integer data bit for bit."""
    import torch
    mode = "3xtf32"
    import dense_fp32_matrix_03_gb300 as lib
    from _helpers import sample_rows
    M = N = 3072
    K = 2000
    rows = sample_rows(1, M, 16, seed=51, tile=256)
    for data, exact in ((workloads.random_inputs, False), (workloads.integer_inputs, True)):
        A, B, C0 = data(M, N, K, seed=52)
        prob = Problem(A, B, C0, 2.0, -1.0, tA, tB)
        torch.cuda.synchronize()
        n0 = lib.sgemm_kernel_launches()
        C = run_host(prob, mode, panel_rows=512)
        launched = lib.sgemm_kernel_launches() - n0
        assert 6 <= launched <= 12, f"{launched} launches"
        Cref, D = prob.oracle(oracle_mod, rows=rows)
        got = np.stack([C[q, i] for q, i in rows])
        if exact:
            assert np.array_equal(got.astype(np.float64), Cref)
        else:
            assert oracle_mod.max_rel_err(got, Cref, D) <= TOL[mode]
