"""GPU tests of how the library composes with the caller's CUDA machinery:
calls from several host threads on their own streams at once, and calls
captured into a CUDA graph and replayed.  Every result is checked against
the fp64 oracle (integer inputs: bit for bit)."""
import threading

import numpy as np
import pytest

import workloads
from _helpers import Problem

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


def device_problem(prob):
    import torch
    dev = torch.device("cuda", 0)
    return (torch.from_numpy(prob.Abuf).to(dev), torch.from_numpy(prob.Bbuf).to(dev),
            torch.from_numpy(prob.Cbuf).to(dev))


def call_ws(lib, mode, prob, A, B, C, ws, wsb, stream):
    return lib.sgemm_batched_ex_ws(mode, prob.M, prob.N, prob.K, prob.alpha, A, prob.lda, B,
                                   prob.ldb, prob.beta, C, prob.ldc, prob.transA, prob.transB,
                                   prob.sA, prob.sB, prob.sC, prob.Q, ws, wsb, stream)


def test_concurrent_host_threads_on_their_own_streams(oracle_mod):
    """Four host threads, each with its own stream, workspace and problem
    (different shapes and paths), call the library 5 times at once."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    jobs = []
    for t, (mode, shape) in enumerate([("3xtf32", (700, 520, 900)), ("fp32", (513, 1030, 260)),
                                       ("tf32", (1100, 300, 1600)), ("3xtf32", (256, 256, 2048))]):
        A, B, C0 = workloads.integer_inputs(*shape, seed=50 + t)
        prob = Problem(A, B, C0, 2.0, 1.0, 0, t % 2)
        wsb = lib.sgemm_workspace_size(mode, prob.M, prob.N, prob.K, 1)
        jobs.append(dict(mode=mode, prob=prob, dev=device_problem(prob),
                         ws=torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda"),
                         wsb=wsb, stream=torch.cuda.Stream()))
    errors = []

    def work(j):
        try:
            A, B, C = j["dev"]
            C0 = C.clone()
            for _ in range(5):
                C.copy_(C0)  # on torch's current stream of this thread
                torch.cuda.current_stream().synchronize()
                st = call_ws(lib, j["mode"], j["prob"], A, B, C, j["ws"], j["wsb"], j["stream"])
                if st != lib.SGEMM_OK:
                    errors.append(lib.sgemm_status_string(st))
                j["stream"].synchronize()
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    for j in jobs:
        prob = j["prob"]
        Cref, _ = prob.oracle(oracle_mod)
        got = prob.extract(j["dev"][2].cpu().numpy())
        assert np.array_equal(got.astype(np.float64), Cref), j["mode"]


@pytest.mark.parametrize("mode", MODES)
def test_calls_captured_in_a_cuda_graph(oracle_mod, mode):
    """Three calls (a split-K product through the workspace, a batched
    transposed one, and a K = 0 scaling) captured into one graph, replayed
    twice on new inputs copied into the same buffers."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    probs = [Problem(*workloads.integer_inputs(256, 1024, 1024, seed=60), 1.0, 0.0),
             Problem(*workloads.integer_inputs(130, 96, 200, Q=3, seed=61), 2.0, -1.0, 1, 1)]
    bufs = [device_problem(p) for p in probs]
    wss = []
    for p in probs:
        wsb = lib.sgemm_workspace_size(mode, p.M, p.N, p.K, p.Q)
        wss.append((torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda"), wsb))
    Cs = torch.from_numpy(np.arange(64 * 48, dtype=np.float32).reshape(64, 48)).cuda()
    s = torch.cuda.Stream()
    # one call outside the capture first (library and driver state set up)
    with torch.cuda.stream(s):
        for p, (A, B, C), (ws, wsb) in zip(probs, bufs, wss):
            assert call_ws(lib, mode, p, A, B, C.clone(), ws, wsb, s) == lib.SGEMM_OK
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for p, (A, B, C), (ws, wsb) in zip(probs, bufs, wss):
            assert call_ws(lib, mode, p, A, B, C, ws, wsb, s) == lib.SGEMM_OK
        assert lib.sgemm_batched_ex_ws(mode, 64, 48, 0, 1.0, None, 1, None, 48, 0.5, Cs, 48, 0,
                                       0, 0, 0, 0, 1, None, 0, s) == lib.SGEMM_OK
    for rep in range(2):
        for i, p in enumerate(probs):
            A, B, C0 = workloads.integer_inputs(p.M, p.N, p.K, Q=p.Q, seed=70 + 10 * rep + i)
            fresh = Problem(A, B, C0, p.alpha, p.beta, p.transA, p.transB)
            for dst, src in zip(bufs[i], (fresh.Abuf, fresh.Bbuf, fresh.Cbuf)):
                dst.copy_(torch.from_numpy(src))
            probs[i] = fresh
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert lib.sgemm_poll_error() == lib.SGEMM_OK
        for p, (_, _, C) in zip(probs, bufs):
            Cref, _ = p.oracle(oracle_mod)
            assert np.array_equal(p.extract(C.cpu().numpy()).astype(np.float64), Cref)
    # the captured K = 0 call halves Cs once per replay
    want = (np.arange(64 * 48, dtype=np.float64).reshape(64, 48) * 0.5 ** 2)
    assert np.array_equal(Cs.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("mode,route", [("3xtf32", "planes"), ("3xtf32", "inline"),
                                        ("3xtf32", "raw"), ("tf32", "planes"), ("tf32", "raw")])
def test_large_shape_routes_captured_in_a_cuda_graph(oracle_mod, mode, route):
    """A call on each large-shape tensor-core route, forced -- the planes
    route (the operand pass, then the product launched as a programmatic
    dependent of it), the raw route with a lo pass, the raw route with the lo
    planes made in the kernel -- each split along K (24 of its 100 tiles)
    with its split-K fix-up and, beta != 0, C loaded and stored by TMA in the
    epilogue, captured into a graph and replayed twice on new integer
    inputs: the whole output bit for bit."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    M = N = 2560
    K = 2000
    assert lib.sgemm_tune_force(route) == lib.SGEMM_OK
    try:
        prob = Problem(*workloads.integer_inputs(M, N, K, seed=90), 2.0, -1.0)
        A, B, C = device_problem(prob)
        wsb = lib.sgemm_workspace_size(mode, M, N, K, 1)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            assert call_ws(lib, mode, prob, A, B, C, ws, wsb, s) == lib.SGEMM_OK
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            assert call_ws(lib, mode, prob, A, B, C, ws, wsb, s) == lib.SGEMM_OK
        assert lib.sgemm_last_split_count() > 1, "expected a split plan"
        for rep in range(2):
            fresh = Problem(*workloads.integer_inputs(M, N, K, seed=92 + rep), 2.0, -1.0)
            for dst, src in zip((A, B, C), (fresh.Abuf, fresh.Bbuf, fresh.Cbuf)):
                dst.copy_(torch.from_numpy(src))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert lib.sgemm_poll_error() == lib.SGEMM_OK
            got = fresh.extract(C.cpu().numpy())
            Cref, _ = fresh.oracle(oracle_mod)
            assert np.array_equal(got.astype(np.float64), Cref)
    finally:
        lib.sgemm_tune_force("auto")
