"""GPU parity of the split-K path (sgemm_batched_ex_ws): the tiles of a
grid's last, partial wave (every tile of a grid smaller than the GPU) are cut
along K, each slice's partial tile goes through the caller's workspace, and
the last slice of every region sums them in slice order.  Checked against the
fp64 oracle like every other path."""
import math

import numpy as np
import pytest

import workloads
from _helpers import TOL, Problem

pytestmark = pytest.mark.gpu

MODES = ["fp32", "3xtf32", "tf32"]
SPLIT_SHAPES = [  # (M, N, K, Q, transA, transB, alpha, beta): all split on every path
    (1024, 1024, 1024, 1, 0, 0, 1.0, 0.0),
    (600, 700, 777, 1, 0, 0, 1.0, -2.0),     # ragged, lda not TMA-describable
    (256, 256, 600, 1, 0, 0, 1.5, 0.5),
    (128, 128, 1024, 1, 0, 0, 1.0, 0.0),
    (512, 512, 512, 1, 1, 1, 0.5, 1.0),
    (300, 200, 2000, 1, 0, 1, 1.0, 0.25),    # skinny output, long K
    (200, 150, 600, 3, 1, 0, -1.0, 0.5),     # batched
    (1, 7, 4000, 1, 0, 0, 1.0, 0.0),         # a single row
    (1664, 1664, 2048, 1, 0, 0, 1.0, 0.5),   # 169 tiles: one whole wave, the rest split
    (1000, 1500, 777, 1, 0, 0, 1.0, -2.0),   # 96 tiles, under one wave: all split
]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()


def make_problem(shape, seed):
    M, N, K, Q, tA, tB, alpha, beta = shape
    A, B, C0 = workloads.random_inputs(M, N, K, Q=Q, seed=seed)
    return Problem(A, B, C0, alpha, beta, transA=tA, transB=tB)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", SPLIT_SHAPES)
def test_split_k_parity(oracle_mod, mode, shape):
    import dense_fp32_matrix_03_gb300 as lib
    M, N, K, Q = shape[:4]
    assert lib.sgemm_workspace_size(mode, M, N, K, Q) > 0, "shape expected to split"
    prob = make_problem(shape, seed=M + N + K)
    C = prob.run_gpu(mode, api="ws")
    Cref, D = prob.oracle(oracle_mod)
    err = oracle_mod.max_rel_err(C, Cref, D)
    assert err <= TOL[mode], f"{mode} {shape}: max rel err {err:.3e}"


@pytest.mark.parametrize("mode,route", [("3xtf32", "inline"), ("3xtf32", "planes"),
                                        ("tf32", "raw")])
@pytest.mark.parametrize("shape", [(2560, 2560, 2000, 0), (2500, 2400, 2000, 1)])
def test_split_k_on_a_dirty_workspace(oracle_mod, mode, route, shape):
    """The shared-memory-operand kernel's split plan on a workspace filled
    with garbage first (the workspace needs no initialisation: every slot the
    fix-up reads was written by the same call), the call made twice; integer
    data bit for bit over the whole output, against the oracle.  100 tiles of
    256 x 256 on 76 CTA pairs: one whole wave and 24 split tiles; the product
    kernel and the fix-up launch (and the planes route's pass).  The second
    shape is ragged (partial tiles on both edges) with C's pitch odd, so the
    fix-up writes C with scalar stores."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    M, N, K, odd = shape
    assert lib.sgemm_tune_force(route) == lib.SGEMM_OK
    try:
        A, B, C0 = workloads.integer_inputs(M, N, K, seed=M + N)
        prob = Problem(A, B, C0, 2.0, -1.0, pads=(0, 0, 1 if odd else 0))
        wsb = lib.sgemm_workspace_size(mode, M, N, K, 1)
        for fill in (0xFF, 0x5A):
            torch.cuda.synchronize()
            n0 = lib.sgemm_kernel_launches()
            C = prob.run_gpu(mode, api="ws", ws_bytes=wsb, ws_fill=fill)
            launched = lib.sgemm_kernel_launches() - n0
            assert lib.sgemm_last_split_count() > 1, "expected a split plan"
            assert launched == (3 if route == "planes" else 2), launched
            Cref, _ = prob.oracle(oracle_mod)
            assert np.array_equal(C.astype(np.float64), Cref)
    finally:
        lib.sgemm_tune_force("auto")


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_fp32_operand_transposition_in_the_workspace(oracle_mod, tA, tB):
    """The FP32 path copies a K-inner A (N >= 1024) or B (M >= 1024) into the
    workspace transposed; with odd leading dimensions, unaligned bases, a
    broadcast A and every layout the result matches the oracle, and on
    integer data bit for bit."""
    M, N, K, Q = 1030, 1100, 64, 2
    A, B, C0 = workloads.random_inputs(M, N, K, Q=Q, seed=31 + 2 * tA + tB)
    for strideA in (None, 0):
        prob = Problem(A, B, C0, 0.75, -0.5, transA=tA, transB=tB, pads=(3, 5, 7),
                       offsets=(1, 2, 3), strideA=strideA)
        C = prob.run_gpu("fp32", api="ws")
        Cref, D = prob.oracle(oracle_mod)
        assert oracle_mod.max_rel_err(C, Cref, D) <= TOL["fp32"]
    Ai, Bi, Ci = workloads.integer_inputs(M, N, K, Q=Q, seed=7)
    prob = Problem(Ai, Bi, Ci, 2.0, 1.0, transA=tA, transB=tB, pads=(1, 3, 0))
    C = prob.run_gpu("fp32", api="ws")
    Cref, _ = prob.oracle(oracle_mod)
    assert np.array_equal(C.astype(np.float64), Cref)


@pytest.mark.parametrize("mode", MODES)
def test_split_k_integer_bit_exact(oracle_mod, mode):
    A, B, C0 = workloads.integer_inputs(700, 900, 1500, seed=5)
    prob = Problem(A, B, C0, 2.0, -1.0)
    C = prob.run_gpu(mode, api="ws")
    Cref, _ = prob.oracle(oracle_mod)
    assert np.array_equal(C.astype(np.float64), Cref)


@pytest.mark.parametrize("mode", MODES)
def test_split_k_is_deterministic(mode):
    prob = make_problem((600, 700, 777, 1, 0, 0, 1.0, 0.5), seed=9)
    C1 = prob.run_gpu(mode, api="ws")
    C2 = prob.run_gpu(mode, api="ws")
    assert np.array_equal(C1, C2)


@pytest.mark.parametrize("mode", MODES)
def test_small_or_missing_workspace_runs_unsplit(oracle_mod, mode):
    prob = make_problem((1024, 1024, 1024, 1, 0, 1, 1.0, 0.0), seed=3)
    Cref, D = prob.oracle(oracle_mod)
    for nbytes in (0, 1024):
        C = prob.run_gpu(mode, api="ws", ws_bytes=nbytes)
        assert oracle_mod.max_rel_err(C, Cref, D) <= TOL[mode]


def planned_workspace(mode, M, N, K, Q, sms, pair_slots=None):
    """The split plan as the library's header and planner describe it, for
    every kernel the mode may run (FP32: 256 x 128 tiles where the FMAs pair,
    128 x 128 with both operands K-inner, each TMA- or cp.async-fed, one unit
    per multiprocessor; tensor cores: the direct kernel's 128 x 128 tiles on
    every multiprocessor and the pair kernel's 256 x 128 tiles (256 x 256 for
    TF32 with K >= 1536), one unit per CTA pair, and the planes route's
    256 x 256 pair tiles): whole waves of units, then the last wave's r tiles cut into s
    slices (s <= 16, each >= 64 deep for FP32 and >= 256 for the tensor
    paths), s minimising t_tile * (floor(T/G) + ceil(r*s/G)/s) + 3 us +
    2 * ws / bw (G units at once; bw 8 TB/s up to 64 MB of workspace, else
    3 TB/s; t_tile from the kernel's per-multiprocessor rate times its
    multiprocessors per unit), used only if it saves 1%; returns the largest
    workspace over the kernels (one BM x BN fp32 slot per split unit), 0 when
    none splits; on the FP32 path plus room for transposed copies of A and B
    (256-byte rounded); on the tensor paths plus room for 128-byte-pitched
    copies of A and B, or, where the planes route pays, for their TF32
    planes if larger (two planes for 3xTF32, one for TF32; rows of
    round_up(K, 32) values).  The route table (tune_table.h) adds the FP32
    64 x 64 tile where it sends the shape to it, and decides the planes on
    the tensor paths: always with route PLANES, never with PAIR or DIRECT,
    by the time model with AUTO.  The raw route's lo planes (3xTF32) are
    counted with route RAW only: rows of round_up(inner, 32) values, for
    either layout.  The 256 x 256 tiles' plan is also taken at the in-kernel
    3xTF32 form's rate."""
    rates = {("fp32", "direct"): 0.24e12, ("fp32", "tma"): 0.40e12,
             ("3xtf32", "direct"): 0.47e12, ("3xtf32", "pair"): 1.8e12,
             ("tf32", "direct"): 0.55e12, ("tf32", "pair"): 3.6e12,
             ("3xtf32", "planes"): 2.45e12, ("tf32", "planes"): 6.4e12,
             ("3xtf32", "inline"): 2.35e12}
    if pair_slots is None:
        pair_slots = sms // 2
    if mode == "fp32":
        kernels = [(bm, bn, feed, sms, 1) for (bm, bn) in ((256, 128), (128, 128))
                   for feed in ("direct", "tma")]
        # the 64 x 64 tile where the route table sends this shape
        import dense_fp32_matrix_03_gb300 as lib
        if lib.sgemm_tune_route(mode, M, N, K, Q) == lib.SGEMM_ROUTE_SMALL:
            kernels += [(64, 64, feed, sms, 1) for feed in ("direct", "tma")]
    else:
        # the pair kernel: 256 x 128 tiles, 256 x 256 for TF32 with K >= 1536
        wide = mode == "tf32" and K >= 1536
        kernels = [(128, 128, "direct", sms, 1), (256, 256 if wide else 128, "pair", pair_slots, 2),
                   (256, 256, "planes", pair_slots, 2)]
        if mode == "3xtf32":  # the raw route's in-kernel form, same tiles
            kernels.append((256, 256, "inline", pair_slots, 2))
    def plan(bm, bn, feed, G, per_unit):
        """(workspace, modelled seconds) of the best split plan."""
        T = Q * math.ceil(M / bm) * math.ceil(N / bn)
        full, rem = divmod(T, G)
        t_tile = 2.0 * bm * bn * float(K) / (rates[(mode, feed)] * per_unit)
        if rem == 0:
            return 0, t_tile * full
        smax = min(16, K // (64 if mode == "fp32" else 256))
        t_whole = t_tile * float(full + 1)
        best_t, best, best_ws = t_whole, 1, 0
        for s in range(2, smax + 1):
            ws = rem * s * bm * bn * 4
            waves = (rem * s + G - 1) // G
            bw = 8e12 if ws <= (64 << 20) else 3e12
            t = t_tile * (float(full) + float(waves) / s) + 3e-6 + 2.0 * float(ws) / bw
            if t < best_t:
                best_t, best, best_ws = t, s, ws
        if best > 1 and best_t <= 0.99 * t_whole:
            return best_ws, best_t
        return 0, t_whole

    need = max(plan(*k)[0] for k in kernels)
    if mode == "fp32":
        # room for transposed copies of A (N >= 1024) and B (M >= 1024)
        def repack(inner, outer):
            return (Q * outer * ((inner + 3) // 4 * 4) * 4 + 255) // 256 * 256
        need += (repack(M, K) if N >= 1024 else 0) + (repack(N, K) if M >= 1024 else 0)
    else:
        # room for 128-byte-pitched copies of A and B, either layout
        r32 = lambda x: (x + 31) // 32 * 32
        r256 = lambda b: (b + 255) // 256 * 256

        def copy(rows):
            return r256(Q * max(rows * r32(K), K * r32(rows)) * 4)
        planes = 2 if mode == "3xtf32" else 1
        # the planes route where it pays: the modelled time of its tiles' plan
        # plus its pass ((M + N) * K * Q * 4 * (1 + planes) bytes at 6.0 TB/s)
        # and 7 us, against the modelled time of the pair kernel's plan
        import dense_fp32_matrix_03_gb300 as lib
        route = lib.sgemm_tune_route(mode, M, N, K, Q)
        t_pair = plan(*kernels[1])[1]
        t_planes = plan(*kernels[2])[1] + (M + N) * K * Q * 4.0 * (1 + planes) / 6.0e12 + 7e-6
        room = copy(M) + copy(N)
        # route RAW on 3xTF32 (a lo pass into the workspace): room for the lo
        # planes of either layout (rows of round_up(inner, 32) values); the
        # cost models' raw form needs none (TF32 has no pass, 3xTF32 makes its
        # lo planes in the kernel)
        if route == lib.SGEMM_ROUTE_RAW and mode == "3xtf32":
            lo = (r256(Q * max(M * r32(K), K * r32(M)) * 4) +
                  r256(Q * max(N * r32(K), K * r32(N)) * 4))
            room = max(room, lo)
        if (route == lib.SGEMM_ROUTE_PLANES or
                (route == lib.SGEMM_ROUTE_AUTO and t_planes < t_pair)):
            room = max(room, r256(planes * Q * M * r32(K) * 4) + r256(planes * Q * N * r32(K) * 4))
        need += room
    return need


SIZE_CASES = [("fp32", 4092, 4092, 4092, 1), ("3xtf32", 4092, 4092, 4092, 1),
              ("fp32", 256, 256, 256, 1), ("tf32", 256, 256, 256, 1),
              ("fp32", 1024, 1024, 128, 1), ("3xtf32", 1024, 1024, 128, 1),
              ("fp32", 1000, 1500, 777, 1), ("tf32", 1000, 1500, 777, 1),
              ("fp32", 1024, 1024, 32, 1), ("3xtf32", 1024, 1024, 512, 32),
              ("fp32", 8192, 8192, 8192, 1), ("tf32", 2048, 2048, 2048, 1),
              ("fp32", 1, 7, 4000, 1), ("3xtf32", 1664, 1664, 2048, 1)]


@pytest.mark.parametrize("case", SIZE_CASES)
def test_workspace_size_follows_the_plan(case):
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert lib.sgemm_workspace_size(*case) == planned_workspace(*case, sms)


def test_workspace_size_query():
    import dense_fp32_matrix_03_gb300 as lib
    assert lib.sgemm_workspace_size("fp32", 1000, 1000, 32, 1) == 0      # one k-block: no split
    assert lib.sgemm_workspace_size("fp32", 1024, 1024, 32, 1) > 0       # room to transpose A, B
    # tensor path: no split (>= 256 per slice), room for aligned copies of A and B only
    # (the planes route does not pay at this size)
    assert lib.sgemm_workspace_size("3xtf32", 1024, 1024, 128, 1) == 2 * 1024 * 128 * 4
    # the planes route at 4096^3: two planes each of A and B, 4 * 4096 * 4096 floats
    assert lib.sgemm_workspace_size("3xtf32", 4096, 4096, 4096, 1) >= 4 * 4096 * 4096 * 4
    assert lib.sgemm_workspace_size("fp32", 1024, 1024, 128, 1) > 0     # 2 slices of 64
    assert lib.sgemm_workspace_size("fp32", 0, 10, 10, 1) == 0
    assert lib.sgemm_workspace_size(7, 100, 100, 100, 1) == 0


def test_misaligned_workspace_is_rejected():
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    a = torch.ones(64, 64, device="cuda")
    c = torch.zeros(64, 64, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    st = lib.sgemm_batched_ex_ws("fp32", 64, 64, 64, 1.0, a, 64, a, 64, 0.0, c, 64, 0, 0, 0, 0, 0,
                                 1, ws.data_ptr() + 16, 4096)
    assert st == lib.SGEMM_ERR_INVALID_ARG
