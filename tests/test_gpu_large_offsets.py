"""GPU parity where element offsets pass 2**31: an output of more than 2**31
elements (row * ldc overflows 32 bits) and an A operand of more than 2**31
elements, on every path, through the plain and the workspace entry points.

The operands are integer-valued, so every result is exact in fp32 and the
sampled rows must equal the fp64 oracle bit for bit.  Only the sampled rows
travel to the host: row i of C depends on row i of op(A) and on B alone, so
the oracle is run on those rows of A as a small problem of its own."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

MODES = ["fp32", "3xtf32", "tf32"]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()


def int_tensor(shape, seed, device):
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.randint(-8, 9, shape, generator=g, device=device).to(torch.float32)


def check_rows(oracle_mod, A_rows, B, C_rows, alpha):
    """C_rows (host) against the oracle on the same rows of A."""
    n, K = A_rows.shape
    N = B.shape[1]
    Cref, _ = oracle_mod.sgemm_ref(n, N, K, alpha, A_rows, K, B, N, 0.0, None, N)
    assert np.array_equal(C_rows.astype(np.float64), Cref.reshape(n, N))


def run(lib, mode, api, M, N, K, A, B, C, alpha):
    import torch
    if api == "ws":
        wsb = lib.sgemm_workspace_size(mode, M, N, K, 1)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=C.device)
        st = lib.sgemm_batched_ex_ws(mode, M, N, K, alpha, A, A.stride(0), B, B.stride(0), 0.0,
                                     C, C.stride(0), 0, 0, 0, 0, 0, 1, ws, wsb)
    else:
        st = lib.sgemm_batched_ex(mode, M, N, K, alpha, A, A.stride(0), B, B.stride(0), 0.0, C,
                                  C.stride(0), 0, 0, 0, 0, 0, 1)
    assert st == lib.SGEMM_OK, lib.sgemm_status_string(st)
    assert lib.sgemm_poll_error(None) == lib.SGEMM_OK


def sample(M, seed):
    rng = np.random.default_rng(seed)
    rows = {0, M - 1, M - 2, (2 ** 31) // 32768, M // 2}
    rows |= set(int(x) for x in rng.integers(0, M, 12))
    return sorted(r for r in rows if 0 <= r < M)


@pytest.mark.parametrize("api", ["ex", "ws"])
@pytest.mark.parametrize("mode", MODES)
def test_output_past_2_pow_31_elements(oracle_mod, mode, api):
    """C of 70000 x 32768 = 2.29e9 elements (9.2 GB), K = 16."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    M, N, K = 70000, 32768, 16
    A = int_tensor((M, K), 1, dev)
    B = int_tensor((K, N), 2, dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    assert C.numel() > 2 ** 31
    run(lib, mode, api, M, N, K, A, B, C, 2.0)
    rows = sample(M, 3)
    idx = torch.tensor(rows, device=dev)
    check_rows(oracle_mod, A[idx].cpu().numpy(), B.cpu().numpy(), C[idx].cpu().numpy(), 2.0)
    del A, B, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("api", ["ex", "ws"])
@pytest.mark.parametrize("mode", MODES)
def test_a_operand_past_2_pow_31_elements(oracle_mod, mode, api):
    """A of 70000 x 32768 = 2.29e9 elements (9.2 GB), N = 24 (the last tile
    column ragged), every partial sum below 2**24 (|a*b| <= 64, K = 32768
    gives at most 2**21)."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    M, N, K = 70000, 24, 32768
    A = int_tensor((M, K), 4, dev)
    B = int_tensor((K, N), 5, dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    assert A.numel() > 2 ** 31
    run(lib, mode, api, M, N, K, A, B, C, 1.0)
    rows = sample(M, 6)
    idx = torch.tensor(rows, device=dev)
    check_rows(oracle_mod, A[idx].cpu().numpy(), B.cpu().numpy(), C[idx].cpu().numpy(), 1.0)
    del A, B, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tB", [1, 0])
def test_half_path_past_2_pow_31_elements(oracle_mod, tB):
    """The 16-bit-input path: C of 70000 x 32768 (> 2^31 elements) with K =
    64, and A of 70000 x 32768 bf16 values (> 2^31) with N = 24; B read
    directly (tB = 1) or copied transposed (tB = 0).  Integer data, sampled
    rows bit-exact."""
    import torch
    import workloads
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    for M, N, K, seed in ((70000, 32768, 64, 7), (70000, 24, 32768, 9)):
        A = int_tensor((M, K), seed, dev)
        B = int_tensor((K, N), seed + 1, dev)
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
        assert max(A.numel(), C.numel()) > 2 ** 31
        Ah = A.to(torch.bfloat16)
        Bh = (B.t().contiguous() if tB else B).to(torch.bfloat16)
        ldb = K if tB else N
        wsb = lib.sgemm_half_workspace_size("bf16", M, N, K, 0, tB, K, ldb, 1)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        st = lib.sgemm_half_batched("bf16", M, N, K, 1.0, Ah, K, Bh, ldb, 0.0, C, N, 0, tB, 0, 0,
                                    0, 1, ws, wsb)
        assert st == lib.SGEMM_OK, lib.sgemm_status_string(st)
        assert lib.sgemm_poll_error(None) == lib.SGEMM_OK
        rows = sample(M, seed + 2)
        idx = torch.tensor(rows, device=dev)
        check_rows(oracle_mod, A[idx].cpu().numpy(), B.cpu().numpy(), C[idx].cpu().numpy(), 1.0)
        del A, B, C, Ah, Bh, ws
        torch.cuda.empty_cache()
