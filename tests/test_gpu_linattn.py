"""GPU parity of the chunked linear-attention kernels (include/linear_attention.h)
against the fp64 oracle (oracle/linattn.py), element by element, through the
C ABI.

Accuracy metric, as for the SGEMM paths: |x - x_ref| / (D + 1e-30) <= 2e-5
for every output and chunk state, D the oracle's sum of the absolute values
of the terms (oracle.linattn.magnitudes); integer-valued inputs without
decay are exact in fp32 and must match bit for bit.  Shapes cover both head
dimensions, ragged last chunks, one-token and one-chunk sequences, an initial
state, no decay, and the benchmark workload (64 heads x 4096 tokens x 128),
the latter checked on sampled heads (heads are independent)."""
import numpy as np
import pytest

import workloads
from oracle import linattn

pytestmark = pytest.mark.gpu

TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_03_gb300 as lib
    lib.load()


def dev(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_chunked(q, k, v, g, h0, scale, want_state=True):
    """state pass then output pass; returns (o, h, state_out) on the host"""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    BH, T, DK = q.shape
    DV = v.shape[2]
    NT = -(-T // 64)
    dq, dk, dv, dg, dh0 = dev(q), dev(k), dev(v), dev(g), dev(h0)
    h = torch.full((BH, max(NT, 1), DK, DV), float("nan"), device="cuda")
    o = torch.full((BH, T, DV), float("nan"), device="cuda")
    so = torch.full((BH, DK, DV), float("nan"), device="cuda") if want_state else None
    assert lib.la_chunk_state(BH, T, DK, DV, dk, dv, dg, dh0, h, so) == lib.SGEMM_OK
    assert lib.la_chunk_output(BH, T, DK, DV, scale, dq, dk, dv, dg, h, o) == lib.SGEMM_OK
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    return (o.cpu().numpy(), h[:, :NT].cpu().numpy(),
            None if so is None else so.cpu().numpy())


def run_fused(q, k, v, g, h0, scale, want_state=True):
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    BH, T, DK = q.shape
    DV = v.shape[2]
    o = torch.full((BH, T, DV), float("nan"), device="cuda")
    so = torch.full((BH, DK, DV), float("nan"), device="cuda") if want_state else None
    assert lib.la_chunk_fused(BH, T, DK, DV, scale, dev(q), dev(k), dev(v), dev(g), dev(h0), o,
                              so) == lib.SGEMM_OK
    assert lib.sgemm_poll_error() == lib.SGEMM_OK
    return o.cpu().numpy(), None if so is None else so.cpu().numpy()


def check(q, k, v, g, h0, scale):
    o_ref, h_ref, s_ref = linattn.chunked(q, k, v, g, scale, h0, 64)
    Do, Dh, Ds = linattn.magnitudes(q, k, v, g, scale, h0, 64)
    o, h, s = run_chunked(q, k, v, g, h0, scale)
    errs = {"o": linattn.max_rel_err(o, o_ref, Do), "h": linattn.max_rel_err(h, h_ref, Dh),
            "state": linattn.max_rel_err(s, s_ref, Ds)}
    of, sf = run_fused(q, k, v, g, h0, scale)
    errs["o_fused"] = linattn.max_rel_err(of, o_ref, Do)
    errs["state_fused"] = linattn.max_rel_err(sf, s_ref, Ds)
    for name, e in errs.items():
        assert e <= TOL, f"{name}: {e:.3e}"
    return errs


@pytest.mark.parametrize("T", [1, 63, 64, 65, 300])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_chunked_and_fused_match_the_oracle(dk, dv, T):
    q, k, v, g, h0, scale = workloads.linattn_inputs(3, T, dk, dv, seed=T + dk + dv,
                                                     with_h0=True)
    check(q, k, v, g, h0, scale)


@pytest.mark.parametrize("decay,h0", [(False, False), (False, True), (True, False)])
def test_without_decay_or_initial_state(decay, h0):
    q, k, v, g, s0, scale = workloads.linattn_inputs(2, 200, 128, 128, seed=21, decay=decay,
                                                     with_h0=h0)
    check(q, k, v, g, s0, scale)


def test_small_workload():
    q, k, v, g, h0, scale = workloads.la_make("la_b2h2_t300_d64", with_h0=True)
    check(q, k, v, g, h0, scale)


def test_integer_inputs_without_decay_are_exact():
    rng = np.random.default_rng(5)
    BH, T, DK, DV = 2, 300, 128, 128
    q, k, v = (rng.integers(-3, 4, size=(BH, T, d)).astype(np.float32) for d in (DK, DK, DV))
    h0 = rng.integers(-3, 4, size=(BH, DK, DV)).astype(np.float32)
    o_ref, h_ref, s_ref = linattn.chunked(q, k, v, None, 1.0, h0, 64)
    o, h, s = run_chunked(q, k, v, None, h0, 1.0)
    assert np.array_equal(o.astype(np.float64), o_ref)
    assert np.array_equal(h.astype(np.float64), h_ref)
    assert np.array_equal(s.astype(np.float64), s_ref)
    of, sf = run_fused(q, k, v, None, h0, 1.0)
    assert np.array_equal(of.astype(np.float64), o_ref)
    assert np.array_equal(sf.astype(np.float64), s_ref)


def test_no_tokens_copies_the_initial_state():
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    h0 = torch.randn(3, 64, 128, device="cuda")
    so = torch.zeros(3, 64, 128, device="cuda")
    assert lib.la_chunk_state(3, 0, 64, 128, None, None, None, h0, None, so) == lib.SGEMM_OK
    torch.cuda.synchronize()
    assert torch.equal(so, h0)
    so.zero_()
    assert lib.la_chunk_fused(3, 0, 64, 128, 1.0, None, None, None, None, None, None, so) == \
        lib.SGEMM_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(so) == 0


def test_benchmark_workload_sampled_heads():
    """64 heads x 4096 tokens x 128: the whole call on the GPU, every output
    of four sampled heads against the oracle run on those heads alone."""
    q, k, v, g, h0, scale = workloads.la_make("la_b4h16_t4096_d128")
    o, h, s = run_chunked(q, k, v, g, h0, scale)
    of, sf = run_fused(q, k, v, g, h0, scale)
    heads = [0, 17, 42, 63]
    sub = lambda x: None if x is None else x[heads]
    o_ref, h_ref, s_ref = linattn.chunked(sub(q), sub(k), sub(v), sub(g), scale, None, 64)
    Do, Dh, Ds = linattn.magnitudes(sub(q), sub(k), sub(v), sub(g), scale, None, 64)
    for name, x, ref, D in [("o", o[heads], o_ref, Do), ("h", h[heads], h_ref, Dh),
                            ("state", s[heads], s_ref, Ds), ("o_fused", of[heads], o_ref, Do),
                            ("state_fused", sf[heads], s_ref, Ds)]:
        e = linattn.max_rel_err(x, ref, D)
        assert e <= TOL, f"{name}: {e:.3e}"
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(of))
