"""CPU-only checks of the C ABI: the library loads, exports every entry point
that include/sgemm.h declares, and rejects invalid arguments on the host
before touching a GPU."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_03_gb300 import build
    build.build()
    import dense_fp32_matrix_03_gb300 as m
    m.load()
    return m


def declared_functions():
    """Every function the headers under include/ declare."""
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:\w+\s+)+\**\s*(sgemm\w*|la_\w+)\s*\(", text,
                                flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("sgemm", "sgemm_ex", "sgemm_batched", "sgemm_batched_ex", "sgemm_poll_error",
                 "sgemm_status_string", "sgemm_set_default_mode", "la_chunk_state",
                 "la_chunk_output", "la_chunk_fused", "la_state_bytes"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert name in lib.SIGNATURES, f"binding lacks {name}"
    assert set(lib.SIGNATURES) == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.sgemm_version() >= 100
    for code in range(0, 5):
        assert lib.sgemm_status_string(code)
    assert lib.sgemm_status_string(99) == "unknown status"


def test_default_mode_roundtrip(lib):
    old = lib.sgemm_get_default_mode()
    try:
        for mode in (lib.SGEMM_MODE_3XTF32, lib.SGEMM_MODE_TF32, lib.SGEMM_MODE_FP32):
            assert lib.sgemm_set_default_mode(mode) == lib.SGEMM_OK
            assert lib.sgemm_get_default_mode() == mode
        assert lib.sgemm_set_default_mode(7) == lib.SGEMM_ERR_INVALID_ARG
        assert lib.sgemm_set_default_mode(lib.SGEMM_MODE_DEFAULT) == lib.SGEMM_ERR_INVALID_ARG
    finally:
        lib.sgemm_set_default_mode(old)


FAKE = 1 << 40  # a never-dereferenced, 16-byte aligned address


def ex(lib, **kw):
    a = dict(mode=0, M=8, N=8, K=8, alpha=1.0, A=FAKE, lda=8, B=FAKE, ldb=8, beta=0.0, C=FAKE,
             ldc=8, transA=0, transB=0, strideA=0, strideB=0, strideC=0, Q=1)
    a.update(kw)
    return lib.sgemm_batched_ex(a["mode"], a["M"], a["N"], a["K"], a["alpha"], a["A"], a["lda"],
                                a["B"], a["ldb"], a["beta"], a["C"], a["ldc"], a["transA"],
                                a["transB"], a["strideA"], a["strideB"], a["strideC"], a["Q"])


@pytest.mark.parametrize("bad", [
    dict(M=-1), dict(N=-1), dict(K=-1), dict(Q=-1),
    dict(lda=7), dict(ldb=7), dict(ldc=7),
    dict(transA=1, M=9, lda=8), dict(transB=1, K=9, ldb=8, lda=9),
    dict(C=0), dict(A=0), dict(B=0),
    dict(Q=2, strideC=7 * 8 + 7),          # batch outputs would overlap
    dict(Q=2, strideA=-1, strideC=64), dict(Q=2, strideB=-8, strideC=64),
    dict(mode=3), dict(mode=-2),
])
def test_invalid_arguments_are_rejected_before_any_launch(lib, bad):
    assert ex(lib, **bad) == lib.SGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("empty", [dict(M=0), dict(N=0), dict(Q=0),
                                   dict(M=0, C=0, A=0, B=0)])
def test_empty_problems_are_a_no_op(lib, empty):
    assert ex(lib, **empty) == lib.SGEMM_OK


def test_null_operands_allowed_when_not_read(lib):
    # alpha == 0 or K == 0: A and B are not read, so NULL passes validation.
    # Validation passes; without a GPU the call then reports UNSUPPORTED.
    rc = ex(lib, A=0, B=0, alpha=0.0)
    assert rc in (lib.SGEMM_OK, lib.SGEMM_ERR_UNSUPPORTED)
    rc = ex(lib, A=0, B=0, K=0, lda=1)
    assert rc in (lib.SGEMM_OK, lib.SGEMM_ERR_UNSUPPORTED)


def test_plain_sgemm_validates_too(lib):
    assert lib.sgemm(4, 4, 4, 1.0, FAKE, 3, FAKE, 4, 0.0, FAKE, 4) == lib.SGEMM_ERR_INVALID_ARG
    # the explicit-mode single GEMM: bad leading dimensions, a bad mode, NULL C
    assert lib.sgemm_ex(0, 4, 4, 4, 1.0, FAKE, 3, FAKE, 4, 0.0, FAKE, 4) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_ex(1, 4, 4, 4, 1.0, FAKE, 4, FAKE, 3, 0.0, FAKE, 4) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_ex(2, 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 3) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_ex(5, 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_ex(0, 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, 0, 4) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_ex(0, 0, 4, 4, 1.0, 0, 4, 0, 4, 0.0, 0, 4) == lib.SGEMM_OK
    assert lib.sgemm_batched(4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, 0, 0, 0, 0, 10, 2) \
        == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_selftest_wait_timeout(0) == lib.SGEMM_ERR_INVALID_ARG


def host(lib, **kw):
    a = dict(mode=0, M=8, N=8, K=8, alpha=1.0, A=FAKE, lda=8, B=FAKE, ldb=8, beta=0.0, C=FAKE,
             ldc=8, transA=0, transB=0, panel_rows=0, dev=FAKE, dev_bytes=1 << 20)
    a.update(kw)
    return lib.sgemm_host(a["mode"], a["M"], a["N"], a["K"], a["alpha"], a["A"], a["lda"], a["B"],
                          a["ldb"], a["beta"], a["C"], a["ldc"], a["transA"], a["transB"],
                          a["panel_rows"], a["dev"], a["dev_bytes"])


@pytest.mark.parametrize("bad", [
    dict(M=-1), dict(K=-1), dict(lda=7), dict(ldb=7), dict(ldc=7),
    dict(transA=1, M=9, lda=8), dict(transB=2), dict(panel_rows=-1),
    dict(C=0), dict(A=0), dict(B=0), dict(dev=0), dict(dev=FAKE + 16), dict(mode=5),
])
def test_host_entry_rejects_invalid_arguments(lib, bad):
    assert host(lib, **bad) == lib.SGEMM_ERR_INVALID_ARG


def test_host_entry_empty_is_a_no_op(lib):
    assert host(lib, M=0, A=0, B=0, C=0, dev=0) == lib.SGEMM_OK
    assert host(lib, N=0, A=0, B=0, C=0, dev=0) == lib.SGEMM_OK


def test_peak_probe_rejects_invalid_arguments(lib):
    assert lib.sgemm_peak_probe(7, 16)[0] == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_peak_probe(-1, 16)[0] == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_peak_probe("ffma", 0)[0] == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_peak_probe("ffma", (1 << 16) + 1)[0] == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_peak_probe("tf32_ss", (1 << 22) + 1)[0] == lib.SGEMM_ERR_INVALID_ARG
    assert lib._lib.sgemm_peak_probe(0, 16, None, None) == lib.SGEMM_ERR_INVALID_ARG


def half(lib, **kw):
    a = dict(type_=0, M=8, N=8, K=8, alpha=1.0, A=FAKE, lda=8, B=FAKE, ldb=8, beta=0.0, C=FAKE,
             ldc=8, transA=0, transB=1, strideA=0, strideB=0, strideC=0, Q=1, ws=0, wsb=0)
    a.update(kw)
    return lib.sgemm_half_batched(a["type_"], a["M"], a["N"], a["K"], a["alpha"], a["A"],
                                  a["lda"], a["B"], a["ldb"], a["beta"], a["C"], a["ldc"],
                                  a["transA"], a["transB"], a["strideA"], a["strideB"],
                                  a["strideC"], a["Q"], a["ws"], a["wsb"])


@pytest.mark.parametrize("bad", [
    dict(type_=2), dict(type_=-1), dict(M=-1), dict(lda=7), dict(ldb=7), dict(ldc=7),
    dict(C=0), dict(A=0), dict(B=0), dict(ws=FAKE + 16, wsb=1024), dict(ws=0, wsb=1024),
    dict(Q=2, strideC=7),
])
def test_half_entry_rejects_invalid_arguments(lib, bad):
    assert half(lib, **bad) == lib.SGEMM_ERR_INVALID_ARG


def test_half_entry_empty_is_a_no_op(lib):
    assert half(lib, M=0, A=0, B=0, C=0) == lib.SGEMM_OK


def tune_table_entries():
    """(mode, class, batched) -> route, parsed from the committed header."""
    text = open(os.path.join(ROOT, "dense_fp32_matrix_03_gb300", "csrc", "tune_table.h")).read()
    out = {}
    for m in re.finditer(r"^\s*\{(-?\d+), (\d+), (\d+), (\d+)\},", text, flags=re.M):
        mode, cls, batched, route = map(int, m.groups())
        if mode >= 0:
            out[(mode, cls, batched)] = route
    return out


def test_tune_hooks_validate_arguments(lib):
    assert lib.sgemm_tune_force(8) == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_tune_force(-1) == lib.SGEMM_ERR_INVALID_ARG
    assert lib.sgemm_tune_route(7, 8, 8, 8, 1) == -1
    assert lib.sgemm_tune_route(0, -1, 8, 8, 1) == -1
    try:
        assert lib.sgemm_tune_force("direct") == lib.SGEMM_OK
        assert lib.sgemm_tune_route("tf32", 64, 64, 64, 1) == lib.SGEMM_ROUTE_DIRECT
        assert lib.sgemm_tune_route("fp32", 64, 64, 64, 1) == lib.SGEMM_ROUTE_AUTO
        assert lib.sgemm_tune_force("models") == lib.SGEMM_OK
        assert lib.sgemm_tune_route("fp32", 128, 128, 128, 1) == lib.SGEMM_ROUTE_AUTO
        assert lib.sgemm_tune_force("raw") == lib.SGEMM_OK
        assert lib.sgemm_tune_route("3xtf32", 64, 64, 64, 1) == lib.SGEMM_ROUTE_RAW
        assert lib.sgemm_tune_route("fp32", 64, 64, 64, 1) == lib.SGEMM_ROUTE_AUTO
    finally:
        assert lib.sgemm_tune_force("auto") == lib.SGEMM_OK


def test_route_lookup_follows_the_committed_table(lib):
    """For every mode and size class, single and batched, the route the
    library picks is the header's entry, or AUTO where it has none.  Shapes:
    M = N = K = 2^c (class c), and Q = 8 of M = N = K = 2^(c-1)."""
    table = tune_table_entries()
    for mode in (0, 1, 2):
        for cls in range(7, 14):
            for batched in (0, 1):
                n = 2 ** (cls - batched)
                Q = 8 if batched else 1
                want = table.get((mode, cls, batched), 0)
                if mode == 0 and want not in (0, 1):
                    want = 0
                if mode != 0 and want == 1:
                    want = 0
                assert lib.sgemm_tune_route(mode, n, n, n, Q) == want, (mode, cls, batched)


def test_linear_attention_rejects_invalid_arguments(lib):
    F = FAKE
    # head dimensions other than 64 / 128, negative sizes, too many heads
    for (BH, T, DK, DV) in [(1, 8, 32, 64), (1, 8, 64, 96), (-1, 8, 64, 64), (1, -1, 64, 64),
                            (65536, 8, 64, 64)]:
        assert lib.la_chunk_state(BH, T, DK, DV, F, F, None, None, F, None) == \
            lib.SGEMM_ERR_INVALID_ARG
        assert lib.la_chunk_output(BH, T, DK, DV, 1.0, F, F, F, None, F, F) == \
            lib.SGEMM_ERR_INVALID_ARG
        assert lib.la_chunk_fused(BH, T, DK, DV, 1.0, F, F, F, None, None, F, None) == \
            lib.SGEMM_ERR_INVALID_ARG
        assert lib.la_state_bytes(BH, T, DK, DV) == 0
    # NULL operands that are read or written; misaligned pointers
    assert lib.la_chunk_state(2, 8, 64, 64, 0, F, None, None, F, None) == lib.SGEMM_ERR_INVALID_ARG
    assert lib.la_chunk_state(2, 8, 64, 64, F, F, None, None, 0, None) == lib.SGEMM_ERR_INVALID_ARG
    assert lib.la_chunk_output(2, 8, 64, 64, 1.0, F, F, F, None, 0, F) == lib.SGEMM_ERR_INVALID_ARG
    assert lib.la_chunk_fused(2, 8, 64, 64, 1.0, F, F, F, None, None, 0, None) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.la_chunk_fused(2, 8, 64, 64, 1.0, F + 4, F, F, None, None, F, None) == \
        lib.SGEMM_ERR_INVALID_ARG
    assert lib.la_chunk_state(2, 8, 64, 64, F, F, F + 2, None, F, None) == \
        lib.SGEMM_ERR_INVALID_ARG
    # empty problems
    assert lib.la_chunk_fused(0, 8, 64, 64, 1.0, 0, 0, 0, None, None, 0, None) == lib.SGEMM_OK
    assert lib.la_chunk_output(3, 0, 64, 64, 1.0, 0, 0, 0, None, 0, 0) == lib.SGEMM_OK
    assert lib.la_state_bytes(2, 65, 128, 64) == 2 * 2 * 128 * 64 * 4
