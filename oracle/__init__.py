"""CPU oracle for single-precision GEMM -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this package.  The library (dense_fp32_matrix_03_gb300) never imports
it, and this package never imports the library: the two share no code.

The arithmetic lives in oracle_sgemm.c (plain C, fp64 accumulation); this
module compiles it with gcc and calls it through ctypes.  See oracle_sgemm.c
for the definition it follows and the readings taken where the pages are
silent.  Every function of the oracle is pinned by tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_sgemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_sgemm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle_sgemm.c (or another source given as src, which the
    mutation tests use) into a shared library with gcc, with OpenMP when the
    compiler supports it.  Returns the library path."""
    with _lock:
        if (not force and os.path.exists(out)
                and os.path.getmtime(out) >= os.path.getmtime(src)):
            return out
        os.makedirs(os.path.dirname(out), exist_ok=True)
        cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
        if cc is None:
            raise RuntimeError("oracle: no C compiler found (gcc/cc)")
        base = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                "-std=c99", src, "-lm"]
        tmp = out + f".tmp{os.getpid()}"
        r = subprocess.run(base[:-1] + ["-fopenmp", "-o", tmp, "-lm"],
                           capture_output=True, text=True)
        if r.returncode != 0:  # no OpenMP runtime: build the serial form
            r = subprocess.run(base + ["-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle: gcc failed:\n" + r.stderr)
        os.replace(tmp, out)
        return out


def load(path: str):
    """Open a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, fp, dp = ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_sgemm.argtypes = [
        ctypes.c_int, ctypes.c_int, i64, i64, i64, ctypes.c_float,
        fp, i64, i64, fp, i64, i64, ctypes.c_float, fp, i64, i64, i64,
        fp, i64, dp, dp]
    lib.oracle_sgemm.restype = ctypes.c_int
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def num_threads() -> int:
    """Threads the oracle's parallel loop uses (OMP_NUM_THREADS, else all)."""
    return int(_load().oracle_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def sgemm_ref(M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, *, transA=0, transB=0,
              strideA=0, strideB=0, strideC=0, Q=1, rows=None, lib=None):
    """C_ref and D (both float64) for C = alpha*op(A)@op(B) + beta*C0.

    A, B, C0 are flat-indexable float32 numpy buffers in the library's storage
    convention (row-major, leading dimensions lda/ldb/ldc in elements, batch
    q at q*strideX).  C0 may be None when beta == 0.

    rows=None: returns arrays of shape (Q, M, N) (or (M, N) when Q == 1).
    rows=[(q, i), ...]: returns arrays of shape (len(rows), N), one per row.
    lib: a library from load(); the default is the built oracle.
    """
    lib = _load() if lib is None else lib
    A = np.ascontiguousarray(A, dtype=np.float32).reshape(-1)
    B = np.ascontiguousarray(B, dtype=np.float32).reshape(-1)
    C0 = None if C0 is None else np.ascontiguousarray(C0, dtype=np.float32).reshape(-1)
    alpha, beta = np.float32(alpha), np.float32(beta)
    M, N, K, Q = int(M), int(N), int(K), int(Q)
    if rows is None:
        rows_arr, nrows = None, 0
        out_shape = (Q, M, N) if Q != 1 else (M, N)
        n_out = Q * M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
        if rows_arr.size and (rows_arr[:, 0].min() < 0 or rows_arr[:, 0].max() >= Q
                              or rows_arr[:, 1].min() < 0 or rows_arr[:, 1].max() >= M):
            raise ValueError("oracle: row index out of range")
        nrows = rows_arr.shape[0]
        out_shape = (nrows, N)
        n_out = nrows
    # bounds of what the loops read, checked here so the C code can trust them
    if n_out and N and K and alpha != 0:
        a_need = (Q - 1) * strideA + ((K - 1) * lda + M if transA else (M - 1) * lda + K)
        b_need = (Q - 1) * strideB + ((N - 1) * ldb + K if transB else (K - 1) * ldb + N)
        if a_need > A.size or b_need > B.size:
            raise ValueError("oracle: A or B buffer too small for the given shape")
    if n_out and N and beta != 0:
        if C0 is None or (Q - 1) * strideC + (M - 1) * ldc + N > C0.size:
            raise ValueError("oracle: C0 missing or too small")
    Cref = np.empty(n_out * N, dtype=np.float64)
    D = np.empty(n_out * N, dtype=np.float64)
    rc = lib.oracle_sgemm(int(transA), int(transB), M, N, K, alpha, _ptr(A), int(lda),
                          int(strideA), _ptr(B), int(ldb), int(strideB), beta, _ptr(C0),
                          int(ldc), int(strideC), Q, _ptr(rows_arr), nrows,
                          _ptr(Cref), _ptr(D))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm failed ({rc})")
    return Cref.reshape(out_shape), D.reshape(out_shape)


def max_rel_err(C, Cref, D) -> float:
    """The accuracy metric: max over entries of |C - C_ref| / (D + 1e-30).

    NaN anywhere in C where C_ref is finite counts as an infinite error."""
    C = np.asarray(C, dtype=np.float64)
    diff = np.abs(C - Cref)
    diff = np.where(np.isnan(diff) & ~np.isnan(Cref), np.inf, diff)
    if diff.size == 0:
        return 0.0
    return float(np.nanmax(diff / (D + 1e-30)))
