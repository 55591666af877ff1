"""Python binding of libsgemm_gb300.so: single-precision GEMM on one GB300.

A thin ctypes layer over the C ABI in include/sgemm.h, with the same names:
it only marshals arguments (a torch tensor is passed by its data_ptr(), a
torch stream by its cuda_stream handle) and returns the C status code.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback: the first call fails loudly (ImportError) if the library has not
been built.

    C = alpha * op(A) @ op(B) + beta * C        (row-major, fp32)

Build the library with `python -m dense_fp32_matrix_03_gb300.build`.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libsgemm_gb300.so")

SGEMM_OK = 0
SGEMM_ERR_INVALID_ARG = 1
SGEMM_ERR_UNSUPPORTED = 2
SGEMM_ERR_LAUNCH = 3
SGEMM_ERR_TIMEOUT = 4
SGEMM_ERR_SCRATCH_LIMIT = 5

SGEMM_PROBE_FFMA = 0
SGEMM_PROBE_FFMA2 = 1
SGEMM_PROBE_TF32_SS = 2
SGEMM_PROBE_TF32_TS = 3
SGEMM_PROBE_BF16_SS = 4
PROBES = {"ffma": SGEMM_PROBE_FFMA, "ffma2": SGEMM_PROBE_FFMA2, "tf32_ss": SGEMM_PROBE_TF32_SS,
          "tf32_ts": SGEMM_PROBE_TF32_TS, "bf16_ss": SGEMM_PROBE_BF16_SS}

SGEMM_HALF_BF16 = 0
SGEMM_HALF_FP16 = 1
HALF_TYPES = {"bf16": SGEMM_HALF_BF16, "fp16": SGEMM_HALF_FP16}

SGEMM_ROUTE_AUTO = 0
SGEMM_ROUTE_SMALL = 1
SGEMM_ROUTE_PAIR = 2
SGEMM_ROUTE_DIRECT = 3
SGEMM_ROUTE_PLANES = 4
SGEMM_ROUTE_RAW = 5
SGEMM_ROUTE_INLINE = 6
SGEMM_ROUTE_MODELS = 7
ROUTES = {"auto": SGEMM_ROUTE_AUTO, "small": SGEMM_ROUTE_SMALL, "pair": SGEMM_ROUTE_PAIR,
          "direct": SGEMM_ROUTE_DIRECT, "planes": SGEMM_ROUTE_PLANES, "raw": SGEMM_ROUTE_RAW,
          "inline": SGEMM_ROUTE_INLINE, "models": SGEMM_ROUTE_MODELS}

SGEMM_MODE_DEFAULT = -1
SGEMM_MODE_FP32 = 0
SGEMM_MODE_3XTF32 = 1
SGEMM_MODE_TF32 = 2
MODES = {"fp32": SGEMM_MODE_FP32, "3xtf32": SGEMM_MODE_3XTF32, "tf32": SGEMM_MODE_TF32}

# Exported symbols declared in include/sgemm.h: name -> (restype, argtypes)
_i, _f, _p, _ll = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_longlong
SIGNATURES = {
    "sgemm": (_i, [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]),
    "sgemm_ex": (_i, [_i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]),
    "sgemm_batched": (_i, [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i, _i, _ll, _ll, _ll,
                           _i, _p]),
    "sgemm_batched_ex": (_i, [_i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i, _i, _ll, _ll,
                              _ll, _i, _p]),
    "sgemm_workspace_size": (ctypes.c_size_t, [_i, _i, _i, _i, _i]),
    "sgemm_batched_ex_ws": (_i, [_i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i, _i, _ll, _ll,
                                 _ll, _i, _p, ctypes.c_size_t, _p]),
    "sgemm_batched_ex_noalloc": (_i, [_i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i, _i, _ll,
                                      _ll, _ll, _i, _p]),
    "sgemm_half_workspace_size": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i, _i, _i, _i]),
    "sgemm_half_batched": (_i, [_i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i, _i, _ll, _ll,
                                _ll, _i, _p, ctypes.c_size_t, _p]),
    "sgemm_host_buffer_size": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i, _i]),
    "sgemm_host": (_i, [_i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i, _i, _i, _p,
                        ctypes.c_size_t, _p]),
    "sgemm_peak_probe": (_i, [_i, _ll, ctypes.POINTER(ctypes.c_double), _p]),
    "sgemm_tune_force": (_i, [_i]),
    "sgemm_tune_route": (_i, [_i, _i, _i, _i, _i]),
    "sgemm_set_default_mode": (_i, [_i]),
    "sgemm_get_default_mode": (_i, []),
    "sgemm_status_string": (ctypes.c_char_p, [_i]),
    "sgemm_poll_error": (_i, [_p]),
    "sgemm_selftest_wait_timeout": (_i, [_ll, _p]),
    "sgemm_kernel_launches": (ctypes.c_ulonglong, []),
    "sgemm_last_split_count": (_i, []),
    "sgemm_version": (_i, []),
    # include/linear_attention.h
    "la_state_bytes": (ctypes.c_size_t, [_i, _i, _i, _i]),
    "la_chunk_state": (_i, [_i, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p]),
    "la_chunk_output": (_i, [_i, _i, _i, _i, _f, _p, _p, _p, _p, _p, _p, _p]),
    "la_chunk_fused": (_i, [_i, _i, _i, _i, _f, _p, _p, _p, _p, _p, _p, _p, _p]),
}


class SgemmError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(f"sgemm status {status}: {sgemm_status_string(status)}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m dense_fp32_matrix_03_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


class _Lazy:
    """Opens the library on first use, so that the build module of this
    package can be imported before the library exists."""

    def __init__(self):
        self._h = None

    def __getattr__(self, name):
        if self._h is None:
            self._h = _load()
        return getattr(self._h, name)


_lib = _Lazy()


def load():
    """Open the library now (raises ImportError if it was not built)."""
    return _lib.sgemm_version


def _ptr(x):
    """Device address of a tensor (data_ptr) or a raw integer address."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    """cudaStream_t of a torch stream, a raw handle, or torch's current stream
    when None (0, the legacy default stream, without torch)."""
    if s is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s) or None


def sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    return _lib.sgemm(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                      _stream(stream))


def sgemm_ex(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_ex(mode, M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                         _stream(stream))


def sgemm_batched(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, strideA,
                  strideB, strideC, Q, stream=None) -> int:
    return _lib.sgemm_batched(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                              int(transA), int(transB), strideA, strideB, strideC, Q,
                              _stream(stream))


def sgemm_batched_ex(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
                     strideA, strideB, strideC, Q, stream=None) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_batched_ex(mode, M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                                 _ptr(C), ldc, int(transA), int(transB), strideA, strideB,
                                 strideC, Q, _stream(stream))


def sgemm_workspace_size(mode, M, N, K, Q=1) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return int(_lib.sgemm_workspace_size(mode, M, N, K, Q))


def sgemm_batched_ex_ws(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
                        strideA, strideB, strideC, Q, workspace, workspace_bytes,
                        stream=None) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_batched_ex_ws(mode, M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                                    _ptr(C), ldc, int(transA), int(transB), strideA, strideB,
                                    strideC, Q, _ptr(workspace), int(workspace_bytes),
                                    _stream(stream))


def sgemm_batched_ex_noalloc(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
                             strideA, strideB, strideC, Q, stream=None) -> int:
    """Split-K GEMM whose scratch is a fixed array inside the library: for
    callers that may not allocate device memory (see include/sgemm.h)."""
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_batched_ex_noalloc(mode, M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                                         _ptr(C), ldc, int(transA), int(transB), strideA, strideB,
                                         strideC, Q, _stream(stream))


def sgemm_half_workspace_size(type_, M, N, K, transA, transB, lda, ldb, Q=1) -> int:
    if isinstance(type_, str):
        type_ = HALF_TYPES[type_]
    return int(_lib.sgemm_half_workspace_size(type_, M, N, K, int(transA), int(transB), lda, ldb,
                                              Q))


def sgemm_half_batched(type_, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB,
                       strideA, strideB, strideC, Q, workspace, workspace_bytes,
                       stream=None) -> int:
    """A, B: device buffers of 16-bit values (torch bfloat16 / float16 tensors
    or raw addresses); C fp32 (see include/sgemm.h)."""
    if isinstance(type_, str):
        type_ = HALF_TYPES[type_]
    return _lib.sgemm_half_batched(type_, M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                                   _ptr(C), ldc, int(transA), int(transB), strideA, strideB,
                                   strideC, Q, _ptr(workspace), int(workspace_bytes),
                                   _stream(stream))


def sgemm_host_buffer_size(mode, M, N, K, transA=0, transB=0, panel_rows=0) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return int(_lib.sgemm_host_buffer_size(mode, M, N, K, int(transA), int(transB), panel_rows))


def sgemm_host(mode, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, transA, transB, panel_rows,
               dev, dev_bytes, stream=None) -> int:
    """A, B, C: host buffers (CPU tensors, ideally pinned, or raw addresses);
    dev: the device buffer (see include/sgemm.h)."""
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_host(mode, M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                           int(transA), int(transB), panel_rows, _ptr(dev), int(dev_bytes),
                           _stream(stream))


def sgemm_peak_probe(kind, iters, stream=None):
    """(status, flops) of one probe launch on `stream`."""
    if isinstance(kind, str):
        kind = PROBES[kind]
    flops = ctypes.c_double(0.0)
    st = _lib.sgemm_peak_probe(kind, iters, ctypes.byref(flops), _stream(stream))
    return st, flops.value


def sgemm_tune_force(route) -> int:
    """Process-wide forced kernel route (measurement; see include/sgemm.h)."""
    if isinstance(route, str):
        route = ROUTES[route]
    return _lib.sgemm_tune_force(route)


def sgemm_tune_route(mode, M, N, K, Q=1) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_tune_route(mode, M, N, K, Q)


def sgemm_set_default_mode(mode) -> int:
    if isinstance(mode, str):
        mode = MODES[mode]
    return _lib.sgemm_set_default_mode(mode)


def sgemm_get_default_mode() -> int:
    return _lib.sgemm_get_default_mode()


def sgemm_status_string(status: int) -> str:
    return _lib.sgemm_status_string(status).decode()


def sgemm_poll_error(stream=None) -> int:
    return _lib.sgemm_poll_error(_stream(stream))


def sgemm_selftest_wait_timeout(wait_cycles: int, stream=None) -> int:
    return _lib.sgemm_selftest_wait_timeout(wait_cycles, _stream(stream))


def sgemm_kernel_launches() -> int:
    return int(_lib.sgemm_kernel_launches())


def sgemm_last_split_count() -> int:
    return int(_lib.sgemm_last_split_count())


def sgemm_version() -> int:
    return _lib.sgemm_version()


# ---- chunked linear attention (include/linear_attention.h)

def la_state_bytes(BH, T, DK, DV) -> int:
    return int(_lib.la_state_bytes(BH, T, DK, DV))


def la_chunk_state(BH, T, DK, DV, k, v, g, h0, h, state_out, stream=None) -> int:
    return _lib.la_chunk_state(BH, T, DK, DV, _ptr(k), _ptr(v), _ptr(g), _ptr(h0), _ptr(h),
                               _ptr(state_out), _stream(stream))


def la_chunk_output(BH, T, DK, DV, scale, q, k, v, g, h, o, stream=None) -> int:
    return _lib.la_chunk_output(BH, T, DK, DV, scale, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                _ptr(h), _ptr(o), _stream(stream))


def la_chunk_fused(BH, T, DK, DV, scale, q, k, v, g, h0, o, state_out, stream=None) -> int:
    return _lib.la_chunk_fused(BH, T, DK, DV, scale, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(h0), _ptr(o), _ptr(state_out), _stream(stream))


def check(status: int) -> None:
    """Raise SgemmError for a non-zero status."""
    if status != SGEMM_OK:
        raise SgemmError(status)
