"""Helpers shared by the GPU parity tests: lay out logical matrices in the
library's storage conventions, run the library through the C ABI, and run
the oracle on the very same buffers."""
from __future__ import annotations

import numpy as np

TOL = {"fp32": 2e-5, "3xtf32": 2e-5, "tf32": 2e-3}


def layout(mat: np.ndarray, trans: bool, pad: int = 0, offset: int = 0):
    """Store a logical (Q x) R x Cc float32 matrix row-major, transposed when
    `trans`, with leading dimension = stored row length + pad, and the whole
    buffer shifted by `offset` elements.  Returns (flat, ld, stride, offset)."""
    m = mat if mat.ndim == 3 else mat[None]
    if trans:
        m = np.swapaxes(m, 1, 2)
    Q, R, Cc = m.shape
    ld = Cc + pad
    stride = R * ld
    buf = np.full(offset + Q * stride + 1, np.float32(0.125), dtype=np.float32)
    view = buf[offset:offset + Q * stride].reshape(Q, R, ld)
    view[:, :, :Cc] = m
    return buf, ld, stride, offset


class Problem:
    """One GEMM call: logical A (Q,M,K), B (Q,K,N), C0 (Q,M,N) and storage."""

    def __init__(self, A, B, C0, alpha, beta, transA=0, transB=0, pads=(0, 0, 0),
                 offsets=(0, 0, 0), strideA=None, strideB=None):
        A = A if A.ndim == 3 else A[None]
        B = B if B.ndim == 3 else B[None]
        C0 = C0 if C0.ndim == 3 else C0[None]
        self.Q, self.M, self.K = A.shape
        self.N = B.shape[2]
        self.alpha, self.beta = np.float32(alpha), np.float32(beta)
        self.transA, self.transB = int(transA), int(transB)
        self.Abuf, self.lda, sA, self.offA = layout(A, transA, pads[0], offsets[0])
        self.Bbuf, self.ldb, sB, self.offB = layout(B, transB, pads[1], offsets[1])
        self.Cbuf, self.ldc, sC, self.offC = layout(C0, False, pads[2], offsets[2])
        self.sA = sA if strideA is None else strideA
        self.sB = sB if strideB is None else strideB
        self.sC = sC

    def run_gpu(self, mode: str, api: str = "ex", stream=None, ws_bytes=None, ws_fill=None):
        """Runs the library on the device and returns C as (Q, M, N) float32.
        api="ws" passes a split-K workspace of ws_bytes (default: the size the
        library asks for), every byte set to ws_fill first when given."""
        import torch
        import dense_fp32_matrix_03_gb300 as lib
        dev = torch.device("cuda", 0)
        A = torch.from_numpy(self.Abuf).to(dev)
        B = torch.from_numpy(self.Bbuf).to(dev)
        C = torch.from_numpy(self.Cbuf).to(dev)
        pa = A.data_ptr() + 4 * self.offA
        pb = B.data_ptr() + 4 * self.offB
        pc = C.data_ptr() + 4 * self.offC
        if api == "ws":
            if ws_bytes is None:
                ws_bytes = lib.sgemm_workspace_size(mode, self.M, self.N, self.K, self.Q)
            ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
            if ws_fill is not None:
                ws.fill_(ws_fill)
            self.last_ws_bytes = ws_bytes
            self.last_ws = ws
            st = lib.sgemm_batched_ex_ws(mode, self.M, self.N, self.K, self.alpha, pa, self.lda,
                                         pb, self.ldb, self.beta, pc, self.ldc, self.transA,
                                         self.transB, self.sA, self.sB, self.sC, self.Q, ws,
                                         ws_bytes, stream)
        elif api == "noalloc":
            st = lib.sgemm_batched_ex_noalloc(mode, self.M, self.N, self.K, self.alpha, pa,
                                              self.lda, pb, self.ldb, self.beta, pc, self.ldc,
                                              self.transA, self.transB, self.sA, self.sB,
                                              self.sC, self.Q, stream)
        elif api == "sgemm_ex":
            assert self.Q == 1 and not self.transA and not self.transB
            st = lib.sgemm_ex(mode, self.M, self.N, self.K, self.alpha, pa, self.lda, pb,
                              self.ldb, self.beta, pc, self.ldc, stream)
        elif api == "sgemm":
            assert self.Q == 1 and not self.transA and not self.transB
            assert lib.sgemm_get_default_mode() == lib.MODES[mode]
            st = lib.sgemm(self.M, self.N, self.K, self.alpha, pa, self.lda, pb, self.ldb,
                           self.beta, pc, self.ldc, stream)
        else:
            st = lib.sgemm_batched_ex(mode, self.M, self.N, self.K, self.alpha, pa, self.lda,
                                      pb, self.ldb, self.beta, pc, self.ldc, self.transA,
                                      self.transB, self.sA, self.sB, self.sC, self.Q, stream)
        assert st == lib.SGEMM_OK, lib.sgemm_status_string(st)
        assert lib.sgemm_poll_error(stream) == lib.SGEMM_OK
        out = C.cpu().numpy()
        return self.extract(out)

    def extract(self, flat):
        v = flat[self.offC:self.offC + self.Q * self.sC].reshape(self.Q, self.M, self.ldc)
        return v[:, :, :self.N].copy()

    def oracle(self, oracle_mod, rows=None):
        """C_ref and D from the oracle on the same buffers ((Q,M,N) or rows)."""
        Cref, D = oracle_mod.sgemm_ref(
            self.M, self.N, self.K, self.alpha, self.Abuf[self.offA:], self.lda,
            self.Bbuf[self.offB:], self.ldb, self.beta, self.Cbuf[self.offC:], self.ldc,
            transA=self.transA, transB=self.transB, strideA=self.sA, strideB=self.sB,
            strideC=self.sC, Q=self.Q, rows=rows)
        if rows is None and self.Q == 1:
            Cref, D = Cref[None], D[None]
        return Cref, D


def sample_rows(Q: int, M: int, n: int, seed: int = 0, tile: int = 128):
    """(q, i) rows to check at full size: the first and last rows, rows around
    tile boundaries and the ragged last tile, plus random rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for q in {0, Q - 1}:
        for i in (0, 1, M - 1, M - 2, min(tile - 1, M - 1), min(tile, M - 1),
                  (M // tile) * tile - 1 if M > tile else 0, ((M - 1) // tile) * tile):
            if 0 <= i < M:
                rows.add((q, i))
    while len(rows) < n:
        rows.add((int(rng.integers(Q)), int(rng.integers(M))))
    return sorted(rows)
