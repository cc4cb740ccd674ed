"""CPU oracle for the tovl hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and this package imports nothing from
the product path.

The arithmetic lives in ``oracle.c`` (plain C loops, see its header for the
passages each function follows); this module only builds it with gcc and
marshals numpy arrays.  bf16 tensors cross this boundary as ``uint16`` bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CHUNK_ROWS = 64       # watermark granularity (sync-protocol page, section 4)
BLOCK_ROWS = 128      # GEMM gate granularity (row-block counter, section 5)


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-std=c11", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_int64
            sig = {
                "oracle_num_threads": ([], I),
                "oracle_set_num_threads": ([I], None),
                "oracle_bf16_to_f32": ([P, P, L], None),
                "oracle_f32_to_bf16": ([P, P, L], None),
                "oracle_gather": ([P, I, I, I, P], None),
                "oracle_dispatch": ([P, I, I, P, I, L, P], None),
                "oracle_copy_perm": ([P, L, I, P, P], None),
                "oracle_combine": ([P, I, P, P, I, I, P, P], None),
                "oracle_reduce_partials": ([P, I, L, I, P], None),
                "oracle_matmul_f32": ([P, P, I, I, I, P], None),
                "oracle_matmul_rows_f32": ([P, P, I, I, P, I, P], None),
                "oracle_grouped_matmul_f32": ([P, P, I, P, I, I, P], None),
                "oracle_gather_expected": ([L, I, I, P], None),
                "oracle_perm_expected": ([P, L, I, I, P], None),
                "oracle_dispatch_plan": ([P, I, I, I, I, L, P, P, P, P, P, P], I),
                "oracle_ctrl_state": ([L, I, I, I, I, P, P, P], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_to_f32(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, np.float32)
    _load().oracle_bf16_to_f32(_p(h), _p(out), h.size)
    return out


def f32_to_bf16(f) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().oracle_f32_to_bf16(_p(f), _p(out), f.size)
    return out


def gather(shards) -> np.ndarray:
    """``G[s*R + i] = shards[s][i]`` for a list of [R, K] uint16 arrays."""
    shards = [_u16(s) for s in shards]
    S = len(shards)
    R, K = shards[0].shape
    for s in shards:
        assert s.shape == (R, K)
    G = np.empty((S * R, K), np.uint16)
    table = (ctypes.c_void_p * S)(*[s.ctypes.data for s in shards])
    _load().oracle_gather(ctypes.cast(table, ctypes.c_void_p), S, R, K, _p(G))
    return G


def dispatch(x, dst, k: int, m_pad: int) -> np.ndarray:
    x = _u16(x)
    T, H = x.shape
    dst = np.ascontiguousarray(dst, dtype=np.int32)
    D = np.empty((m_pad, H), np.uint16)
    _load().oracle_dispatch(_p(x), T, H, _p(dst), k, m_pad, _p(D))
    return D


def combine(Y, dst, w):
    """Token-ordered staging ``S[t*k+j] = Y[dst[t*k+j]]`` and the combined
    rows ``C[t] = bf16(sum_j w[t,j] * S[t*k+j])`` (fp32 products and sums in
    ascending j).  ``Y`` is [rows, N] uint16 bf16 bits, ``dst`` the [T, k]
    (or flat) destination rows of the dispatch plan, ``w`` [T, k] fp32."""
    Y = _u16(Y)
    N = Y.shape[1]
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, k = w.shape
    dst = np.ascontiguousarray(dst, dtype=np.int32).reshape(-1)
    assert dst.size == T * k
    assert dst.size == 0 or (dst.min() >= 0 and dst.max() < Y.shape[0])
    S = np.empty((T * k, N), np.uint16)
    C = np.empty((T, N), np.uint16)
    _load().oracle_combine(_p(Y), N, _p(dst), _p(w), T, k, _p(S), _p(C))
    return S, C


def reduce_partials(P) -> np.ndarray:
    """``O[m] = bf16(sum_s f32(P[s, m]))``, fp32 sums in ascending s; ``P`` is
    [S, M, N] uint16 bf16 bits."""
    P = _u16(P)
    S, M, N = P.shape
    O = np.empty((M, N), np.uint16)
    _load().oracle_reduce_partials(_p(P), S, M, N, _p(O))
    return O


def gemm_reduce_scatter(X, W):
    """Row-parallel layer on logical shards: ``P_s = bf16(X_s W_s)`` (fp32
    accumulation, ascending k) and ``O = reduce_partials(P)``.  ``X`` is
    [S, M, Ks], ``W`` [S, Ks, N], both uint16 bf16 bits.  Returns (P, O)."""
    X = _u16(X)
    W = _u16(W)
    S, M, Ks = X.shape
    assert W.shape[0] == S and W.shape[1] == Ks
    P = np.stack([f32_to_bf16(matmul_f32(X[s], W[s])) for s in range(S)])
    return P, reduce_partials(P)


def copy_perm(src, perm) -> np.ndarray:
    src = np.ascontiguousarray(src, dtype=np.uint8)
    n, row_bytes = src.shape
    perm = np.ascontiguousarray(perm, dtype=np.int32)
    dst = np.empty_like(src)
    _load().oracle_copy_perm(_p(src), n, row_bytes, _p(perm), _p(dst))
    return dst


def matmul_f32(A, W) -> np.ndarray:
    A, W = _u16(A), _u16(W)
    M, K = A.shape
    K2, N = W.shape
    assert K == K2
    O = np.empty((M, N), np.float32)
    _load().oracle_matmul_f32(_p(A), _p(W), M, N, K, _p(O))
    return O


def matmul_rows_f32(A, W, rows) -> np.ndarray:
    A, W = _u16(A), _u16(W)
    M, K = A.shape
    K2, N = W.shape
    assert K == K2
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.min(initial=0) >= 0 and rows.max(initial=0) < M
    O = np.empty((rows.size, N), np.float32)
    _load().oracle_matmul_rows_f32(_p(A), _p(W), N, K, _p(rows), rows.size, _p(O))
    return O


def grouped_matmul_f32(D, W, off) -> np.ndarray:
    D, W = _u16(D), _u16(W)
    E, K, N = W.shape
    off = np.ascontiguousarray(off, dtype=np.int32)
    assert off.shape == (E + 1,) and D.shape[1] == K and D.shape[0] >= off[E]
    O = np.zeros((D.shape[0], N), np.float32)
    _load().oracle_grouped_matmul_f32(_p(D), _p(W), E, _p(off), N, K, _p(O))
    return O


def gather_expected(n_rows: int, chunk_rows: int = CHUNK_ROWS) -> np.ndarray:
    n_chunks = (n_rows + chunk_rows - 1) // chunk_rows
    out = np.empty(n_chunks, np.int32)
    _load().oracle_gather_expected(n_rows, chunk_rows, n_chunks, _p(out))
    return out


def perm_expected(perm, chunk_rows: int = CHUNK_ROWS) -> np.ndarray:
    perm = np.ascontiguousarray(perm, dtype=np.int32)
    n_chunks = (perm.size + chunk_rows - 1) // chunk_rows
    out = np.empty(n_chunks, np.int32)
    _load().oracle_perm_expected(_p(perm), perm.size, chunk_rows, n_chunks, _p(out))
    return out


class DispatchPlan:
    """Routing plan of one dispatch round (see ``oracle_dispatch_plan``)."""

    def __init__(self, counts, off, dst, src, pad, blk_e):
        self.counts, self.off, self.dst, self.src, self.pad, self.blk_e = \
            counts, off, dst, src, pad, blk_e

    @property
    def m_pad(self) -> int:
        return int(self.off[-1])

    @property
    def n_blocks(self) -> int:
        return int(self.pad.size)


def dispatch_plan(topk, E: int, block_rows: int = BLOCK_ROWS, max_rows: int | None = None) -> DispatchPlan:
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    T, k = topk.shape
    if max_rows is None:
        max_rows = T * k + E * (block_rows - 1)
    counts = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    dst = np.empty(T * k, np.int32)
    src = np.empty(max(max_rows, 1), np.int32)
    pad = np.empty(max(max_rows // block_rows, 1), np.int32)
    blk_e = np.empty_like(pad)
    nb = _load().oracle_dispatch_plan(_p(topk), T, k, E, block_rows, max_rows, _p(counts),
                                      _p(off), _p(dst), _p(src), _p(pad), _p(blk_e))
    if nb < 0:
        raise ValueError("routing has an expert id outside [0, E) or exceeds max_rows")
    m_pad = int(off[E])
    return DispatchPlan(counts, off, dst, src[:m_pad].copy(), pad[:nb].copy(), blk_e[:nb].copy())


def ctrl_state(R: int, n_chunks: int, n_blocks: int, chunk_rows: int = CHUNK_ROWS,
               block_rows: int = BLOCK_ROWS):
    slots = np.empty(n_chunks, np.int32)
    cnts = np.empty(n_chunks, np.int32)
    rbcnts = np.empty(n_blocks, np.int32)
    _load().oracle_ctrl_state(R, n_chunks, n_blocks, chunk_rows, block_rows, _p(slots),
                              _p(cnts), _p(rbcnts))
    return slots, cnts, rbcnts
