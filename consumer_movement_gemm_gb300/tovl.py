"""ctypes binding of libtovl.so (include/tovl.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  Functions keep the C names; tensors are passed as raw device
pointers taken from torch tensors, which serve only as device memory and
streams.  If the library is missing or cannot load, every call raises
``TovlError`` -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtovl.so")

TOVL_OK = 0
TOVL_ERR_INVALID = 1
TOVL_ERR_UNSUPPORTED = 2
TOVL_ERR_CUDA = 3
TOVL_ERR_TIMEOUT = 4
TOVL_ERR_OOM = 5
TOVL_COPY_VECTOR = 0
TOVL_COPY_BULK = 1
TOVL_COPY_AUTO = 2

OPT_PRODUCERS = 1
OPT_CONSUMERS = 2
OPT_COPY_MODE = 3
OPT_STATS = 4
OPT_TIMEOUT_NS = 5
OPT_COPY_CTAS = 6
OPT_COPY_WAITERS = 7
OPT_FAULT_GATE_OFFSET = 8
OPT_K_SLICES = 9
OPT_PAIRS = 10
OPT_MAX_PAIRS = 11
OPT_COOP_PAIRS = 12
OPT_COOPERATIVE = 13
OPT_PRODUCER_MODE = 14
OPT_PDL = 15
OPT_ROLE_SWITCH = 16
OPT_DISPATCH_ALIGN = 17
OPT_EMBEDDED = 18
OPT_RS_EPILOGUE = 19
OPT_L2_HINTS = 20
OPT_WIDE_TILES = 23


class TovlError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        self.code = code
        msg = f"{what}: {error_string(code) if _lib else code}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class tovl_config(ctypes.Structure):
    _fields_ = [
        ("device", ctypes.c_int),
        ("chunk_rows", ctypes.c_int),
        ("gate_rows", ctypes.c_int),
        ("producer_ctas", ctypes.c_int),
        ("consumer_ctas", ctypes.c_int),
        ("wait_timeout_ns", ctypes.c_longlong),
        ("copy_mode", ctypes.c_int),
        ("max_rows", ctypes.c_longlong),
        ("max_pairs", ctypes.c_int),
        ("max_experts", ctypes.c_int),
        ("k_slices", ctypes.c_int),
    ]


# every exported symbol of include/tovl.h with its ctypes signature
_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
_IP = ctypes.POINTER(ctypes.c_int)
_LLP = ctypes.POINTER(ctypes.c_longlong)
_ULLP = ctypes.POINTER(ctypes.c_ulonglong)
SIGNATURES = {
    "tovl_default_config": ([ctypes.POINTER(tovl_config), _I], None),
    "tovl_create": ([ctypes.POINTER(_P), ctypes.POINTER(tovl_config)], _I),
    "tovl_destroy": ([_P], _I),
    "tovl_gather_gemm": ([_P, ctypes.POINTER(_P), _I, _I, _I, _P, _I, _P, _P, _P], _I),
    "tovl_dispatch_rows": ([_I, _I, _I], _LL),
    "tovl_dispatch_rows_aligned": ([_I, _I, _I, _I], _LL),
    "tovl_dispatch_grouped_gemm": ([_P, _P, _I, _I, _P, _I, _I, _P, _I, _P, _P, _P, _P], _I),
    "tovl_combine": ([_P, _P, _I, _P, _P, _P, _P], _I),
    "tovl_gemm_reduce_scatter": ([_P, _P, _I, _I, _I, _P, _I, _P, _P, _P], _I),
    "tovl_gemm_only": ([_P, _P, _I, _I, _P, _I, _P, _P], _I),
    "tovl_copy_only": ([_P, ctypes.POINTER(_P), _I, _I, _I, _P, _P], _I),
    "tovl_gated_copy": ([_P, _P, _P, _LL, _I, _P, _I, _I, _P], _I),
    "tovl_sync_status": ([_P], _I),
    "tovl_ctrl_sizes": ([_P, _IP, _IP], _I),
    "tovl_read_ctrl": ([_P, _P, _P, _P, _LLP], _I),
    "tovl_read_plan": ([_P, _P, _P, _P, _P, _P, _IP], _I),
    "tovl_set_option": ([_P, _I, _LL], _I),
    "tovl_get_option": ([_P, _I, _LLP], _I),
    "tovl_read_stats": ([_P, _ULLP, _I], _I),
    "tovl_read_latency": ([_P, _P, _P, _I], _I),
    "tovl_read_trace": ([_P, _I, _P, _LL], _I),
    "tovl_dispatch_plan_noalloc": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "tovl_num_sms": ([_P], _I),
    "tovl_error_string": ([_I], ctypes.c_char_p),
    "tovl_last_error": ([_P], ctypes.c_char_p),
}

_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libtovl.so (built by ``build.py``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise TovlError(TOVL_ERR_UNSUPPORTED, "libtovl.so not built",
                                "run consumer_movement_gemm_gb300.build")
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def error_string(code: int) -> str:
    return load().tovl_error_string(code).decode()


def _check(h, rc: int, what: str):
    if rc != TOVL_OK:
        detail = load().tovl_last_error(h).decode() if h else ""
        raise TovlError(rc, what, detail)


def _ptr(t) -> int:
    """Device pointer of a torch tensor (or an int address)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def default_config(device: int = 0) -> tovl_config:
    cfg = tovl_config()
    load().tovl_default_config(ctypes.byref(cfg), device)
    return cfg


def dispatch_rows(T: int, k: int, E: int) -> int:
    return load().tovl_dispatch_rows(T, k, E)


def dispatch_rows_aligned(T: int, k: int, E: int, align: int) -> int:
    """Rows a dispatch buffer needs with expert segments aligned to ``align``."""
    return int(load().tovl_dispatch_rows_aligned(T, k, E, align))


def dispatch_plan_noalloc(topk, E: int, expert_offsets, dst_rows, stream=None) -> None:
    """Routing plan without allocating (library-owned fixed scratch)."""
    T, k = topk.shape
    rc = load().tovl_dispatch_plan_noalloc(_ptr(topk), T, k, E, _ptr(expert_offsets), _ptr(dst_rows),
                                           _stream(stream))
    _check(None, rc, "tovl_dispatch_plan_noalloc")


class Handle:
    """Owns one tovl handle (control plane + sequence number)."""

    def __init__(self, device: int = 0, **cfg_fields):
        cfg = default_config(device)
        for k, v in cfg_fields.items():
            setattr(cfg, k, v)
        h = ctypes.c_void_p()
        _check(None, load().tovl_create(ctypes.byref(h), ctypes.byref(cfg)), "tovl_create")
        self.h = h
        self.cfg = cfg

    def close(self):
        if getattr(self, "h", None):
            load().tovl_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # ------------------------------------------------------------ hot path
    def gather_gemm(self, shards, W, gathered, out, stream=None):
        """shards: list of [R, K] bf16 device tensors (or one [S, R, K] tensor)."""
        ptrs, S, R, K = _shard_ptrs(shards)
        rc = load().tovl_gather_gemm(self.h, ptrs, S, R, K, _ptr(W), W.shape[1], _ptr(gathered), _ptr(out),
                                     _stream(stream))
        _check(self.h, rc, "tovl_gather_gemm")

    def dispatch_grouped_gemm(self, x, topk, W, dispatched, expert_offsets, out, stream=None):
        T, H = x.shape
        k = topk.shape[1]
        E, _, N = W.shape
        rc = load().tovl_dispatch_grouped_gemm(self.h, _ptr(x), T, H, _ptr(topk), k, E, _ptr(W), N,
                                               _ptr(dispatched), _ptr(expert_offsets), _ptr(out),
                                               _stream(stream))
        _check(self.h, rc, "tovl_dispatch_grouped_gemm")

    # ------------------------------------------------------------ controls
    def gemm_only(self, A, W, out, stream=None):
        M, K = A.shape
        rc = load().tovl_gemm_only(self.h, _ptr(A), M, K, _ptr(W), W.shape[1], _ptr(out), _stream(stream))
        _check(self.h, rc, "tovl_gemm_only")

    def copy_only(self, shards, gathered, stream=None):
        ptrs, S, R, K = _shard_ptrs(shards)
        rc = load().tovl_copy_only(self.h, ptrs, S, R, K, _ptr(gathered), _stream(stream))
        _check(self.h, rc, "tovl_copy_only")

    def gemm_reduce_scatter(self, X, W, partials, out, stream=None):
        """Row-parallel layer on logical shards: ``partials[s] = X[s] @ W[s]``
        and ``out = sum_s partials[s]``.  X [S, M, Ks], W [S, Ks, N]."""
        S, M, Ks = X.shape
        N = W.shape[2]
        rc = load().tovl_gemm_reduce_scatter(self.h, _ptr(X), S, M, Ks, _ptr(W), N, _ptr(partials), _ptr(out),
                                             _stream(stream))
        _check(self.h, rc, "tovl_gemm_reduce_scatter")

    def combine(self, y, gate_w, staging, combined, stream=None):
        """Combine of the last dispatch round: ``staging[t*k+j] = y[dst(t,j)]``
        and ``combined[t] = bf16(sum_j gate_w[t,j] * staging[t*k+j])``."""
        N = y.shape[1]
        import torch
        if gate_w.dtype != torch.float32:
            raise TypeError("gate weights must be float32")
        rc = load().tovl_combine(self.h, _ptr(y), N, _ptr(gate_w), _ptr(staging), _ptr(combined), _stream(stream))
        _check(self.h, rc, "tovl_combine")

    def gated_copy(self, src, dst, perm, gated=True, stamps=False, stream=None):
        n, rb = src.shape
        rc = load().tovl_gated_copy(self.h, _ptr(src), _ptr(dst), n, rb * src.element_size(), _ptr(perm),
                                    1 if gated else 0, 1 if stamps else 0, _stream(stream))
        _check(self.h, rc, "tovl_gated_copy")

    # ------------------------------------------------------------ diagnostics
    def sync_status(self) -> int:
        return load().tovl_sync_status(self.h)

    def ctrl_sizes(self):
        a, b = ctypes.c_int(), ctypes.c_int()
        _check(self.h, load().tovl_ctrl_sizes(self.h, ctypes.byref(a), ctypes.byref(b)), "tovl_ctrl_sizes")
        return a.value, b.value

    def read_ctrl(self):
        import numpy as np
        nc, nb = self.ctrl_sizes()
        slots = np.zeros(nc, np.int32)
        cnts = np.zeros(nc, np.int32)
        rb = np.zeros(nb, np.int32)
        seq = ctypes.c_longlong()
        rc = load().tovl_read_ctrl(self.h, slots.ctypes.data, cnts.ctypes.data, rb.ctypes.data, ctypes.byref(seq))
        _check(self.h, rc, "tovl_read_ctrl")
        return slots, cnts, rb, seq.value

    def read_plan(self, T: int, k: int, E: int):
        import numpy as np
        rows = dispatch_rows_aligned(T, k, E, self.get_option(OPT_DISPATCH_ALIGN))
        counts = np.zeros(E, np.int32)
        dst = np.zeros(T * k, np.int32)
        src = np.zeros(max(rows, 1), np.int32)
        pad = np.zeros(max(rows // 128, 1), np.int32)
        blk = np.zeros(max(rows // 128, 1), np.int32)
        m_pad = ctypes.c_int()
        rc = load().tovl_read_plan(self.h, counts.ctypes.data, dst.ctypes.data, src.ctypes.data, pad.ctypes.data,
                                   blk.ctypes.data, ctypes.byref(m_pad))
        _check(self.h, rc, "tovl_read_plan")
        m = m_pad.value
        return counts, dst, src[:m].copy(), pad[:m // 128].copy(), blk[:m // 128].copy(), m

    def set_option(self, option: int, value: int):
        _check(self.h, load().tovl_set_option(self.h, option, int(value)), "tovl_set_option")

    def get_option(self, option: int) -> int:
        v = ctypes.c_longlong()
        _check(self.h, load().tovl_get_option(self.h, option, ctypes.byref(v)), "tovl_get_option")
        return v.value

    def read_stats(self):
        arr = (ctypes.c_ulonglong * 8)()
        _check(self.h, load().tovl_read_stats(self.h, arr, 8), "tovl_read_stats")
        return list(arr)

    def read_latency(self, n: int):
        import numpy as np
        pub = np.zeros(n, np.int64)
        obs = np.zeros(n, np.int64)
        rc = load().tovl_read_latency(self.h, pub.ctypes.data, obs.ctypes.data, n)
        _check(self.h, rc, "tovl_read_latency")
        return pub, obs

    def read_trace(self, what: int, n: int):
        import numpy as np
        out = np.zeros(n, np.int64)
        _check(self.h, load().tovl_read_trace(self.h, what, out.ctypes.data, n), "tovl_read_trace")
        return out

    @property
    def num_sms(self) -> int:
        return load().tovl_num_sms(self.h)


def _shard_ptrs(shards):
    if hasattr(shards, "dim") and shards.dim() == 3:
        shards = [shards[s] for s in range(shards.shape[0])]
    S = len(shards)
    R, K = shards[0].shape
    arr = (ctypes.c_void_p * S)(*[_ptr(s) for s in shards])
    return arr, S, R, K
