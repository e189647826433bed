"""CPU oracle for shared-prefix paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The
library (``shared_prefix_kv_gb300``) never imports it and shares no code with
it: the only thing both sides consume is the seeded input generator in
``workloads``.

The arithmetic lives in ``oracle.c`` (plain C, double precision, the
definition of paged attention written out: gather every token of the request
through its block table, softmax of the scaled scores, weighted sum of V).
This module compiles it with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# ORACLE_SRC_OVERRIDE points the oracle at another copy of oracle.c; the
# mutation test uses it to plant mistakes in a temporary copy and check that
# the pins catch them.
_SRC = os.environ.get("ORACLE_SRC_OVERRIDE") or os.path.join(_HERE, "oracle.c")
_OUT_DIR = (os.path.dirname(_SRC) if os.environ.get("ORACLE_SRC_OVERRIDE")
            else os.path.join(_HERE, "_build"))
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_req", ctypes.c_int32), ("num_groups", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("max_blocks_per_req", ctypes.c_int32), ("num_pool_blocks", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("scale", ctypes.c_double),
        ("q", ctypes.c_void_p), ("pool", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("group_of_req", ctypes.c_void_p),
        ("group_parent", ctypes.c_void_p), ("prefix_len", ctypes.c_void_p),
        ("suffix_len", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attention.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_gather_kv.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_longlong]
            lib.oracle_gather_kv.restype = ctypes.c_longlong
            lib.oracle_num_tokens.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int]
            lib.oracle_num_tokens.restype = ctypes.c_longlong
            lib.oracle_attention_chunked.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_int]
            lib.oracle_attention_chunked.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _c(a: Optional[np.ndarray], dtype) -> Optional[np.ndarray]:
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class _Marshalled:
    """Keeps the contiguous copies alive while C holds pointers to them."""

    def __init__(self, p, scale: Optional[float] = None):
        self.q = np.ascontiguousarray(p.q)
        self.pool = np.ascontiguousarray(p.pool)
        self.bt = _c(p.block_table, np.int32)
        self.gor = _c(p.group_of_req, np.int32)
        self.gpar = _c(p.group_parent, np.int32)
        self.plen = _c(p.prefix_len, np.int32)
        self.slen = _c(p.suffix_len, np.int32)
        s = _Problem()
        s.num_req = self.slen.shape[0]
        s.num_groups = self.plen.shape[0]
        s.num_q_heads = p.num_q_heads
        s.num_kv_heads = p.num_kv_heads
        s.head_dim = p.head_dim
        s.block_size = p.block_size
        s.max_blocks_per_req = self.bt.shape[1]
        s.num_pool_blocks = self.pool.shape[0]
        s.dtype = p.dtype
        s.scale = p.scale if scale is None else scale
        s.q = self.q.ctypes.data
        s.pool = self.pool.ctypes.data
        s.block_table = self.bt.ctypes.data
        s.group_of_req = self.gor.ctypes.data
        s.group_parent = None if self.gpar is None else self.gpar.ctypes.data
        s.prefix_len = self.plen.ctypes.data
        s.suffix_len = self.slen.ctypes.data
        self.s = s


def attention(p, requests: Optional[Sequence[int]] = None, nthreads: int = 0):
    """Oracle output for problem `p` (a ``workloads.Problem`` or anything with
    the same fields).  Returns (out [n][Hq][d] float64, lse [n][Hq] float64)
    for the listed requests (all when None)."""
    lib = _load()
    m = _Marshalled(p)
    req = None if requests is None else np.ascontiguousarray(requests, dtype=np.int32)
    n = m.s.num_req if req is None else req.shape[0]
    out = np.zeros((n, p.num_q_heads, p.head_dim), np.float64)
    lse = np.zeros((n, p.num_q_heads), np.float64)
    rc = lib.oracle_attention(ctypes.byref(m.s), None if req is None else req.ctypes.data,
                              n, out.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_attention failed with status {rc}")
    return out, lse


def attention_chunked(p, q_len, q, nthreads: int = 0):
    """Chunked prefill: request r of problem `p` carries q_len[r] queries,
    rows of `q` ([sum q_len][Hq][d], p's dtype) in request order; query i of
    request r attends causally to the first n_tok - q_len[r] + i + 1 tokens of
    its token list.  Returns (out [Q][Hq][d] float64, lse [Q][Hq] float64)."""
    lib = _load()
    m = _Marshalled(p)
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    qq = np.ascontiguousarray(q)
    if ql.shape[0] != m.s.num_req or qq.shape[0] != int(ql.sum()):
        raise OracleError("q_len / q rows do not match the problem")
    n = qq.shape[0]
    out = np.zeros((n, p.num_q_heads, p.head_dim), np.float64)
    lse = np.zeros((n, p.num_q_heads), np.float64)
    rc = lib.oracle_attention_chunked(ctypes.byref(m.s), ql.ctypes.data, qq.ctypes.data,
                                      out.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_attention_chunked failed with status {rc}")
    return out, lse


def gather_kv(p, r: int, kvh: int):
    """Dense K, V (float64 [n][d]) that request r reads for KV head kvh."""
    lib = _load()
    m = _Marshalled(p)
    n = lib.oracle_num_tokens(ctypes.byref(m.s), int(r))
    if n < 0:
        raise OracleError(f"oracle_num_tokens failed with status {n}")
    K = np.zeros((max(n, 1), p.head_dim), np.float64)
    V = np.zeros((max(n, 1), p.head_dim), np.float64)
    rc = lib.oracle_gather_kv(ctypes.byref(m.s), int(r), int(kvh), K.ctypes.data,
                              V.ctypes.data, max(n, 1))
    if rc < 0:
        raise OracleError(f"oracle_gather_kv failed with status {rc}")
    return K[:n], V[:n]


def max_threads() -> int:
    return int(_load().oracle_max_threads())
