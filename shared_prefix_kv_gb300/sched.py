"""Python binding of the token-batch simulation (include/psattn_sched.h).

Argument marshalling only; the simulation runs in the library.  See the
header for the model it follows.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib, PsattnError, ERR_NOMEM

SCHED_REORDER = 1

EXPORTED_SYMBOLS = ("psattn_token_batches",)


class SchedParams(ctypes.Structure):
    _fields_ = [("n_chunk", ctypes.c_int32), ("m_threshold", ctypes.c_int64),
                ("max_requests", ctypes.c_int32), ("flags", ctypes.c_uint32)]


_vp = ctypes.c_void_p
_lib.psattn_token_batches.argtypes = [_vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int32, _vp,
                                      _vp, _vp, _vp, _vp, ctypes.c_int32, _vp]
_lib.psattn_token_batches.restype = ctypes.c_int


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))


def _p(a):
    return a.ctypes.data_as(_vp) if a.size else None


def token_batches(group_prefix, group_of_req, distinct_len, decode_len, n_chunk: int,
                  m_threshold: int = -1, max_requests: int = 0, reorder: bool = False):
    """Returns (group_order int32 [S], iter_tokens int32 [T, 4], iter_mem int64 [T])."""
    gp, gor = _i32(group_prefix), _i32(group_of_req)
    dl, ol = _i32(distinct_len), _i32(decode_len)
    prm = SchedParams(int(n_chunk), int(m_threshold), int(max_requests),
                      SCHED_REORDER if reorder else 0)
    order = np.zeros(max(1, gp.size + gor.size), np.int32)
    nsg, nit = ctypes.c_int32(0), ctypes.c_int32(0)
    cap = 1024
    while True:
        tok = np.zeros((cap, 4), np.int32)
        mem = np.zeros(cap, np.int64)
        rc = _lib.psattn_token_batches(_p(gp), gp.size, _p(gor), _p(dl), _p(ol), gor.size,
                                       ctypes.byref(prm), _p(order), ctypes.byref(nsg), _p(tok),
                                       _p(mem), cap, ctypes.byref(nit))
        if rc == ERR_NOMEM and nit.value > cap:
            cap = nit.value
            continue
        if rc != 0:
            raise PsattnError(rc, "psattn_token_batches")
        n = nit.value
        return order[:nsg.value].copy(), tok[:n].copy(), mem[:n].copy()
