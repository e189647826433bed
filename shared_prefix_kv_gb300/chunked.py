"""Python binding of the prefill-chunk expansion (include/psattn_chunked.h).

Argument marshalling only; the expansion runs in the library.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib, PsattnError, Shape

EXPORTED_SYMBOLS = ("psattn_chunked_expand", "psattn_chunked_expand_ragged")

_vp = ctypes.c_void_p
_lib.psattn_chunked_expand.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, _vp,
                                       _vp, _vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32]
_lib.psattn_chunked_expand.restype = ctypes.c_int
_lib.psattn_chunked_expand_ragged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32]
_lib.psattn_chunked_expand_ragged.restype = ctypes.c_int


def _i32(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return None if a is None or a.size == 0 else a.ctypes.data_as(_vp)


def expand(shape: Shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
           q_len, level_tokens: int = 256):
    """Returns (Shape, block_table [R'][maxb], group_of_req [R'], group_parent [G'],
    prefix_len [G'], suffix_len [R']) of the equivalent decode batch."""
    bt, gor, gpar = _i32(block_table), _i32(group_of_req), _i32(group_parent)
    plen, slen, ql = _i32(prefix_len), _i32(suffix_len), _i32(q_len)
    out_shape = Shape()
    args = [ctypes.byref(shape), _p(bt), _p(gor), _p(gpar), _p(plen), _p(slen), _p(ql),
            int(level_tokens), ctypes.byref(out_shape)]
    rc = _lib.psattn_chunked_expand(*args, None, None, None, None, None, 0, 0)
    if rc not in (0, -8):
        raise PsattnError(rc, "psattn_chunked_expand")
    R2, G2, maxb = out_shape.num_req, out_shape.num_groups, shape.max_blocks_per_req
    obt = np.zeros((max(R2, 1), maxb), np.int32)
    ogor, oslen = np.zeros(max(R2, 1), np.int32), np.zeros(max(R2, 1), np.int32)
    opar, oplen = np.zeros(max(G2, 1), np.int32), np.zeros(max(G2, 1), np.int32)
    rc = _lib.psattn_chunked_expand(*args, _p(obt), _p(ogor), _p(opar), _p(oplen), _p(oslen),
                                    R2, G2)
    if rc != 0:
        raise PsattnError(rc, "psattn_chunked_expand")
    return out_shape, obt[:R2], ogor[:R2], opar[:G2], oplen[:G2], oslen[:R2]


def expand_ragged(shape: Shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
                  q_len):
    """The ragged form: (Shape, block_table, group_of_req, group_parent, prefix_len,
    suffix_len, leaf_len) for psattn_plan_ragged (Plan(..., leaf_len=...))."""
    bt, gor, gpar = _i32(block_table), _i32(group_of_req), _i32(group_parent)
    plen, slen, ql = _i32(prefix_len), _i32(suffix_len), _i32(q_len)
    out_shape = Shape()
    args = [ctypes.byref(shape), _p(bt), _p(gor), _p(gpar), _p(plen), _p(slen), _p(ql),
            ctypes.byref(out_shape)]
    rc = _lib.psattn_chunked_expand_ragged(*args, None, None, None, None, None, None, 0, 0)
    if rc not in (0, -8):
        raise PsattnError(rc, "psattn_chunked_expand_ragged")
    R2, G2, maxb = out_shape.num_req, out_shape.num_groups, shape.max_blocks_per_req
    obt = np.zeros((max(R2, 1), maxb), np.int32)
    ogor, oslen, oleaf = (np.zeros(max(R2, 1), np.int32) for _ in range(3))
    opar, oplen = np.zeros(max(G2, 1), np.int32), np.zeros(max(G2, 1), np.int32)
    rc = _lib.psattn_chunked_expand_ragged(*args, _p(obt), _p(ogor), _p(opar), _p(oplen),
                                           _p(oslen), _p(oleaf), R2, G2)
    if rc != 0:
        raise PsattnError(rc, "psattn_chunked_expand_ragged")
    return out_shape, obt[:R2], ogor[:R2], opar[:G2], oplen[:G2], oslen[:R2], oleaf[:R2]

