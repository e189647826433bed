"""Python binding of the prefix-grouping calls (include/psattn_forest.h).

Argument marshalling only: the requests' token ids go in as a list of int
sequences (or one int32 array plus int64 offsets); every step runs in the
library.  See the header for what the calls compute.
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import numpy as np

from . import _lib, PsattnError

FOREST_SINGLE = 1

EXPORTED_SYMBOLS = ("psattn_forest_group", "psattn_cht_batches", "psattn_cht_group")

_vp = ctypes.c_void_p
_lib.psattn_forest_group.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_uint32,
                                     _vp, _vp, _vp, _vp, ctypes.c_int32, _vp, _vp]
_lib.psattn_forest_group.restype = ctypes.c_int
_lib.psattn_cht_batches.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, _vp, _vp, _vp]
_lib.psattn_cht_batches.restype = ctypes.c_int
_lib.psattn_cht_group.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                  ctypes.c_int32, ctypes.c_uint32, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, ctypes.c_int32, _vp, _vp]
_lib.psattn_cht_group.restype = ctypes.c_int


def pack(requests: Sequence[Sequence[int]]):
    """Token lists -> (tokens int32 [total], offsets int64 [R + 1])."""
    lens = [len(r) for r in requests]
    offsets = np.zeros(len(requests) + 1, np.int64)
    offsets[1:] = np.cumsum(lens)
    tokens = (np.concatenate([np.asarray(r, np.int32) for r in requests])
              if requests and offsets[-1] > 0 else np.zeros(1, np.int32))
    return np.ascontiguousarray(tokens, np.int32), offsets


def _args(requests, tokens, offsets):
    if requests is not None:
        tokens, offsets = pack(requests)
    tokens = np.ascontiguousarray(tokens, np.int32)
    offsets = np.ascontiguousarray(offsets, np.int64)
    if tokens.size == 0:
        tokens = np.zeros(1, np.int32)
    return tokens, offsets, int(offsets.shape[0] - 1)


def forest_group(requests=None, chunk: int = 16, single: bool = False, tokens=None, offsets=None):
    """psattn_forest_group: returns dict(group_of_req, group_parent, prefix_len,
    suffix_len, saved_tokens) ready for psattn_plan (group_parent is None in
    single-level mode)."""
    tokens, offsets, R = _args(requests, tokens, offsets)
    cap = max(R, 1)
    gor = np.zeros(max(R, 1), np.int32)
    slen = np.zeros(max(R, 1), np.int32)
    gpar = np.zeros(cap, np.int32)
    plen = np.zeros(cap, np.int32)
    ng = ctypes.c_int32(0)
    saved = ctypes.c_int64(0)
    rc = _lib.psattn_forest_group(tokens.ctypes.data, offsets.ctypes.data, R, int(chunk),
                                  FOREST_SINGLE if single else 0, gor.ctypes.data,
                                  gpar.ctypes.data, plen.ctypes.data, slen.ctypes.data, cap,
                                  ctypes.addressof(ng), ctypes.addressof(saved))
    if rc != 0:
        raise PsattnError(rc, "psattn_forest_group")
    n = ng.value
    return {"group_of_req": gor[:R].copy(), "group_parent": None if single else gpar[:n].copy(),
            "prefix_len": plen[:n].copy(), "suffix_len": slen[:R].copy(),
            "saved_tokens": int(saved.value)}


def cht_batches(requests=None, chunk: int = 16, max_batch: int = 64, max_new_chunks: int = 0,
                tokens=None, offsets=None):
    """psattn_cht_batches: returns (batch_of_req int32 [R], order int32 [R], num_batches)."""
    tokens, offsets, R = _args(requests, tokens, offsets)
    bor = np.zeros(max(R, 1), np.int32)
    order = np.zeros(max(R, 1), np.int32)
    nb = ctypes.c_int32(0)
    rc = _lib.psattn_cht_batches(tokens.ctypes.data, offsets.ctypes.data, R, int(chunk),
                                 int(max_batch), int(max_new_chunks), bor.ctypes.data,
                                 order.ctypes.data, ctypes.addressof(nb))
    if rc != 0:
        raise PsattnError(rc, "psattn_cht_batches")
    return bor[:R].copy(), order[:R].copy(), int(nb.value)


def cht_group(requests=None, chunk: int = 16, max_batch: int = 64, max_new_chunks: int = 0,
              single: bool = False, tokens=None, offsets=None):
    """psattn_cht_group: CHT batches, each with its own group forest.  Returns
    dict(batch_of_req, order, num_batches, batch_group_offset, group_of_req,
    group_parent, prefix_len, suffix_len, saved_tokens), group ids global."""
    tokens, offsets, R = _args(requests, tokens, offsets)
    n = max(R, 1)
    bor, order = np.zeros(n, np.int32), np.zeros(n, np.int32)
    bgo = np.zeros(R + 1, np.int32)
    gor, slen = np.zeros(n, np.int32), np.zeros(n, np.int32)
    gpar, plen = np.zeros(n, np.int32), np.zeros(n, np.int32)
    nb, ng, saved = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int64(0)
    rc = _lib.psattn_cht_group(tokens.ctypes.data, offsets.ctypes.data, R, int(chunk),
                               int(max_batch), int(max_new_chunks),
                               FOREST_SINGLE if single else 0, bor.ctypes.data,
                               order.ctypes.data, ctypes.addressof(nb), bgo.ctypes.data,
                               gor.ctypes.data, gpar.ctypes.data, plen.ctypes.data,
                               slen.ctypes.data, n, ctypes.addressof(ng), ctypes.addressof(saved))
    if rc != 0:
        raise PsattnError(rc, "psattn_cht_group")
    b, g = nb.value, ng.value
    return {"batch_of_req": bor[:R].copy(), "order": order[:R].copy(), "num_batches": b,
            "batch_group_offset": bgo[:b + 1].copy(), "group_of_req": gor[:R].copy(),
            "group_parent": gpar[:g].copy(), "prefix_len": plen[:g].copy(),
            "suffix_len": slen[:R].copy(), "saved_tokens": int(saved.value)}


def batch_grouping(res, b):
    """Batch b of a cht_group result as a batch of its own: (request ids,
    group_of_req, group_parent, prefix_len, suffix_len) with group ids local
    to the batch, ready for psattn_plan."""
    lo, hi = int(res["batch_group_offset"][b]), int(res["batch_group_offset"][b + 1])
    req = np.nonzero(res["batch_of_req"] == b)[0]
    gor = res["group_of_req"][req].astype(np.int32)
    gor = np.where(gor >= 0, gor - lo, -1).astype(np.int32)
    gpar = res["group_parent"][lo:hi]
    gpar = np.where(gpar >= 0, gpar - lo, -1).astype(np.int32)
    return req, gor, gpar, res["prefix_len"][lo:hi].copy(), res["suffix_len"][req].copy()
