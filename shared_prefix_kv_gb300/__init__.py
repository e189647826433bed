"""Python binding of the psattn C ABI (include/psattn.h).

Argument marshalling only: host arrays go in as numpy int32 arrays, device
buffers as raw pointers (an int, or any object with ``data_ptr()`` such as a
torch tensor), streams as raw ``cudaStream_t`` values.  Every step of the
attention runs inside the library's kernels.

The library is loaded from ``shared_prefix_kv_gb300/_build/libpsattn.so``.
If it has not been built, importing raises ImportError: there is no fallback.
Build it with ``python -c "import __graft_entry__ as g; g.build()"`` (or
``python shared_prefix_kv_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpsattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"psattn library not built: {LIB_PATH} is missing "
                      "(run shared_prefix_kv_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

OK = 0
ERR_INVALID_ARG = -1
ERR_BLOCK_OOB = -2
ERR_GROUP_MISMATCH = -3
ERR_EMPTY_REQUEST = -4
ERR_UNSUPPORTED = -5
ERR_CUDA = -6
ERR_DEVICE = -7
ERR_NOMEM = -8
ERR_GROUP_CYCLE = -9

F32, BF16 = 0, 1
NO_DEDUP, FLATTEN, NO_TENSOR_PREFIX, SIMT, NO_FOLD = 1, 2, 4, 8, 16

EXPORT_WARP_ITEMS, EXPORT_DENSE_ITEMS, EXPORT_REQ, EXPORT_GROUP, EXPORT_MEMBERS, EXPORT_LEN_ADD = range(6)

EXPORTED_SYMBOLS = ("psattn_plan", "psattn_plan_host", "psattn_decode", "psattn_plan_info_get",
                    "psattn_plan_export", "psattn_plan_status", "psattn_plan_destroy",
                    "psattn_status_string", "psattn_selftest_wait_timeout",
                    "psattn_plan_ragged", "psattn_plan_host_ragged", "psattn_decode_noalloc")


class Shape(ctypes.Structure):
    _fields_ = [("num_req", ctypes.c_int32), ("num_groups", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_blocks_per_req", ctypes.c_int32), ("num_pool_blocks", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("warp_items", ctypes.c_int64), ("dense_items", ctypes.c_int64),
                ("partial_slots", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("unique_kv_bytes", ctypes.c_int64), ("planned_kv_bytes", ctypes.c_int64),
                ("qo_bytes", ctypes.c_int64), ("suffix_chunk_max", ctypes.c_int32),
                ("prefix_chunk_max", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("dense_item_warps", ctypes.c_int32)]


_vp = ctypes.c_void_p
_lib.psattn_plan.argtypes = [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, ctypes.c_uint32,
                             _vp, ctypes.POINTER(_vp)]
_lib.psattn_plan.restype = ctypes.c_int
_lib.psattn_plan_host.argtypes = [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp,
                                  ctypes.c_uint32, ctypes.c_int32, ctypes.POINTER(_vp)]
_lib.psattn_plan_host.restype = ctypes.c_int
_lib.psattn_plan_ragged.argtypes = [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp,
                                    ctypes.c_uint32, _vp, ctypes.POINTER(_vp)]
_lib.psattn_plan_ragged.restype = ctypes.c_int
_lib.psattn_plan_host_ragged.argtypes = [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp,
                                         ctypes.c_uint32, ctypes.c_int32, ctypes.POINTER(_vp)]
_lib.psattn_plan_host_ragged.restype = ctypes.c_int
_lib.psattn_decode.argtypes = [_vp] * 9 + [_vp]
_lib.psattn_decode.restype = ctypes.c_int
_lib.psattn_plan_info_get.argtypes = [_vp, ctypes.POINTER(PlanInfo)]
_lib.psattn_plan_info_get.restype = ctypes.c_int
_lib.psattn_plan_export.argtypes = [_vp, ctypes.c_int32, _vp, ctypes.c_int64]
_lib.psattn_plan_export.restype = ctypes.c_int64
_lib.psattn_plan_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32)]
_lib.psattn_plan_status.restype = ctypes.c_int
_lib.psattn_selftest_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]
_lib.psattn_selftest_wait_timeout.restype = ctypes.c_int
_lib.psattn_plan_destroy.argtypes = [_vp]
_lib.psattn_plan_destroy.restype = None
_lib.psattn_status_string.argtypes = [ctypes.c_int]
_lib.psattn_status_string.restype = ctypes.c_char_p


class PsattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {psattn_status_string(status)} ({status})")
        self.status = status


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if isinstance(x, np.ndarray):
        return int(x.ctypes.data)
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _i32(a) -> Optional[np.ndarray]:
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def make_shape(num_req, num_groups, num_q_heads, num_kv_heads, head_dim, block_size,
               max_blocks_per_req, num_pool_blocks, dtype, scale) -> Shape:
    return Shape(num_req, num_groups, num_q_heads, num_kv_heads, head_dim, block_size,
                 max_blocks_per_req, num_pool_blocks, dtype, float(scale))


def psattn_status_string(status: int) -> str:
    return _lib.psattn_status_string(int(status)).decode()


def psattn_plan(shape: Shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
                flags: int = 0, stream: int = 0) -> int:
    """Returns an opaque plan handle (int); raises PsattnError on a bad status."""
    arrs = [_i32(block_table), _i32(group_of_req), _i32(group_parent), _i32(prefix_len),
            _i32(suffix_len)]
    out = _vp()
    rc = _lib.psattn_plan(ctypes.byref(shape), *[_ptr(a) for a in arrs], flags,
                          stream or None, ctypes.byref(out))
    if rc != OK:
        raise PsattnError(rc, "psattn_plan")
    return out.value


def psattn_plan_host(shape: Shape, block_table, group_of_req, group_parent, prefix_len,
                     suffix_len, flags: int = 0, num_sms: int = 148) -> int:
    arrs = [_i32(block_table), _i32(group_of_req), _i32(group_parent), _i32(prefix_len),
            _i32(suffix_len)]
    out = _vp()
    rc = _lib.psattn_plan_host(ctypes.byref(shape), *[_ptr(a) for a in arrs], flags,
                               int(num_sms), ctypes.byref(out))
    if rc != OK:
        raise PsattnError(rc, "psattn_plan_host")
    return out.value


def psattn_plan_ragged(shape: Shape, block_table, group_of_req, group_parent, prefix_len,
                       suffix_len, leaf_len, flags: int = 0, stream: int = 0) -> int:
    arrs = [_i32(block_table), _i32(group_of_req), _i32(group_parent), _i32(prefix_len),
            _i32(suffix_len), _i32(leaf_len)]
    out = _vp()
    rc = _lib.psattn_plan_ragged(ctypes.byref(shape), *[_ptr(a) for a in arrs], flags,
                                 stream or None, ctypes.byref(out))
    if rc != OK:
        raise PsattnError(rc, "psattn_plan_ragged")
    return out.value


def psattn_plan_host_ragged(shape: Shape, block_table, group_of_req, group_parent, prefix_len,
                            suffix_len, leaf_len, flags: int = 0, num_sms: int = 148) -> int:
    arrs = [_i32(block_table), _i32(group_of_req), _i32(group_parent), _i32(prefix_len),
            _i32(suffix_len), _i32(leaf_len)]
    out = _vp()
    rc = _lib.psattn_plan_host_ragged(ctypes.byref(shape), *[_ptr(a) for a in arrs], flags,
                                      int(num_sms), ctypes.byref(out))
    if rc != OK:
        raise PsattnError(rc, "psattn_plan_host_ragged")
    return out.value


def psattn_decode(plan: int, q, kv_pool, block_table, group_of_req, prefix_len, suffix_len,
                  out, lse, stream: int = 0) -> None:
    rc = _lib.psattn_decode(plan, _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(group_of_req),
                            _ptr(prefix_len), _ptr(suffix_len), _ptr(out), _ptr(lse),
                            stream or None)
    if rc != OK:
        raise PsattnError(rc, "psattn_decode")


def psattn_plan_info_get(plan: int) -> dict:
    info = PlanInfo()
    rc = _lib.psattn_plan_info_get(plan, ctypes.byref(info))
    if rc != OK:
        raise PsattnError(rc, "psattn_plan_info_get")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


def psattn_plan_export(plan: int, which: int) -> np.ndarray:
    n = _lib.psattn_plan_export(plan, which, None, 0)
    if n < 0:
        raise PsattnError(int(n), "psattn_plan_export")
    buf = np.zeros(max(n, 1), np.int32)
    _lib.psattn_plan_export(plan, which, buf.ctypes.data, n)
    return buf[:n]


def psattn_selftest_wait_timeout(limit_us: int):
    """Returns (status, device_flags) of one kernel wait that nothing completes."""
    flags = ctypes.c_uint32(0)
    rc = _lib.psattn_selftest_wait_timeout(int(limit_us), ctypes.byref(flags))
    return rc, flags.value


def psattn_plan_status(plan: int):
    flags = ctypes.c_uint32(0)
    rc = _lib.psattn_plan_status(plan, ctypes.byref(flags))
    return rc, flags.value


def psattn_plan_destroy(plan: int) -> None:
    _lib.psattn_plan_destroy(plan)


_lib.psattn_decode_noalloc.argtypes = [_vp] * 9 + [_vp]
_lib.psattn_decode_noalloc.restype = ctypes.c_int
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def psattn_decode_noalloc(plan: int, q, kv_pool, block_table, group_of_req, prefix_len,
                          suffix_len, out, lse, stream: int = 0) -> None:
    """psattn_decode for callers that cannot allocate device memory: the
    workspace lives in the library's fixed device array (see psattn.h)."""
    rc = _lib.psattn_decode_noalloc(plan, _ptr(q), _ptr(kv_pool), _ptr(block_table),
                                    _ptr(group_of_req), _ptr(prefix_len), _ptr(suffix_len),
                                    _ptr(out), _ptr(lse), stream or None)
    if rc != OK:
        raise PsattnError(rc, "psattn_decode_noalloc")


class Plan:
    """Owns a plan handle; ``close()`` (or the context manager) frees it."""

    def __init__(self, shape: Shape, block_table, group_of_req, group_parent, prefix_len,
                 suffix_len, flags: int = 0, stream: int = 0, host_only_sms: Optional[int] = None,
                 leaf_len=None):
        if leaf_len is not None and host_only_sms is None:
            self.handle = psattn_plan_ragged(shape, block_table, group_of_req, group_parent,
                                             prefix_len, suffix_len, leaf_len, flags, stream)
        elif leaf_len is not None:
            self.handle = psattn_plan_host_ragged(shape, block_table, group_of_req, group_parent,
                                                  prefix_len, suffix_len, leaf_len, flags,
                                                  host_only_sms)
        elif host_only_sms is None:
            self.handle = psattn_plan(shape, block_table, group_of_req, group_parent, prefix_len,
                                      suffix_len, flags, stream)
        else:
            self.handle = psattn_plan_host(shape, block_table, group_of_req, group_parent,
                                           prefix_len, suffix_len, flags, host_only_sms)
        self.shape = shape

    def decode(self, q, kv_pool, block_table, group_of_req, prefix_len, suffix_len, out, lse,
               stream: int = 0) -> None:
        psattn_decode(self.handle, q, kv_pool, block_table, group_of_req, prefix_len,
                      suffix_len, out, lse, stream)

    def info(self) -> dict:
        return psattn_plan_info_get(self.handle)

    def export(self, which: int) -> np.ndarray:
        return psattn_plan_export(self.handle, which)

    def status(self):
        return psattn_plan_status(self.handle)

    def close(self) -> None:
        if self.handle:
            psattn_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
