"""ctypes loader for libspconv.so (argument marshalling only).

The library is built in-tree by ``sparse_weight_direct_gb300/build.py`` (the
repository's ``__graft_entry__.build()`` calls it).  If it is missing, loading
raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
# SPCONV_LIBRARY selects another build of the same library (the bounds-checked
# libspconv_debug.so, the trace build libspconv_trace.so); the default is the
# in-tree libspconv.so.
LIB_PATH = os.environ.get("SPCONV_LIBRARY") or os.path.join(HERE, "libspconv.so")

SPCONV_OK = 0
SPCONV_ERR_INVALID_ARG = -1
SPCONV_ERR_BAD_CSR = -2
SPCONV_ERR_UNSUPPORTED = -3
SPCONV_ERR_ALLOC = -4
SPCONV_ERR_CUDA = -5
SPCONV_ERR_MISMATCH = -6
SPCONV_ERR_DEVICE = -7

# Every symbol include/spconv.h declares.
EXPORTS = ("spconv_pack", "spconv_pack_ex", "spconv_forward", "spconv_forward_ex",
           "spconv_forward_host", "spconv_forward_host_noalloc", "spconv_packed_free",
           "spconv_status_string",
           "spconv_pack_host", "spconv_device_status", "spconv_selftest_wait",
           "spconv_packed_info_get", "spconv_launch_info_get", "spconv_packed_copy_array",
           "spconv_trace_read")

_lock = threading.Lock()
_lib = None


class SpconvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})" if what
                         else f"{status_string(status)} (status {status})")


class PackedInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("C", "H", "W", "M", "R", "S", "stride", "pad", "E", "F")] + [
        ("nnz", ctypes.c_int64), ("entries", ctypes.c_int64)] + [
        (n, ctypes.c_int32) for n in
        ("tile_rows", "shift", "tile_cols", "tiles_y", "tiles_x", "in_rows", "in_cols",
         "phase_pitch", "row_pitch", "plane", "chunk", "num_chunks", "slots_per_warp", "warps",
         "groups", "num_slots", "on_device")] + [
        (n, ctypes.c_int64) for n in
        ("device_bytes", "smem_bytes", "max_warp_nnz", "mean_warp_nnz")] + [
        (n, ctypes.c_int32) for n in
        ("hdr_words", "blob_stage_bytes", "in_stage_bytes", "lane_rows", "dense_groups",
         "dense_mask_words", "format", "batch_hint", "blob_stride", "tap_pairs",
         "plane_stage", "col_blocks", "tile_images", "pair_off")]


class LaunchInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kernel", "grid_x", "grid_y", "grid_z", "block_threads", "cluster", "push",
                 "group_fast", "tma", "pdl")] + [("smem_bytes", ctypes.c_int64)]


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                f"g.build()'` (or python sparse_weight_direct_gb300/build.py); "
                "there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        i, p = ctypes.c_int, ctypes.c_void_p
        L.spconv_pack.argtypes = [i] * 8 + [p, p, p, p, ctypes.POINTER(ctypes.c_void_p)]
        L.spconv_pack.restype = i
        L.spconv_pack_host.argtypes = [i] * 8 + [p, p, p, ctypes.POINTER(ctypes.c_void_p)]
        L.spconv_pack_host.restype = i
        L.spconv_pack_ex.argtypes = [i] * 8 + [p, p, p, i, i, i, p,
                                               ctypes.POINTER(ctypes.c_void_p)]
        L.spconv_pack_ex.restype = i
        L.spconv_forward.argtypes = [i] * 9 + [p, p, p, p]
        L.spconv_forward.restype = i
        L.spconv_forward_ex.argtypes = [i] * 9 + [p, p, p, i, p, p]
        L.spconv_forward_ex.restype = i
        L.spconv_forward_host.argtypes = [i] * 9 + [p, p, p, i, p, p, p, p]
        L.spconv_forward_host.restype = i
        L.spconv_forward_host_noalloc.argtypes = [i] * 9 + [p, p, p, i, p, p]
        L.spconv_forward_host_noalloc.restype = i
        L.spconv_packed_free.argtypes = [p]
        L.spconv_packed_free.restype = None
        L.spconv_status_string.argtypes = [i]
        L.spconv_status_string.restype = ctypes.c_char_p
        L.spconv_packed_info_get.argtypes = [p, ctypes.POINTER(PackedInfo)]
        L.spconv_packed_info_get.restype = i
        L.spconv_launch_info_get.argtypes = [p, i, ctypes.POINTER(LaunchInfo)]
        L.spconv_launch_info_get.restype = i
        L.spconv_packed_copy_array.argtypes = [p, i, p, ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_int64)]
        L.spconv_packed_copy_array.restype = i
        L.spconv_device_status.argtypes = [p, p, ctypes.POINTER(ctypes.c_int32)]
        L.spconv_device_status.restype = i
        L.spconv_selftest_wait.argtypes = [i, p, ctypes.POINTER(ctypes.c_int32)]
        L.spconv_selftest_wait.restype = i
        L.spconv_trace_read.argtypes = [p, ctypes.c_int64]
        L.spconv_trace_read.restype = i
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return lib().spconv_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def check(rc: int, what: str) -> None:
    if rc != SPCONV_OK:
        raise SpconvError(rc, what)
