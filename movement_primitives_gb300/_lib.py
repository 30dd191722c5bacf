"""ctypes view of liblayoutcopy.so: struct mirrors and function prototypes.

Argument marshalling only.  The library must have been built (``build.py``,
or ``__graft_entry__.build()``); importing this module without it raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# LC_LIBRARY_PATH points at another build of the same library (e.g. one
# compiled with different tuning knobs); by default the in-tree build is used.
LIB_PATH = os.environ.get("LC_LIBRARY_PATH") or os.path.join(HERE, "liblayoutcopy.so")
MAX_RANK = 8
STATIC_STAGING_BYTES = 32 * 1024 * 1024  # LC_STATIC_STAGING_BYTES
WARP_UNIT_MAX_P = 32  # LC_WARP_UNIT_MAX_P
WARP_UNIT_MAX_BYTES = 8192  # LC_WARP_UNIT_MAX_BYTES
LOOP_MAX_THREADS = 1024  # LC_LOOP_MAX_THREADS

OK = 0
STATUS_NAMES = {
    0: "LC_OK", 1: "LC_ERR_NULL", 2: "LC_ERR_RANK", 3: "LC_ERR_SHAPE",
    4: "LC_ERR_EXTENT_MISMATCH", 5: "LC_ERR_ELEM_BYTES", 6: "LC_ERR_BAD_STRIDE",
    7: "LC_ERR_NOT_INJECTIVE", 8: "LC_ERR_OVERLAP", 9: "LC_ERR_ALIGN",
    10: "LC_ERR_NO_SWIZZLE", 11: "LC_ERR_CUDA", 12: "LC_ERR_TIMEOUT",
    13: "LC_ERR_UNSUPPORTED", 14: "LC_ERR_OVERFLOW", 15: "LC_ERR_STAGING",
    16: "LC_ERR_LOOP_LAYOUT", 17: "LC_ERR_UNDECIDED", 18: "LC_ERR_NOT_MAPPED",
}
STATUS = {v: k for k, v in STATUS_NAMES.items()}
KERNELS = {"auto": 0, "vec_copy": 1, "warp_permute": 2, "tile_transpose": 3, "smem_transpose": 4,
           "tma_copy": 5, "warp_shuffle": 6, "smem_staged": 7}


class CTileLayout(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MAX_RANK),
                ("stride", ctypes.c_int64 * MAX_RANK),
                ("offset", ctypes.c_int64),
                ("tile_stride", ctypes.c_int64)]


_M = MAX_RANK + 1


class CPlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("elem_bytes", ctypes.c_int32),
                ("n_modes", ctypes.c_int32),
                ("extent", ctypes.c_int64 * _M), ("src_stride", ctypes.c_int64 * _M),
                ("dst_stride", ctypes.c_int64 * _M), ("total", ctypes.c_int64),
                ("vec", ctypes.c_int32), ("run", ctypes.c_int64),
                ("unit_modes", ctypes.c_int32), ("P", ctypes.c_int32),
                ("k", ctypes.c_int32), ("shift", ctypes.c_int32), ("mask", ctypes.c_int32),
                ("conflicts_read", ctypes.c_int32), ("conflicts_write", ctypes.c_int32),
                ("units_per_chunk", ctypes.c_int64),
                ("tile_rows", ctypes.c_int32), ("tile_cols", ctypes.c_int32),
                ("stages", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("block", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("tile_form", ctypes.c_int32)]


class CWarpUnit(ctypes.Structure):
    _R = MAX_RANK
    _fields_ = [("n_modes", ctypes.c_int32),
                ("extent", ctypes.c_int32 * _R), ("src_stride", ctypes.c_int32 * _R),
                ("dst_stride", ctypes.c_int32 * _R),
                ("P", ctypes.c_int32), ("k", ctypes.c_int32), ("shift", ctypes.c_int32),
                ("mask", ctypes.c_int32), ("conflicts_read", ctypes.c_int32),
                ("conflicts_write", ctypes.c_int32), ("src_cosize", ctypes.c_int32),
                ("dst_cosize", ctypes.c_int32)]


class CLoopLayout(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MAX_RANK),
                ("thread_stride", ctypes.c_int64 * MAX_RANK),
                ("slot_stride", ctypes.c_int64 * MAX_RANK)]


class CLoopPlanInfo(ctypes.Structure):
    _fields_ = [("num_threads", ctypes.c_int32), ("slots_per_thread", ctypes.c_int64),
                ("points_per_tile", ctypes.c_int64), ("vec", ctypes.c_int32), ("split", ctypes.c_int32)]


class CSmemSwizzle(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("chunk_log2", ctypes.c_int32), ("row_log2", ctypes.c_int32)]


class CGmemSmem(ctypes.Structure):
    _fields_ = [("n_modes", ctypes.c_int32),
                ("extent", ctypes.c_int64 * MAX_RANK), ("g_stride", ctypes.c_int64 * MAX_RANK),
                ("s_stride", ctypes.c_int64 * MAX_RANK),
                ("g_offset", ctypes.c_int64), ("s_offset", ctypes.c_int64),
                ("elem_bytes", ctypes.c_int32), ("vec", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("outer", ctypes.c_int64), ("total", ctypes.c_int64), ("guarded", ctypes.c_int32),
                ("swizzle", CSmemSwizzle),
                ("div_m", ctypes.c_uint32 * MAX_RANK), ("div_s", ctypes.c_int32 * MAX_RANK)]


_P_LAYOUT = ctypes.POINTER(CTileLayout)
_P_LOOP = ctypes.POINTER(CLoopLayout)
_P_I32 = ctypes.POINTER(ctypes.c_int32)
_P_I64 = ctypes.POINTER(ctypes.c_int64)

# name -> (restype, argtypes); every symbol declared in include/layout_copy.h
PROTOTYPES = {
    "lc_layout_copy": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                      ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]),
    "lc_layout_copy_ex": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                         ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_void_p]),
    "lc_layout_copy_host": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                           ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p,
                                           ctypes.c_int64, ctypes.c_void_p]),
    "lc_layout_copy_mapped": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                             ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]),
    "lc_host_staging_bytes": (ctypes.c_int64, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, ctypes.c_int64]),
    "lc_layout_copy_host_static": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                                  ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]),
    "lc_window_sum_f32": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_void_p]),
    "lc_plan": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, ctypes.c_int64,
                               ctypes.c_int32, ctypes.POINTER(CPlanInfo)]),
    "lc_choose_swizzle": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, _P_I32, _P_I32,
                                         _P_I32, _P_I32, _P_I32]),
    "lc_swizzle_conflicts": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, _P_I32, _P_I32]),
    "lc_gmem_smem_partition": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32,
                                              ctypes.c_int32, _P_I32, _P_I64]),
    "lc_last_device_error": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64)]),
    "lc_debug_wait_timeout": (ctypes.c_int, [ctypes.c_int64, ctypes.c_void_p]),
    "lc_warp_unit_plan": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, ctypes.POINTER(CWarpUnit)]),
    "lc_warp_unit_run": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(CWarpUnit),
                                        ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]),
    "lc_loop_layout_default": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P_LOOP]),
    "lc_loop_layout_info": (ctypes.c_int, [_P_LOOP, ctypes.c_int64, _P_I32, _P_I64]),
    "lc_loop_plan": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, ctypes.c_int64, _P_LOOP,
                                    ctypes.POINTER(CLoopPlanInfo)]),
    "lc_layout_copy_loop": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                           ctypes.c_int32, ctypes.c_int64, _P_LOOP, ctypes.c_void_p,
                                           ctypes.c_void_p]),
    "lc_gmem_smem_plan": (ctypes.c_int, [_P_LAYOUT, _P_LAYOUT, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.POINTER(CSmemSwizzle), ctypes.POINTER(CGmemSmem)]),
    "lc_layout_copy_staged": (ctypes.c_int, [ctypes.c_void_p, _P_LAYOUT, ctypes.c_void_p, _P_LAYOUT,
                                             ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                             ctypes.POINTER(CSmemSwizzle), ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p]),
    "lc_row_major_strides": (ctypes.c_int, [ctypes.c_int32, _P_I64, _P_I64]),
    "lc_layout_footprint": (ctypes.c_int64, [_P_LAYOUT, ctypes.c_int64]),
    "lc_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "lc_kernel_name": (ctypes.c_char_p, [ctypes.c_int32]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library with prototypes set; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "movement_primitives_gb300: %s is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no fallback implementation)" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib
