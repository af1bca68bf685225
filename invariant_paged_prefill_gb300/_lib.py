"""ctypes view of libbip.so: argument and result types for every C entry point.

Loading fails loudly when the library is missing; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_u64 = ctypes.c_uint64
c_size = ctypes.c_size_t
c_vp = ctypes.c_void_p
c_f32 = ctypes.c_float
P_i32 = ctypes.POINTER(ctypes.c_int32)


class PlanOptions(ctypes.Structure):
    _fields_ = [("split_policy", ctypes.c_int), ("split_budget_bytes", c_size), ("num_sms", c_i32),
                ("wait_limit_ns", c_u64), ("tiles_per_unit", c_i32), ("window_left", c_i32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("batch", "total_q", "num_qo_heads", "num_kv_heads", "head_dim", "page_size",
                                     "kv_dtype", "gqa_group", "tile_positions", "kv_block", "split_len",
                                     "num_units", "num_items", "num_split_units", "grid", "tiles_per_unit")] + \
               [("partial_rows", c_i64), ("kv_blocks", c_i64)] + \
               [(n, c_u64) for n in ("workspace_bytes", "partial_bytes", "scratch_bytes", "upload_bytes")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


# name -> (restype, argtypes); every symbol include/bip.h declares.
SIGNATURES = {
    "bip_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bip_workspace_bound": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_size]),
    "bip_plan": (ctypes.c_int, [ctypes.POINTER(c_vp), P_i32, P_i32, P_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                ctypes.c_int, ctypes.POINTER(PlanOptions), ctypes.POINTER(c_size)]),
    "bip_plan_get_info": (ctypes.c_int, [c_vp, ctypes.POINTER(PlanInfo)]),
    "bip_plan_get_items": (ctypes.c_int, [c_vp, P_i32, c_i32, P_i32]),
    "bip_plan_destroy": (ctypes.c_int, [c_vp]),
    "bip_prefill": (ctypes.c_int, [c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i64, c_vp, c_f32, c_f32, c_vp, c_vp,
                                   c_vp, c_size, c_vp]),
    "bip_prefill_masked": (ctypes.c_int, [c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i64, c_vp, c_vp, c_i64, c_f32,
                                          c_f32, c_vp, c_vp, c_vp, c_size, c_vp]),
    "bip_append_kv": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i64, c_vp, c_f32, c_f32, c_vp,
                                     c_size, c_vp]),
    "bip_graph_plan": (ctypes.c_int, [ctypes.POINTER(c_vp), c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.c_int,
                                      ctypes.POINTER(PlanOptions), ctypes.POINTER(c_size)]),
    "bip_prefill_graph": (ctypes.c_int, [c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_vp, c_f32,
                                         c_f32, c_vp, c_vp, c_vp, c_size, c_vp]),
    "bip_prefill_graph_masked": (ctypes.c_int, [c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_vp,
                                                c_vp, c_i64, c_f32, c_f32, c_vp, c_vp, c_vp, c_size, c_vp]),
    "bip_graph_plan_destroy": (ctypes.c_int, [c_vp]),
    "bip_read_device_status": (ctypes.c_int, [c_vp, c_vp]),
    "bip_prefill_no_alloc": (ctypes.c_int, [c_vp, c_vp, c_i64, c_vp, c_vp, c_i64, c_i64, c_vp, c_f32, c_f32, c_vp,
                                            c_vp, c_vp]),
}

_LIB = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libbip.so (built in-tree) and attach signatures."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"libbip.so not found at {path}; build it with "
            "`python -m invariant_paged_prefill_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.library_path():
        _LIB = lib
    return lib
