"""ctypes loader for libsparcml.so, the C ABI declared in include/sparcml.h.

The library is built in-tree (``build.py``) the first time it is needed.
There is no fallback: if the shared library cannot be built or loaded, every
call raises.
"""
from __future__ import annotations

import ctypes as C
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

u32p = C.c_void_p  # device pointers travel as plain addresses
vp = C.c_void_p

# name -> (restype, argtypes), in the order of include/sparcml.h
SIGNATURES = {
    "sparcml_status_string": (C.c_char_p, [C.c_int]),
    "sparcml_launch_count": (C.c_uint64, []),
    "sparcml_set_fault_injection": (C.c_int, [vp, C.c_int32, vp]),
    "sparcml_get_status": (C.c_int, [vp, vp]),
    "sparcml_topk_ef_workspace_size": (C.c_size_t, [C.c_int32, C.c_uint64, vp, vp, C.c_uint32]),
    "sparcml_topk_ef": (C.c_int, [vp, vp, C.c_int32, C.c_uint64, vp, vp, C.c_uint32, vp, vp, vp,
                                  C.c_uint64, vp, C.c_size_t, vp]),
    "sparcml_topk_ef_traced": (C.c_int, [vp, vp, C.c_int32, C.c_uint64, vp, vp, C.c_uint32, vp,
                                         vp, vp, C.c_uint64, vp, C.c_size_t, vp, vp]),
    "sparcml_topk_ef_fallbacks": (C.c_int64, [vp, vp]),
    "sparcml_topk_total_k": (C.c_uint64, [vp, C.c_uint32]),
    "sparcml_topk_uniform_segments": (C.c_uint32, [C.c_uint64, C.c_uint64, C.c_uint32,
                                                   C.c_uint32, vp, vp]),
    "sparcml_topk_ef_uniform_workspace_size": (C.c_size_t, [C.c_int32, C.c_uint64, C.c_uint64,
                                                            C.c_uint32, C.c_uint32]),
    "sparcml_topk_ef_uniform": (C.c_int, [vp, vp, C.c_int32, C.c_uint64, C.c_uint64, C.c_uint32,
                                          C.c_uint32, vp, vp, vp, C.c_uint64, vp, C.c_size_t,
                                          vp]),
    "sparcml_topk_ef_uniform_traced": (C.c_int, [vp, vp, C.c_int32, C.c_uint64, C.c_uint64,
                                                 C.c_uint32, C.c_uint32, vp, vp, vp, C.c_uint64,
                                                 vp, C.c_size_t, vp, vp]),
    "sparcml_pack_workspace_size": (C.c_size_t, [C.c_int32, C.c_uint64]),
    "sparcml_pack": (C.c_int, [vp, C.c_int32, C.c_uint64, C.c_float, vp, vp, vp, C.c_uint64,
                               vp, C.c_size_t, vp]),
    "sparcml_quantize4": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint32, C.c_uint64,
                                    vp, vp, vp, vp]),
    "sparcml_dequantize4": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint32, vp, vp,
                                      vp]),
    "sparcml_quantize": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint32, C.c_uint32,
                                   C.c_uint64, vp, vp, vp, vp, vp]),
    "sparcml_dequantize": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint32, C.c_uint32,
                                     vp, vp, vp]),
    "sparcml_sparse_reduce_qb": (C.c_int, [vp, vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint32,
                                           C.c_uint32, C.c_uint64, C.c_uint32, C.c_uint32, vp,
                                           vp, C.c_uint64, vp, vp, vp, vp, C.c_size_t, vp]),
    "sparcml_sparse_reduce_workspace_size": (C.c_size_t, [C.c_int32, C.c_uint64]),
    "sparcml_sparse_reduce": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64,
                                        C.c_uint32, C.c_uint32, vp, vp, C.c_uint64, vp, vp, vp,
                                        vp, C.c_size_t, vp]),
    "sparcml_sparse_reduce_traced": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64,
                                               C.c_uint32, C.c_uint32, vp, vp, C.c_uint64, vp,
                                               vp, vp, vp, C.c_size_t, vp, vp]),
    "sparcml_sparse_reduce_op": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64,
                                           C.c_int32, C.c_uint32, C.c_uint32, vp, vp, C.c_uint64,
                                           vp, vp, vp, vp, C.c_size_t, vp]),
    "sparcml_sparse_reduce_q4": (C.c_int, [vp, vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint32,
                                           C.c_uint64, C.c_uint32, C.c_uint32, vp, vp,
                                           C.c_uint64, vp, vp, vp, vp, C.c_size_t, vp]),
    "sparcml_sparse_reduce_noalloc": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64,
                                                C.c_uint32, C.c_uint32, vp, vp, C.c_uint64, vp,
                                                vp, vp, vp, vp]),
    "sparcml_ssar_workspace_size": (C.c_size_t, [C.c_int32, C.c_uint64, C.c_uint64]),
    "sparcml_ssar_allreduce": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64, vp, vp,
                                         C.c_uint64, vp, vp, vp, C.c_size_t, vp]),
    "sparcml_ssar_allreduce_traced": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64,
                                                vp, vp, C.c_uint64, vp, vp, vp, C.c_size_t, vp,
                                                vp]),
    "sparcml_densify": (C.c_int, [vp, vp, vp, C.c_int32, C.c_uint64, C.c_uint64, vp, vp, vp]),
    "sparcml_check_finite": (C.c_int, [vp, C.c_uint64, vp, vp]),
}


def load():
    """Return the loaded library, building it first if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = C.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def path() -> str:
    return _build.LIB
