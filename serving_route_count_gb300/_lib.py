"""ctypes loader of libmoe_gb300.so with the signatures of include/moe_gb300.h.

There is no fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
c_int8_p = ctypes.POINTER(ctypes.c_int8)
c_int32_p = ctypes.POINTER(ctypes.c_int32)
c_uint8_p = ctypes.POINTER(ctypes.c_uint8)
c_size_t_p = ctypes.POINTER(ctypes.c_size_t)
c_int_p = ctypes.POINTER(ctypes.c_int)

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe_gb300.h")


class MoeCheckpoint(ctypes.Structure):
    _fields_ = [("w13", c_void_p), ("s13", c_void_p), ("g13", c_void_p),
                ("w2", c_void_p), ("s2", c_void_p), ("g2", c_void_p),
                ("nf_w13", c_void_p), ("nf_s13", c_void_p), ("nf_w2", c_void_p),
                ("nf_s2", c_void_p), ("a1_gscale", c_void_p), ("a2_gscale", c_void_p)]


# name -> (restype, argtypes)
SIGNATURES = {
    "moe_plan_weights": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int8_p, ctypes.POINTER(c_void_p)]),
    "moe_prepared_bytes": (c_int, [c_void_p, c_size_t_p]),
    "moe_prepare_weights": (c_int, [c_void_p, ctypes.POINTER(MoeCheckpoint), c_void_p, c_size_t,
                                    c_void_p, ctypes.POINTER(c_void_p)]),
    "moe_plan": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                         ctypes.POINTER(c_void_p)]),
    "moe_plan_set_swiglu_alpha_beta": (c_int, [c_void_p, c_float, c_float]),
    "moe_scratch_bytes": (c_int, [c_void_p, c_size_t_p]),
    "moe_plan_set_backend": (c_int, [c_void_p, c_int]),
    "moe_plan_set_fc1_kernel": (c_int, [c_void_p, c_int]),
    "moe_plan_set_expert_offset": (c_int, [c_void_p, c_int]),
    "moe_plan_set_router_weight_on_input": (c_int, [c_void_p, c_int]),
    "moe_plan_set_debug_copies": (c_int, [c_void_p, c_int]),
    "moe_plan_set_wait_probe": (c_int, [c_void_p, ctypes.c_ulonglong]),
    "moe_plan_set_kept_a8": (c_int, [c_void_p, ctypes.c_float, ctypes.c_float]),
    "moe_run": (c_int, [c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p, c_void_p,
                        c_void_p, c_int, c_void_p]),
    "moe_unprepare_weights": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "moe_run_chunked": (c_int, [c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_int, c_void_p]),
    "moe_run_static_scratch": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_int, c_void_p]),
    "moe_io_bytes": (c_int, [c_void_p, c_size_t_p]),
    "moe_run_host": (c_int, [c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_size_t, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "moe_get_device_error": (c_int, [c_void_p, c_void_p, c_void_p, c_int_p]),
    "moe_get_device_error_static": (c_int, [c_void_p, c_void_p, c_int_p]),
    "moe_debug_routing": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p]),
    "moe_debug_actq": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_debug_h": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_plan_set_profile_events": (c_int, [c_void_p, ctypes.POINTER(c_void_p), c_int]),
    "moe_profile_stage_names": (ctypes.c_char_p, [c_void_p]),
    "moe_call_launches": (c_int, [c_void_p, c_int, ctypes.POINTER(c_int)]),
    "moe_destroy_weight_plan": (None, [c_void_p]),
    "moe_destroy_prepared": (None, [c_void_p]),
    "moe_destroy_plan": (None, [c_void_p]),
    "moe_status_str": (ctypes.c_char_p, [c_int]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
}

_LIB = None


def header_functions(path: str = HEADER):
    """Names of the functions declared in the public header."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def load(path: str | None = None):
    """Load (once) and return the CDLL with every signature declared."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with serving_route_count_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib
