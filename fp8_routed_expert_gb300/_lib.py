"""ctypes declarations of the C ABI in include/fp8moe.h.

Loads the in-tree ``libfp8moe.so``.  There is no fallback: if the library is
missing, ``lib()`` raises with the command that builds it.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfp8moe.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "fp8moe.h")

_lib = None


class MoEConfig(ctypes.Structure):
    _fields_ = [("max_tokens", ctypes.c_int64), ("hidden", ctypes.c_int64),
                ("n_experts", ctypes.c_int64), ("inter", ctypes.c_int64),
                ("max_top_k", ctypes.c_int32), ("device", ctypes.c_int32)]


def _constants() -> dict:
    """#define MOE_* integer constants of the header."""
    out = {}
    for m in re.finditer(r"#define\s+(MOE_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read()):
        out[m.group(1)] = int(m.group(2))
    return out


C = _constants()


def exported_functions() -> list[str]:
    """Names of the functions the header declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|int64_t|void|const char \*)\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)))


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
                           "or `python -m fp8_routed_expert_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    sig = {
        "moe_init": ([ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(MoEConfig)], ctypes.c_int),
        "moe_layer_forward": ([vp, vp, i64, vp, vp, vp, vp, vp, vp, i32, vp, vp], ctypes.c_int),
        "moe_layer_forward_nvfp4": ([vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp],
                                    ctypes.c_int),
        "moe_layer_forward_host": ([vp, vp, i64, vp, vp, vp, vp, vp, vp, i32, vp, vp], ctypes.c_int),
        "moe_get_routing": ([vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "moe_status": ([vp], ctypes.c_int),
        "moe_free": ([vp], None),
        "moe_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "moe_set_path": ([vp, ctypes.c_int], ctypes.c_int),
        "moe_resolve_path": ([vp, i64], ctypes.c_int),
        "moe_set_timing": ([vp, ctypes.c_int], ctypes.c_int),
        "moe_kernel_time": ([vp, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                             ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
        "moe_kernel_name": ([ctypes.c_int], ctypes.c_char_p),
        "moe_launch_count": ([vp], ctypes.c_int64),
        "moe_selftest_wait_timeout": ([vp, i64, vp, vp], ctypes.c_int),
        "moe_cache_init": ([ctypes.POINTER(ctypes.c_void_p), vp, vp, vp, i64], ctypes.c_int),
        "moe_cache_forward": ([vp, vp, i64, vp, vp, vp, vp, i32, vp, vp], ctypes.c_int),
        "moe_cache_prefetch": ([vp, vp, i64], ctypes.c_int),
        "moe_cache_guess": ([vp, vp, i64, vp, vp, i32, i32, vp], ctypes.c_int),
        "moe_cache_stats": ([vp, vp, i32], ctypes.c_int),
        "moe_cache_resident": ([vp, vp], ctypes.c_int),
        "moe_cache_free": ([vp], None),
        "moe_set_sm_budget": ([vp, i32], ctypes.c_int),
        "moe_attention_workspace_bytes": ([i64, i64, i32, i32], i64),
        "moe_decode_attention": ([vp, vp, vp, i64, i64, i32, i32, i32, vp, vp, i64, vp],
                                 ctypes.c_int),
        "moe_route_noalloc": ([vp, i64, i64, vp, vp, i64, i32, vp, vp, vp, vp, vp, vp, vp],
                              ctypes.c_int),
        "moe_debug_copy": ([vp, ctypes.c_char_p, vp, i64, ctypes.POINTER(ctypes.c_int64), vp],
                           ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib().moe_strerror(code).decode()} (code {code})")


def check(code: int, where: str) -> None:
    if code != 0:
        raise MoEError(code, where)
