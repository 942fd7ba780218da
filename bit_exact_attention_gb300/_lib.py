"""ctypes loader for libsage2_attn.so (the C ABI declared in include/sage2_attn.h).

No fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build

_lock = threading.Lock()
_lib = None

HEADER = os.path.join(_build.INCLUDE, "sage2_attn.h")

OK, EINVAL, EUNSUPPORTED, EWORKSPACE, ECUDA, EDEVICE_TIMEOUT = 0, -1, -2, -3, -4, -5
FP16, BF16, FP32 = 0, 1, 2


class Sage2Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_str(code)} ({code})")


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "total_bytes", "qcode", "kcode", "vcodeT", "qscale", "kscale", "qmean", "kmean", "vscale",
        "vinv", "dsc", "kpart", "vpart", "status")] + [
        (n, ctypes.c_int) for n in ("Dp", "Tq", "Tkv", "nkv_pad", "nchunk", "code_bytes")]


def header_functions() -> list[str]:
    """Names of the functions include/sage2_attn.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(sage2_\w+)\s*\(", src)
    return sorted(set(names))


def _declare(lib):
    P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "sage2_status_str": ([i], ctypes.c_char_p),
        "sage2_version": ([], i),
        "sage2_workspace_size": ([i] * 8, sz),
        "sage2_workspace_layout": ([i] * 8 + [ctypes.POINTER(WsLayout)], i),
        "sage2_workspace_size_ex": ([i] * 9, sz),
        "sage2_workspace_layout_ex": ([i] * 9 + [ctypes.POINTER(WsLayout)], i),
        "sage2_attn_fwd": ([P, P, P, P, i, i, i, i, i, i, i, i, i, f, P, sz, P], i),
        "sage2_attn_fwd_varlen": ([P, P, P, P, i, i, P, P, i, i, i, i, i, i, i, i, i, f, P, sz, P], i),
        "sage2_prepass": ([P, P, P, i, i, i, i, i, i, i, i, f, P, sz, P], i),
        "sage2_attention": ([P, i, i, i, i, i, i, i, i, f, P, sz, P], i),
        "sage2_prepass_varlen": ([P, P, P, i, P, P, i, i, i, i, i, i, i, i, i, f, P, sz, P], i),
        "sage2_prepass_varlen_ex": ([P, P, P, i, P, P, i, i, i, i, i, i, i, i, i, f, i, P, sz, P], i),
        "sage2_attention_varlen": ([P, i, P, P, i, i, i, i, i, i, i, i, i, f, P, sz, P], i),
        "sage2_attention_varlen_ex": ([P, i, P, P, i, i, i, i, i, i, i, i, i, f, i, P, sz, P], i),
        "sage2_device_status": ([P, P, ctypes.POINTER(i)], i),
        "sage2_noalloc_status": ([P, ctypes.POINTER(i)], i),
        "sage2_debug_tile": ([P, P, i, i, i, i, i, i, i, i, i, f, P, sz, i, i, i, i, P, P, P, P], i),
        "sage2_debug_tile_ex": ([P, P, i, i, i, i, i, i, i, i, i, f, i, P, sz, i, i, i, i, P, P, P, P],
                                i),
        "sage2_debug_timeout": ([i, i, i, i, i, i, P, sz, P], i),
        "sage2_attn_fwd_noalloc": ([P, P, P, P, i, i, i, i, i, i, i, i, i, f, P], i),
        "sage2_host_scratch_size": ([i] * 9, sz),
        "sage2_attn_fwd_host": ([P, P, P, P, i, i, i, i, i, i, i, i, i, f, i, i, P, sz, P], i),
        "sage2_host_status": ([P, P, ctypes.POINTER(i)], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res


def lib(build_if_missing: bool = True):
    """The loaded library (built in-tree first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path}")
            l = ctypes.CDLL(path)
            _declare(l)
            _lib = l
        return _lib


def status_str(code: int) -> str:
    return lib().sage2_status_str(code).decode()


def check(code: int, what: str) -> None:
    if code != OK:
        raise Sage2Error(code, what)
