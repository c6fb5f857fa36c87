"""ctypes binding of ``liblce.so``: the C ABI of ``include/lce.h``, one Python function per entry
point, with the same names.  Argument marshalling only; every step runs in the CUDA library.
There is no fallback: if the library is missing, every call raises."""

from __future__ import annotations

import ctypes
import os
import re

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblce.so")
HEADER_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "include", "lce.h")

LCE_OK = 0
STATUS_NAMES = {
    0: "LCE_OK", 1: "LCE_ERR_INVALID_ARG", 2: "LCE_ERR_UNSUPPORTED_SHAPE",
    3: "LCE_ERR_WORKSPACE_TOO_SMALL", 4: "LCE_ERR_LABEL_OUT_OF_RANGE", 5: "LCE_ERR_CUDA",
    6: "LCE_ERR_TIMEOUT", 7: "LCE_ERR_UNSUPPORTED_DEVICE",
}
REDUCTIONS = {"mean": 0, "sum": 1}
DTYPES = {"bf16": 0, "f32": 1, "tf32x3": 2}
GRAD_PARTS = {"dh": 1, "dw": 2, "both": 3}

_c_i64 = ctypes.c_int64
_c_p = ctypes.c_void_p
_SIGNATURES = {
    "lce_workspace_size": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "lce_strip_columns": (ctypes.c_int64, [_c_i64, _c_i64, ctypes.c_int]),
    "lce_forward": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64,
                                   ctypes.c_int, ctypes.c_int, _c_p, _c_p, _c_p, _c_p,
                                   ctypes.c_size_t, _c_p]),
    "lce_backward": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                    _c_i64, _c_i64, ctypes.c_int, ctypes.c_int, _c_p, _c_p, _c_p,
                                    ctypes.c_size_t, _c_p]),
    "lce_backward_parts": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64,
                                          _c_i64, _c_i64, _c_i64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int32, _c_p, _c_p, _c_p, ctypes.c_size_t,
                                          _c_p]),
    "lce_forward_static_scratch": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_i64,
                                                  _c_i64, ctypes.c_int, ctypes.c_int, _c_p, _c_p,
                                                  _c_p, _c_p, _c_p]),
    "lce_host_buffer_size": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "lce_forward_backward_host": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                                 _c_i64, _c_i64, ctypes.c_int, ctypes.c_int, _c_p,
                                                 _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                                 ctypes.c_size_t, _c_p, _c_p, _c_p]),
    "lce_check_error": (ctypes.c_int, [_c_p, _c_p]),
    "lce_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "lce_last_cuda_error": (ctypes.c_char_p, []),
    "lce_set_tile_config": (ctypes.c_int, [ctypes.c_int32]),
    "lce_test_inject_stall": (ctypes.c_int, [ctypes.c_int32]),
    "lce_launch_count": (ctypes.c_int64, []),
    "lce_trace_begin": (ctypes.c_int, [_c_p, _c_p, _c_p, ctypes.c_int32]),
    "lce_trace_end": (ctypes.c_int32, []),
    "lce_kernel_name": (ctypes.c_char_p, [ctypes.c_int32]),
}

_lib = None


class LceError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{where}: {self.name}")


def load() -> ctypes.CDLL:
    """Load liblce.so (built in-tree by ``build()``); raises if it is not there."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"liblce.so not built at {LIB_PATH}; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def header_symbols() -> list[str]:
    """Names of the functions that include/lce.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lce_[a-z_]+)\s*\(", text)))


def check(status: int, where: str) -> None:
    if status != LCE_OK:
        if status == 5:
            where = f"{where} ({load().lce_last_cuda_error().decode()})"
        raise LceError(status, where)
