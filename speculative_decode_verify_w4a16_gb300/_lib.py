"""ctypes loader for libw4a16sv.so (the C ABI declared in include/w4a16sv.h).

Loading fails loudly when the library has not been built: there is no CPU or
Python fallback for any entry point.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16sv.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "w4a16sv.h")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_DEVICE_TIMEOUT = 4
ERR_DEVICE_INPUT = 5
ERR_WORKSPACE = 6
ERR_BOUNDS = 7

_lock = threading.Lock()
_lib = None

_vp, _i64, _i32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "w4a16_status_string": (ctypes.c_char_p, [_i32]),
    "w4a16_abi_version": (_i32, []),
    "w4a16_packed_weight_bytes": (_sz, [_i64, _i64]),
    "w4a16_packed_scale_bytes": (_sz, [_i64, _i64]),
    "w4a16_quantize": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "w4a16_prepack": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp, _vp]),
    "w4a16_linear_workspace_bytes": (_sz, [_i32, _i64, _i64]),
    "w4a16_linear": (_i32, [_vp, _i32, _i64, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "spec_accept_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "spec_accept": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "w4a16_check_device_status": (_i32, [_vp]),
    "w4a16_item_rounds": (ctypes.c_int, [_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "w4a16_item_begin": (_i64, [_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "w4a16_item_owner": (_i64, [_i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64]),
    "w4a16_linear_logits_workspace_bytes": (_sz, [_i32, _i64, _i64]),
    "w4a16_linear_logits": (_i32, [_vp, _i32, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _sz, _vp]),
    "spec_accept_prestat": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "spec_accept_node": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tree_attention_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "tree_attention": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, ctypes.c_float,
                              _vp, _vp, _sz, _vp]),
    "kv_compact": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "w4a16_linear_noalloc_scratch_bytes": (_sz, []),
    "w4a16_linear_noalloc": (_i32, [_vp, _i32, _i64, _vp, _vp, _i64, _vp, _vp]),
}


class W4A16Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


def _load(path: str):
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """The loaded library (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m speculative_decode_verify_w4a16_gb300.build`")
            _lib = _load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every call of this binding through another build of the same
    ABI (the debug builds the tests load) while the context is open."""
    global _lib
    lib()
    with _lock:
        saved, _lib = _lib, _load(path)
    try:
        yield _lib
    finally:
        with _lock:
            _lib = saved


def status_string(status: int) -> str:
    return lib().w4a16_status_string(int(status)).decode()


def check(status: int, what: str = "") -> None:
    if status != OK:
        raise W4A16Error(status, what)
