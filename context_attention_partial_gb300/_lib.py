"""ctypes view of the C ABI in include/cpattn.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcpattn.so")

MAX_DIMS = 5
MAX_RING_DEGREE = 64

STATUS = {
    0: "CPATTN_OK", 1: "CPATTN_ERR_NULL", 2: "CPATTN_ERR_DTYPE", 3: "CPATTN_ERR_SHAPE",
    4: "CPATTN_ERR_DIVISIBILITY", 5: "CPATTN_ERR_LAYOUT", 6: "CPATTN_ERR_UNSUPPORTED",
    7: "CPATTN_ERR_WORKSPACE", 8: "CPATTN_ERR_CUDA", 9: "CPATTN_ERR_TIMEOUT",
    10: "CPATTN_ERR_BOUNDS",
}
F32, BF16 = 0, 1

# Every symbol include/cpattn.h declares.
EXPORTS = (
    "cpattn_partial", "cpattn_merge", "cpattn_ring_workspace_bytes", "cpattn_ring",
    "cpattn_ulysses_permute", "cpattn_status_string", "cpattn_last_device_status",
    "cpattn_set_wait_timeout_ns", "cpattn_ring_noalloc", "cpattn_ring_noalloc_max_workspace_bytes",
    "cpattn_set_fault_injection", "cpattn_ring_causal", "cpattn_ulysses_anything_permute",
    "cpattn_ulysses_anything_attention", "cpattn_ulysses_permute_batch",
    "cpattn_ulysses_anything_permute_batch", "cpattn_is_check_build", "cpattn_set_check_shrink",
)


class CTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * MAX_DIMS),
        ("stride", ctypes.c_int64 * MAX_DIMS),
    ]


class CpattnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{what}: {self.name}" if what else self.name)


_lock = threading.Lock()
_lib = None


def bind(path: str):
    """Opens a build of the library at `path` and declares every function's
    argument and result types."""
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(CTensor)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.cpattn_partial.argtypes = [P, P, P, ctypes.c_float, P, P, vp]
    lib.cpattn_merge.argtypes = [P, P, P, P, vp]
    lib.cpattn_ring_workspace_bytes.argtypes = [P, i32]
    lib.cpattn_ring_workspace_bytes.restype = ctypes.c_size_t
    lib.cpattn_ring.argtypes = [P, P, P, ctypes.c_float, i32, i32, P, P, vp, ctypes.c_size_t, vp]
    lib.cpattn_ulysses_permute.argtypes = [P, i32, i32, P, vp]
    lib.cpattn_ring_causal.argtypes = [P, P, P, ctypes.c_float, i32, i32, P, P, vp,
                                       ctypes.c_size_t, vp]
    lib.cpattn_ulysses_anything_permute.argtypes = [P, i32, i32, P, vp]
    lib.cpattn_ulysses_permute_batch.argtypes = [i32, P, i32, i32, P, vp]
    lib.cpattn_ulysses_anything_permute_batch.argtypes = [i32, P, i32, i32, P, vp]
    lib.cpattn_ulysses_anything_attention.argtypes = [P, P, P, ctypes.c_float, i32, i32, P, P,
                                                      vp]
    lib.cpattn_ring_noalloc.argtypes = [P, P, P, ctypes.c_float, i32, i32, P, P, vp]
    lib.cpattn_ring_noalloc_max_workspace_bytes.argtypes = []
    lib.cpattn_ring_noalloc_max_workspace_bytes.restype = ctypes.c_size_t
    lib.cpattn_status_string.argtypes = [i32]
    lib.cpattn_status_string.restype = ctypes.c_char_p
    lib.cpattn_last_device_status.argtypes = [vp]
    lib.cpattn_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.cpattn_set_wait_timeout_ns.restype = None
    lib.cpattn_set_fault_injection.argtypes = [i32]
    lib.cpattn_set_fault_injection.restype = None
    lib.cpattn_is_check_build.argtypes = []
    lib.cpattn_is_check_build.restype = ctypes.c_int
    lib.cpattn_set_check_shrink.argtypes = [ctypes.c_int64]
    lib.cpattn_set_check_shrink.restype = None
    for name in ("cpattn_partial", "cpattn_merge", "cpattn_ring", "cpattn_ulysses_permute",
                 "cpattn_last_device_status", "cpattn_ring_noalloc", "cpattn_ring_causal",
                 "cpattn_ulysses_anything_permute", "cpattn_ulysses_anything_attention",
                 "cpattn_ulysses_permute_batch", "cpattn_ulysses_anything_permute_batch"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def load():
    """Loads libcpattn.so (built by ``__graft_entry__.build()``).  Raises if it
    is missing: there is no fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (nvcc, sm_103a); there is no non-CUDA fallback")
        _lib = bind(LIB_PATH)
        return _lib


def describe(data_ptr: int, dtype_code: int, shape, stride) -> CTensor:
    t = CTensor()
    t.data = data_ptr or None
    t.dtype = dtype_code
    t.ndim = len(shape)
    for i, (s, st) in enumerate(zip(shape, stride)):
        t.shape[i] = int(s)
        t.stride[i] = int(st)
    return t


def check(status: int, what: str):
    if status != 0:
        raise CpattnError(status, what)
