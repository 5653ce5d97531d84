"""ctypes loader for libfd_decode.so and the fd_tensor descriptor.

The library must have been built (``python -m decode_attention_20_b300.build``
or ``__graft_entry__.build()``); loading fails loudly otherwise.  There is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfd_decode.so")

FD_F32, FD_BF16, FD_I32, FD_I8, FD_E4M3 = 0, 1, 2, 3, 4
FD_KERNEL_SPLIT, FD_KERNEL_COMBINE, FD_KERNEL_BIF_CTX = 0, 1, 2

STATUS_NAMES = {
    0: "FD_OK", 1: "FD_ERR_NULL", 2: "FD_ERR_SHAPE", 3: "FD_ERR_DTYPE", 4: "FD_ERR_LAYOUT",
    5: "FD_ERR_ARG", 6: "FD_ERR_UNSUPPORTED", 7: "FD_ERR_ARCH", 8: "FD_ERR_CUDA",
    9: "FD_ERR_DEVICE_BOUNDS", 10: "FD_ERR_DEVICE_TIMEOUT",
}


class FdTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
    ]


_T = ctypes.POINTER(FdTensor)
_lib = None


def _declare(lib):
    st = ctypes.c_int32
    sig = {
        "fd_decode_attention": (st, [_T, _T, _T, _T, ctypes.c_int32, ctypes.c_float, _T, _T, ctypes.c_void_p]),
        "fd_decode_attention_noalloc": (st, [_T, _T, _T, _T, ctypes.c_int32, ctypes.c_float, _T, _T, ctypes.c_void_p]),
        "fd_decode_attention_paged": (st, [_T, _T, _T, _T, _T, ctypes.c_int32, ctypes.c_float, _T, _T, ctypes.c_void_p]),
        "fd_decode_attention_multi": (st, [_T, _T, _T, _T, ctypes.c_int32, ctypes.c_float, _T, _T, ctypes.c_void_p]),
        "fd_decode_attention_quant": (st, [_T, _T, _T, _T, _T, _T, ctypes.c_int32, ctypes.c_float, _T, _T, ctypes.c_void_p]),
        "fd_decode_attention_partials": (st, [_T, _T, _T, _T, ctypes.c_int32, ctypes.c_float, _T, _T, ctypes.c_void_p]),
        "fd_lse_combine": (st, [_T, _T, _T, _T, ctypes.c_void_p]),
        "fd_bifurcated_attention": (st, [_T, _T, _T, _T, _T, _T, ctypes.c_float, _T, ctypes.c_void_p]),
        "fd_bifurcated_attention_lse": (st, [_T, _T, _T, _T, _T, _T, ctypes.c_float, ctypes.c_int32, _T, _T, ctypes.c_void_p]),
        "fd_choose_num_splits": (ctypes.c_int32, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]),
        "fd_split_bounds": (st, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
        "fd_workspace_bytes": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]),
        "fd_check_device_error": (st, [ctypes.c_void_p]),
        "fd_status_string": (ctypes.c_char_p, [st]),
        "fd_last_error": (ctypes.c_char_p, []),
        "fd_profile_enable": (st, [ctypes.c_int32]),
        "fd_profile_read": (st, [ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)]),
        "fd_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def lib():
    """The loaded library (loaded once).  Raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m decode_attention_20_b300.build`")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


class FdError(RuntimeError):
    """A non-FD_OK status returned by the library."""

    def __init__(self, status, message):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


def check(status):
    if status != 0:
        msg = lib().fd_last_error().decode(errors="replace")
        raise FdError(status, msg)
    return status


def raw_descriptor(data_ptr, dtype, shape, stride):
    """Descriptor from plain values (pointer as int)."""
    t = FdTensor()
    t.data = data_ptr
    t.dtype = dtype
    t.ndim = len(shape)
    for i in range(4):
        t.shape[i] = shape[i] if i < len(shape) else 0
        t.stride[i] = stride[i] if i < len(stride) else 0
    return t
