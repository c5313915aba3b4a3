"""ctypes binding of libqz (include/qz.h).  Argument marshalling only.

The library is built in-tree by ``weight_only_quantized_dequant_gb300.build``.
There is no fallback: if libqz.so is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int, c_int64, c_size_t, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqz.so")

STATUS = {0: "QZ_OK", 1: "QZ_ERR_INVALID_ARG", 2: "QZ_ERR_ALIGNMENT",
          3: "QZ_ERR_UNSUPPORTED", 4: "QZ_ERR_CUDA", 5: "QZ_ERR_IO", 6: "QZ_ERR_DATA"}
QZ_MAX_BATCH = 64
QZ_MAX_GROUP = 4


class QzError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        msg = f"{fn}: {self.name}"
        if status == 4:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


class Int8Weight(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("scale", c_void_p),
                ("N", c_int64), ("K", c_int64), ("ldq", c_int64)]


class Int4oWeight(ctypes.Structure):
    _fields_ = [("N", c_int64), ("K", c_int64), ("n_out", c_int64),
                ("ld_out", c_int64), ("ld_q4", c_int64),
                ("perm", c_void_p), ("w_out", c_void_p), ("q4", c_void_p),
                ("scale", c_void_p)]


_S = c_int  # qz_status
_SIGS = {
    "qz_status_string": (c_char_p, [c_int]),
    "qz_version": (c_int, []),
    "qz_last_cuda_error": (c_int, []),
    "qz_set_overlap": (_S, [c_int]),
    "qz_get_overlap": (c_int, []),
    "qz_device_error": (_S, [POINTER(c_int), c_int]),
    "qz_quantize_int8": (_S, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_int64,
                              c_void_p, c_void_p]),
    "qz_gemv_int8": (_S, [POINTER(Int8Weight), c_void_p, c_void_p, c_void_p]),
    "qz_gemm_int8": (_S, [POINTER(Int8Weight), c_int64, c_void_p, c_int64, c_void_p,
                          c_int64, c_void_p, c_size_t, c_void_p]),
    "qz_gemm_workspace_bytes": (c_size_t, [c_int64, c_int64, c_int64]),
    "qz_gemv_int8_grouped": (_S, [POINTER(Int8Weight), c_int, c_void_p, POINTER(c_void_p),
                                  c_void_p]),
    "qz_embed_int8": (_S, [POINTER(Int8Weight), c_void_p, c_int64, c_void_p, c_int64, c_void_p]),
    "qz_gemm_int8_grouped": (_S, [POINTER(Int8Weight), c_int, c_int64, c_void_p, c_int64,
                                  POINTER(c_void_p), POINTER(c_int64), c_void_p, c_size_t,
                                  c_void_p]),
    "qz_int4o_layout": (_S, [c_int64, c_int64, c_int64, POINTER(c_int64), POINTER(c_int64)]),
    "qz_saliency_accumulate": (_S, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p]),
    "qz_select_outliers": (_S, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "qz_check_perm": (_S, [c_void_p, c_int64, c_void_p, c_void_p]),
    "qz_quantize_int4_outlier": (_S, [c_void_p, c_int64, c_void_p, c_int64, c_int64, c_int64,
                                      c_void_p, c_int64, c_void_p, c_int64, c_void_p,
                                      c_void_p]),
    "qz_gemv_int4_outlier": (_S, [POINTER(Int4oWeight), c_void_p, c_void_p, c_void_p]),
    "qz_gemm_int4_outlier": (_S, [POINTER(Int4oWeight), c_int64, c_void_p, c_int64,
                                  c_void_p, c_int64, c_void_p, c_size_t, c_void_p]),
    "qz_gemm_int4_outlier_noalloc": (_S, [POINTER(Int4oWeight), c_int64, c_void_p, c_int64,
                                          c_void_p, c_int64, c_void_p]),
    "qz_gemv_int4_outlier_grouped": (_S, [POINTER(Int4oWeight), c_int, c_void_p,
                                          POINTER(c_void_p), c_void_p]),
    "qz_gemv_int8_grouped_mapped": (_S, [POINTER(Int8Weight), c_int, c_void_p,
                                         POINTER(c_void_p), c_void_p]),
    "qz_gemv_int4_outlier_grouped_mapped": (_S, [POINTER(Int4oWeight), c_int, c_void_p,
                                                 POINTER(c_void_p), c_void_p]),
    "qz_gemm_int4_outlier_grouped": (_S, [POINTER(Int4oWeight), c_int, c_int64, c_void_p,
                                          c_int64, POINTER(c_void_p), POINTER(c_int64),
                                          c_void_p, c_size_t, c_void_p]),
    "qz_gemv_int8_sequence": (_S, [POINTER(Int8Weight), POINTER(c_int), c_int, POINTER(c_void_p),
                                   POINTER(c_void_p), c_void_p, c_void_p]),
    "qz_gemv_int4_outlier_sequence": (_S, [POINTER(Int4oWeight), POINTER(c_int), c_int,
                                           POINTER(c_void_p), POINTER(c_void_p), c_void_p,
                                           c_void_p]),
    "qz_pager_create": (_S, [POINTER(c_void_p), POINTER(c_size_t), c_int, c_void_p, c_void_p,
                             c_size_t, c_void_p, c_void_p, POINTER(c_void_p)]),
    "qz_pager_acquire": (_S, [c_void_p, c_int, POINTER(c_void_p)]),
    "qz_pager_release": (_S, [c_void_p, c_int]),
    "qz_pager_destroy": (_S, [c_void_p]),
    "qz_pager_inject_copy_failure": (_S, [c_void_p, c_int]),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libqz.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with weight_only_quantized_dequant_gb300.build"
                " (there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def call(name: str, *args) -> None:
    """Call a qz_* function that returns a status; raise QzError on failure."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise QzError(name, st, lib.qz_last_cuda_error() if st == 4 else 0)


def status(name: str, *args) -> int:
    """Call a qz_* function and return its raw status (for tests of validation)."""
    return getattr(load(), name)(*args)
