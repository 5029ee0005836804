"""ctypes view of libspecverify.so (the C ABI declared in include/spec_verify.h)."""
from __future__ import annotations

import ctypes
import os

from .build import LIB

SV_OK, SV_EINVAL, SV_ECUDA, SV_EUNSUPPORTED = 0, 1, 2, 3
SV_BF16, SV_FP32 = 0, 1
SV_BAD_U, SV_BAD_TOKEN, SV_BAD_Q, SV_BAD_ROW, SV_DEGENERATE_RESIDUAL = 1, 2, 4, 8, 16
SV_INTERNAL_TIMEOUT = 32
SV_BAD_TREE = 64
SV_MAX_TREE_NODES = 256
SV_MAX_V = 1 << 21

# every function the header declares, in declaration order
EXPORTS = ["sv_workspace_bytes", "spec_verify", "spec_verify_stats", "sv_verify_rows",
           "sv_sample_survivors", "spec_verify_noalloc", "sv_filter_logits", "sv_lm_head_workspace_bytes",
           "sv_lm_head_logits", "spec_verify_lm_head", "sv_tree_workspace_bytes", "spec_verify_tree",
           "sv_kernel_launches", "sv_status_string"]


def stats_words(K: int) -> int:
    """SV_STATS_WORDS(K): the counters spec_verify_stats adds to."""
    return 4 + K + 1

_VERIFY_ARGTYPES = [
    ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
    ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int32,
    ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
    ctypes.c_size_t, ctypes.c_void_p]

_lib = None


class NativeLibraryMissing(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise NativeLibraryMissing(
                f"{LIB} is missing; build it with "
                "`python -m speculative_decoding_sampling_gb300.build`")
        L = ctypes.CDLL(LIB)
        L.sv_workspace_bytes.restype = ctypes.c_size_t
        L.sv_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        for name in ("spec_verify", "sv_verify_rows", "sv_sample_survivors"):
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
            fn.argtypes = _VERIFY_ARGTYPES
        L.spec_verify_stats.restype = ctypes.c_int
        L.spec_verify_stats.argtypes = _VERIFY_ARGTYPES[:-1] + [ctypes.c_void_p, ctypes.c_void_p]
        L.sv_filter_logits.restype = ctypes.c_int
        L.sv_filter_logits.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int32,
                                       ctypes.c_float, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.sv_kernel_launches.restype = ctypes.c_int
        L.sv_kernel_launches.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_void_p]
        L.sv_lm_head_workspace_bytes.restype = ctypes.c_size_t
        L.sv_lm_head_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        L.sv_lm_head_logits.restype = ctypes.c_int
        L.sv_lm_head_logits.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.sv_tree_workspace_bytes.restype = ctypes.c_size_t
        L.sv_tree_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        L.spec_verify_tree.restype = ctypes.c_int
        L.spec_verify_tree.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_float, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.spec_verify_lm_head.restype = ctypes.c_int
        L.spec_verify_lm_head.argtypes = ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32] +
                                          _VERIFY_ARGTYPES[2:9] + [ctypes.c_void_p] + _VERIFY_ARGTYPES[9:])
        L.sv_status_string.restype = ctypes.c_char_p
        L.sv_status_string.argtypes = [ctypes.c_int]
        _lib = L
    return _lib
