"""ctypes view of the C ABI in include/attn_gb300.h (no torch types)."""
from __future__ import annotations

import contextlib
import ctypes
import os

from . import build as _build

ATTN_BF16, ATTN_F16, ATTN_F32, ATTN_I32, ATTN_U8, ATTN_E4M3 = 1, 2, 3, 4, 5, 6
ATTN_DETERMINISTIC = 1
ATTN_EAGER_RESCALE = 2

ERRORS = {
    0: "ATTN_OK", -1: "ATTN_E_DTYPE", -2: "ATTN_E_SHAPE", -3: "ATTN_E_LAYOUT",
    -4: "ATTN_E_DEVICE", -5: "ATTN_E_UNSUPPORTED", -6: "ATTN_E_WORKSPACE",
    -7: "ATTN_E_CUDA", -8: "ATTN_E_TIMEOUT", -9: "ATTN_E_SEQLENS", -10: "ATTN_E_ARG", -11: "ATTN_E_INTERNAL", -12: "ATTN_E_TOO_LARGE",
}

# Every symbol the header declares.
EXPORTS = ("attn_fwd", "attn_fwd_fp8", "attn_fwd_fp8_workspace_bytes", "attn_score_recompute",
           "attn_score_workspace_bytes", "attn_sparse_bwd", "attn_sparse_bwd_workspace_bytes",
           "attn_bwd", "attn_bwd_noalloc", "attn_bwd_workspace_bytes", "attn_get_error",
           "attn_strerror", "attn_last_cuda_error", "attn_version", "attn_profile_events",
           "attn_launch_count", "attn_selftest_wait_timeout")

ATTN_STAGE_FWD, ATTN_STAGE_BWD_PREPROCESS, ATTN_STAGE_BWD_MAIN, ATTN_STAGE_BWD_DQ = 0, 1, 2, 3
ATTN_STAGE_SCORE = 4
ATTN_STAGE_SPARSE = 5


class AttnTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
        ("device", ctypes.c_int32),
    ]


PT = ctypes.POINTER(AttnTensor)

_lib = None


def lib_path() -> str:
    return _build.LIB


def load():
    """Load the shared library; raise if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = load_path(lib_path())
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Route every call made inside the block through the library at `path`
    (e.g. the poisoned-staging debug build), then restore the previous one."""
    global _lib
    prev = _lib
    _lib = load_path(path)
    try:
        yield _lib
    finally:
        _lib = prev


def load_path(path):
    """Load and bind one build of the library."""
    if not os.path.exists(path):
        raise RuntimeError(
            "CUDA attention library not built (%s missing); run "
            "softmax_attention_numerics_gb300.build.build() first" % path)
    lib = ctypes.CDLL(path)
    lib.attn_fwd.restype = ctypes.c_int
    lib.attn_fwd.argtypes = [PT, PT, PT, PT, PT, ctypes.c_int32, ctypes.c_int, ctypes.c_float,
                             PT, PT, ctypes.c_uint32, ctypes.c_void_p]
    lib.attn_fwd_fp8.restype = ctypes.c_int
    lib.attn_fwd_fp8.argtypes = [PT, PT, PT, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                 ctypes.c_int, ctypes.c_float, PT, PT, ctypes.c_void_p,
                                 ctypes.c_size_t, ctypes.c_uint32, ctypes.c_void_p]
    lib.attn_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_fwd_fp8_workspace_bytes.argtypes = [PT]
    lib.attn_score_recompute.restype = ctypes.c_int
    lib.attn_score_recompute.argtypes = [PT, PT, PT, PT, ctypes.c_int32, ctypes.c_int,
                                         ctypes.c_float, PT, PT, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.c_uint32, ctypes.c_void_p]
    lib.attn_score_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_score_workspace_bytes.argtypes = [PT, PT, PT, ctypes.c_int32]
    lib.attn_sparse_bwd.restype = ctypes.c_int
    lib.attn_sparse_bwd.argtypes = [PT, PT, PT, PT, PT, PT, PT, PT, ctypes.c_float, PT, PT, PT,
                                    ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32,
                                    ctypes.c_void_p]
    lib.attn_sparse_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_sparse_bwd_workspace_bytes.argtypes = [PT, PT, ctypes.c_int]
    lib.attn_bwd.restype = ctypes.c_int
    lib.attn_bwd.argtypes = [PT, PT, PT, PT, PT, PT, PT, PT, ctypes.c_int32, ctypes.c_int,
                             ctypes.c_float, PT, PT, PT, ctypes.c_void_p, ctypes.c_size_t,
                             ctypes.c_uint32, ctypes.c_void_p]
    lib.attn_bwd_noalloc.restype = ctypes.c_int
    lib.attn_bwd_noalloc.argtypes = [PT, PT, PT, PT, PT, PT, PT, PT, ctypes.c_int32, ctypes.c_int,
                                     ctypes.c_float, PT, PT, PT, ctypes.c_uint32, ctypes.c_void_p]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd_workspace_bytes.argtypes = [PT, PT, ctypes.c_uint32]
    lib.attn_get_error.restype = ctypes.c_int
    lib.attn_get_error.argtypes = [ctypes.c_void_p]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_strerror.argtypes = [ctypes.c_int]
    lib.attn_last_cuda_error.restype = ctypes.c_char_p
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_version.restype = ctypes.c_int
    lib.attn_version.argtypes = []
    lib.attn_profile_events.restype = ctypes.c_int
    lib.attn_profile_events.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.attn_launch_count.restype = ctypes.c_ulonglong
    lib.attn_launch_count.argtypes = []
    lib.attn_selftest_wait_timeout.restype = ctypes.c_int
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    return lib


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        lib = load()
        text = lib.attn_strerror(code).decode()
        if code == -7:
            text += "; " + lib.attn_last_cuda_error().decode()
        super().__init__("%s failed: %s (%s)" % (where, ERRORS.get(code, code), text))


def check(code: int, where: str):
    if code != 0:
        raise AttnError(code, where)
