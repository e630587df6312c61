"""ctypes binding of libtmg.so (include/tmg.h).  Argument marshalling only:
every step of the GEMM runs in the library's CUDA kernels.

Loading fails loudly (TmgError) when the shared library has not been built;
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtmg.so")
# the same library built with bounds checks in its kernels (build.py --debug-bounds)
DEBUG_LIB_PATH = os.path.join(HERE, "libtmg_debug.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = 0, 1, 2, 3, 4, 5
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT", 5: "BOUNDS"}
F32, BF16, E4M3 = 0, 1, 2
EPILOGUES = {"none": 0, "bias": 1, "bias_relu": 2, "bias_silu": 3, "bias_gelu": 4}
PATHS = {"auto": 0, "ffma": 1, "tc": 2, "skinny": 3, "skinny_ffma": 4, "tc_single": 5,
         "tc_pair": 6, "packed_tc": 7}

# Every function include/tmg.h declares.
EXPORTS = ("tmg_gemm", "tmg_gemm_ex", "tmg_gemm_host", "tmg_gemm_fused", "tmg_gemm_w4a8",
           "tmg_gemm_w4a8_preshuffled", "tmg_w4a8_preshuffle", "tmg_w4a8_preshuffled_bytes", "tmg_gemm_mxfp4", "tmg_gemm_skinny_noalloc", "tmg_check", "tmg_last_error",
           "tmg_set_wait_budget_ns", "tmg_debug_wait_timeout", "tmg_debug_bounds_probe", "tmg_debug_build",
           "tmg_launch_count",
           "tmg_version", "tmg_shutdown")


class TmgError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"tmg {STATUS_NAMES.get(status, status)}: {message}")


class Layout(ctypes.Structure):
    _fields_ = [
        ("depth", ctypes.c_int32 * 2),
        ("shape", (ctypes.c_int64 * 2) * 2),
        ("stride", (ctypes.c_int64 * 2) * 2),
    ]


def make_layout(shape, stride) -> Layout:
    """(Shape, Stride) with two top-level modes; each mode an int or a pair,
    e.g. ``make_layout((9, (4, 8)), (1, (9, 36)))``."""
    if len(shape) != 2 or len(stride) != 2:
        raise ValueError("a layout has exactly two top-level modes")
    L = Layout()
    for t in range(2):
        s, d = shape[t], stride[t]
        if isinstance(s, (tuple, list)):
            if len(s) != 2 or not isinstance(d, (tuple, list)) or len(d) != 2:
                raise ValueError("a nested mode holds exactly two sub-modes")
            L.depth[t] = 2
            L.shape[t][0], L.shape[t][1] = int(s[0]), int(s[1])
            L.stride[t][0], L.stride[t][1] = int(d[0]), int(d[1])
        else:
            L.depth[t] = 1
            L.shape[t][0], L.shape[t][1] = int(s), 1
            L.stride[t][0], L.stride[t][1] = int(d), 0
    return L


_lib = None


def use_library(path: str) -> None:
    """Bind every later call to another build of the same ABI (the debug
    build, DEBUG_LIB_PATH); the next lib() call loads it."""
    global _lib, LIB_PATH
    LIB_PATH = path
    _lib = None


def lib():
    """Load libtmg.so once; raise TmgError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise TmgError(ERR_CUDA, f"{LIB_PATH} is missing: build it with "
                                 "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    LP = ctypes.POINTER(Layout)
    L.tmg_gemm.argtypes = [P, P, P, I64, I64, I64, ctypes.c_int, LP, LP, LP, P]
    L.tmg_gemm.restype = ctypes.c_int
    L.tmg_gemm_ex.argtypes = [P, P, P, I64, I64, I64, ctypes.c_int, LP, LP, LP, ctypes.c_int, P]
    L.tmg_gemm_ex.restype = ctypes.c_int
    L.tmg_gemm_host.argtypes = [P, P, P, I64, I64, I64, ctypes.c_int, P]
    L.tmg_gemm_host.restype = ctypes.c_int
    L.tmg_gemm_fused.argtypes = [P, P, P, I64, I64, I64, ctypes.c_int, P, P, P, ctypes.c_int, P]
    L.tmg_gemm_fused.restype = ctypes.c_int
    L.tmg_gemm_w4a8.argtypes = [P, P, P, I64, I64, I64, P]
    L.tmg_gemm_w4a8.restype = ctypes.c_int
    L.tmg_gemm_w4a8_preshuffled.argtypes = [P, P, P, I64, I64, I64, P]
    L.tmg_gemm_w4a8_preshuffled.restype = ctypes.c_int
    L.tmg_w4a8_preshuffle.argtypes = [P, P, I64, I64, P]
    L.tmg_w4a8_preshuffle.restype = ctypes.c_int
    L.tmg_w4a8_preshuffled_bytes.argtypes = [I64, I64]
    L.tmg_w4a8_preshuffled_bytes.restype = ctypes.c_size_t
    L.tmg_gemm_mxfp4.argtypes = [P, P, P, P, P, I64, I64, I64, P]
    L.tmg_gemm_mxfp4.restype = ctypes.c_int
    L.tmg_gemm_skinny_noalloc.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, P]
    L.tmg_gemm_skinny_noalloc.restype = ctypes.c_int
    L.tmg_check.argtypes = [P]
    L.tmg_check.restype = ctypes.c_int
    L.tmg_last_error.argtypes = []
    L.tmg_last_error.restype = ctypes.c_char_p
    L.tmg_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
    L.tmg_set_wait_budget_ns.restype = None
    L.tmg_debug_wait_timeout.argtypes = [ctypes.c_uint64, P]
    L.tmg_debug_wait_timeout.restype = ctypes.c_int
    L.tmg_debug_bounds_probe.argtypes = [P]
    L.tmg_debug_bounds_probe.restype = ctypes.c_int
    L.tmg_debug_build.argtypes = []
    L.tmg_debug_build.restype = ctypes.c_int
    L.tmg_launch_count.argtypes = []
    L.tmg_launch_count.restype = ctypes.c_uint64
    L.tmg_version.argtypes = []
    L.tmg_version.restype = ctypes.c_int
    L.tmg_shutdown.argtypes = []
    L.tmg_shutdown.restype = None
    _lib = L
    return _lib


def raise_on(status: int) -> None:
    if status != OK:
        msg = lib().tmg_last_error()
        raise TmgError(status, msg.decode() if msg else "")
