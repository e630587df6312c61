"""CPU oracle for the tiled GEMM D = A·Bᵀ — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it and
shares no code with it: the oracle is a plain C file (``oracle.c``) compiled
with gcc into ``liboracle.so`` and called here through ctypes.

What it computes, and the passages it follows, is stated at the top of
``oracle.c``.  Every function is pinned by ``tests/test_oracle_pins.py``.
No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32 = 0
BF16 = 1
E4M3 = 2

# Epilogues of the fused GEMM (see orc_gemm_fused in oracle.c).
EPILOGUES = {"none": 0, "bias": 1, "bias_relu": 2, "bias_silu": 3, "bias_gelu": 4}


class Layout(ctypes.Structure):
    """Rank-2 (shape, stride) layout, each top mode with 1 or 2 sub-modes."""

    _fields_ = [
        ("depth", ctypes.c_int32 * 2),
        ("shape", (ctypes.c_int64 * 2) * 2),
        ("stride", (ctypes.c_int64 * 2) * 2),
    ]


def make_layout(shape, stride) -> Layout:
    """Build a layout from nested tuples, e.g. ``((9, (4, 8)), (1, (9, 36)))``.

    Each top mode is an int or a 2-tuple of ints."""
    if len(shape) != 2 or len(stride) != 2:
        raise ValueError("layout must have exactly two top-level modes")
    L = Layout()
    for t in range(2):
        s, d = shape[t], stride[t]
        if isinstance(s, (tuple, list)):
            if len(s) != 2 or len(d) != 2:
                raise ValueError("nested modes hold exactly two sub-modes")
            L.depth[t] = 2
            L.shape[t][0], L.shape[t][1] = int(s[0]), int(s[1])
            L.stride[t][0], L.stride[t][1] = int(d[0]), int(d[1])
        else:
            L.depth[t] = 1
            L.shape[t][0], L.shape[t][1] = int(s), 1
            L.stride[t][0], L.stride[t][1] = int(d), 0
    return L


def row_major(rows: int, cols: int, ld: int | None = None) -> Layout:
    return make_layout((rows, cols), (cols if ld is None else ld, 1))


def col_major(rows: int, cols: int, ld: int | None = None) -> Layout:
    return make_layout((rows, cols), (1, rows if ld is None else ld))


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (OpenMP, no fast-math) if stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        LP = ctypes.POINTER(Layout)
        L.orc_crd2idx.argtypes = [I64, I64, LP]
        L.orc_crd2idx.restype = I64
        L.orc_idx2crd.argtypes = [I64, LP, ctypes.POINTER(I64), ctypes.POINTER(I64)]
        L.orc_idx2crd.restype = None
        L.orc_mode_size.argtypes = [LP, I32]
        L.orc_mode_size.restype = I64
        L.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        L.orc_decode_bf16.restype = ctypes.c_double
        L.orc_decode_f32.argtypes = [ctypes.c_uint32]
        L.orc_decode_f32.restype = ctypes.c_double
        L.orc_decode_e2m1.argtypes = [ctypes.c_uint8]
        L.orc_decode_e2m1.restype = ctypes.c_double
        L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
        L.orc_decode_e4m3.restype = ctypes.c_double
        L.orc_activation.argtypes = [ctypes.c_double, I32]
        L.orc_activation.restype = ctypes.c_double
        L.orc_gemm_fused.argtypes = [P, P, I32, I64, I64, I64, P, P, P, I32, P, I32]
        L.orc_gemm_fused.restype = I32
        L.orc_gemm_fused_entries.argtypes = [P, P, I32, I64, P, P, P, I32, P, P, I64, P, I32]
        L.orc_gemm_fused_entries.restype = I32
        L.orc_decode_int4.argtypes = [ctypes.c_uint8]
        L.orc_decode_int4.restype = I32
        L.orc_gemm_w4a8.argtypes = [P, P, I64, I64, I64, P, I32]
        L.orc_gemm_w4a8.restype = I32
        L.orc_gemm_w4a8_entries.argtypes = [P, P, I64, P, P, I64, P, I32]
        L.orc_gemm_w4a8_entries.restype = I32
        L.orc_decode_e8m0.argtypes = [ctypes.c_uint8]
        L.orc_decode_e8m0.restype = ctypes.c_double
        L.orc_round_bf16.argtypes = [ctypes.c_double]
        L.orc_round_bf16.restype = ctypes.c_uint16
        L.orc_round_bf16_array.argtypes = [P, I64, P]
        L.orc_round_bf16_array.restype = None
        L.orc_read_matrix.argtypes = [P, LP, I32, I64, I64, P]
        L.orc_read_matrix.restype = I32
        L.orc_gemm.argtypes = [P, LP, P, LP, I32, I64, I64, I64, P, I32]
        L.orc_gemm.restype = I32
        L.orc_gemm_entries.argtypes = [P, LP, P, LP, I32, I64, P, P, I64, P, I32]
        L.orc_gemm_entries.restype = I32
        L.orc_gemm_mxfp4.argtypes = [P, P, P, P, I64, I64, I64, P, I32]
        L.orc_gemm_mxfp4.restype = I32
        L.orc_gemm_mxfp4_entries.argtypes = [P, P, P, P, I64, P, P, I64, P, I32]
        L.orc_gemm_mxfp4_entries.restype = I32
        L.orc_read_mxfp4.argtypes = [P, P, I64, I64, P]
        L.orc_read_mxfp4.restype = I32
        L.orc_max_threads.argtypes = []
        L.orc_max_threads.restype = I32
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Raw element bits as a contiguous numpy array (uint32 or uint16)."""
    want = np.uint32 if dtype == F32 else np.uint16
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32 and dtype == F32:
        return x.view(np.uint32)
    if x.dtype != want:
        raise TypeError(f"expected {want} bits, got {x.dtype}")
    return x


def crd2idx(row: int, col: int, layout: Layout) -> int:
    return lib().orc_crd2idx(row, col, ctypes.byref(layout))


def idx2crd(idx: int, layout: Layout) -> tuple[int, int]:
    r, c = ctypes.c_int64(), ctypes.c_int64()
    lib().orc_idx2crd(idx, ctypes.byref(layout), ctypes.byref(r), ctypes.byref(c))
    return r.value, c.value


def mode_size(layout: Layout, t: int) -> int:
    return lib().orc_mode_size(ctypes.byref(layout), t)


def decode_bf16(bits: int) -> float:
    return lib().orc_decode_bf16(bits)


def decode_e2m1(code: int) -> float:
    return lib().orc_decode_e2m1(code)


def decode_e4m3(code: int) -> float:
    return lib().orc_decode_e4m3(code)


def activation(y: float, epilogue: str) -> float:
    return lib().orc_activation(float(y), EPILOGUES[epilogue])


def _elem_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    want = np.uint16 if dtype == BF16 else np.uint8
    x = np.ascontiguousarray(x)
    if x.dtype != want:
        raise TypeError(f"expected {want} elements, got {x.dtype}")
    return x


def _vec(v, n: int):
    if v is None:
        return None, None
    a = np.ascontiguousarray(v, dtype=np.float32)
    if a.shape != (n,):
        raise ValueError(f"vector of shape {a.shape}, expected ({n},)")
    return a, a.ctypes.data


def gemm_fused(A: np.ndarray, B: np.ndarray, dtype: int, M: int, N: int, K: int,
               scale_a=None, scale_b=None, bias=None, epilogue: str = "none",
               threads: int = 0) -> np.ndarray:
    """act(A·Bᵀ * scale_a[m] * scale_b[n] + bias[n]) in fp64, (M, N).
    A (M,K) and B (N,K) dense row-major bits: uint16 (bf16) or uint8 (E4M3)."""
    Ab, Bb = _elem_bits(A, dtype), _elem_bits(B, dtype)
    (sa, psa), (sb, psb), (bi, pbi) = _vec(scale_a, M), _vec(scale_b, N), _vec(bias, N)
    D = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_gemm_fused(_ptr(Ab), _ptr(Bb), dtype, M, N, K, psa, psb, pbi,
                              EPILOGUES[epilogue], _ptr(D), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_fused failed ({rc})")
    return D


def gemm_fused_entries(A: np.ndarray, B: np.ndarray, dtype: int, M: int, N: int, K: int, ms, ns,
                       scale_a=None, scale_b=None, bias=None, epilogue: str = "none",
                       threads: int = 0) -> np.ndarray:
    """Outputs (ms[i], ns[i]) of gemm_fused, each summed directly."""
    Ab, Bb = _elem_bits(A, dtype), _elem_bits(B, dtype)
    (sa, psa), (sb, psb), (bi, pbi) = _vec(scale_a, M), _vec(scale_b, N), _vec(bias, N)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape[0], dtype=np.float64)
    rc = lib().orc_gemm_fused_entries(_ptr(Ab), _ptr(Bb), dtype, K, psa, psb, pbi,
                                      EPILOGUES[epilogue], _ptr(ms), _ptr(ns), ms.shape[0],
                                      _ptr(out), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_fused_entries failed ({rc})")
    return out


def decode_e8m0(byte: int) -> float:
    return lib().orc_decode_e8m0(byte)


def round_bf16(x: float) -> int:
    return lib().orc_round_bf16(float(x))


def round_bf16_array(x: np.ndarray) -> np.ndarray:
    """orc_round_bf16 applied to every element (bf16 bit patterns)."""
    flat = np.ascontiguousarray(np.asarray(x, dtype=np.float64).ravel())
    out = np.empty(flat.shape[0], dtype=np.uint16)
    lib().orc_round_bf16_array(_ptr(flat), flat.shape[0], _ptr(out))
    return out.reshape(np.shape(x))


def read_matrix(x: np.ndarray, layout: Layout, dtype: int, rows: int, cols: int) -> np.ndarray:
    """Decode the (rows, cols) logical matrix stored in ``x`` through layout."""
    xb = _bits(x, dtype)
    out = np.empty((rows, cols), dtype=np.float64)
    rc = lib().orc_read_matrix(_ptr(xb), ctypes.byref(layout), dtype, rows, cols, _ptr(out))
    if rc:
        raise RuntimeError(f"orc_read_matrix failed ({rc})")
    return out


def gemm(A: np.ndarray, layoutA: Layout, B: np.ndarray, layoutB: Layout, dtype: int,
         M: int, N: int, K: int, threads: int = 0) -> np.ndarray:
    """Full D = A·Bᵀ in fp64 as a dense (M, N) array."""
    Ab, Bb = _bits(A, dtype), _bits(B, dtype)
    D = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_gemm(_ptr(Ab), ctypes.byref(layoutA), _ptr(Bb), ctypes.byref(layoutB),
                        dtype, M, N, K, _ptr(D), threads)
    if rc:
        raise RuntimeError(f"orc_gemm failed ({rc})")
    return D


def gemm_entries(A: np.ndarray, layoutA: Layout, B: np.ndarray, layoutB: Layout, dtype: int,
                 K: int, ms, ns, threads: int = 0) -> np.ndarray:
    """D[ms[i], ns[i]] for each i, summed directly from the encoded operands."""
    Ab, Bb = _bits(A, dtype), _bits(B, dtype)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape[0], dtype=np.float64)
    rc = lib().orc_gemm_entries(_ptr(Ab), ctypes.byref(layoutA), _ptr(Bb), ctypes.byref(layoutB),
                                dtype, K, _ptr(ms), _ptr(ns), ms.shape[0], _ptr(out), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_entries failed ({rc})")
    return out


def gemm_mxfp4(A: np.ndarray, B: np.ndarray, sA: np.ndarray, sB: np.ndarray,
               M: int, N: int, K: int, threads: int = 0) -> np.ndarray:
    A, B = np.ascontiguousarray(A, np.uint8), np.ascontiguousarray(B, np.uint8)
    sA, sB = np.ascontiguousarray(sA, np.uint8), np.ascontiguousarray(sB, np.uint8)
    D = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_gemm_mxfp4(_ptr(A), _ptr(B), _ptr(sA), _ptr(sB), M, N, K, _ptr(D), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_mxfp4 failed ({rc})")
    return D


def gemm_mxfp4_entries(A: np.ndarray, B: np.ndarray, sA: np.ndarray, sB: np.ndarray,
                       K: int, ms, ns, threads: int = 0) -> np.ndarray:
    A, B = np.ascontiguousarray(A, np.uint8), np.ascontiguousarray(B, np.uint8)
    sA, sB = np.ascontiguousarray(sA, np.uint8), np.ascontiguousarray(sB, np.uint8)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape[0], dtype=np.float64)
    rc = lib().orc_gemm_mxfp4_entries(_ptr(A), _ptr(B), _ptr(sA), _ptr(sB), K,
                                      _ptr(ms), _ptr(ns), ms.shape[0], _ptr(out), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_mxfp4_entries failed ({rc})")
    return out


def read_mxfp4(X: np.ndarray, S: np.ndarray, rows: int, K: int) -> np.ndarray:
    X, S = np.ascontiguousarray(X, np.uint8), np.ascontiguousarray(S, np.uint8)
    out = np.empty((rows, K), dtype=np.float64)
    rc = lib().orc_read_mxfp4(_ptr(X), _ptr(S), rows, K, _ptr(out))
    if rc:
        raise RuntimeError(f"orc_read_mxfp4 failed ({rc})")
    return out


def max_threads() -> int:
    return lib().orc_max_threads()


def decode_int4(nibble: int) -> int:
    return lib().orc_decode_int4(nibble)


def gemm_w4a8(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, threads: int = 0) -> np.ndarray:
    """Exact int64 D = A·Bᵀ: A (M, K) int8, B (N, K/2) packed int4 (even k low nibble)."""
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    D = np.empty((M, N), dtype=np.int64)
    rc = lib().orc_gemm_w4a8(_ptr(A), _ptr(B), M, N, K, _ptr(D), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_w4a8 failed ({rc})")
    return D


def gemm_w4a8_entries(A: np.ndarray, B: np.ndarray, K: int, ms, ns, threads: int = 0) -> np.ndarray:
    A = np.ascontiguousarray(A, dtype=np.int8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape[0], dtype=np.int64)
    rc = lib().orc_gemm_w4a8_entries(_ptr(A), _ptr(B), K, _ptr(ms), _ptr(ns), ms.shape[0], _ptr(out), threads)
    if rc:
        raise RuntimeError(f"orc_gemm_w4a8_entries failed ({rc})")
    return out
