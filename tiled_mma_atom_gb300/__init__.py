"""tiled_mma_atom_gb300 — tiled GEMM D = A·Bᵀ (fp32 accumulate) for GB300.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
(``csrc/``, built into ``libtmg.so``; ABI in ``include/tmg.h``).  This
package marshals torch tensors into that library's calls and nothing else.
Importing the package does not load the library; the first call does, and
raises ``TmgError`` if it is missing.

Layouts.  A torch tensor's (shape, stride) already is a (Shape, Stride)
layout in the FlyDSL sense ("FlyDSL Kernel Authoring Skill", §2 Layout
System): by default each operand's layout is taken from its tensor —
A over (m,k), B over (n,k), D over (m,n).  Pass an explicit layout
(``make_layout(shape, stride)``, modes nested at most one level) to read a
buffer any other way; the buffer is then addressed through crd2idx from
the tensor's data pointer.
"""
from __future__ import annotations

import torch

from . import _native
from ._native import (BF16, E4M3, EPILOGUES, F32, PATHS, Layout, TmgError, make_layout)  # noqa: F401

__all__ = ["gemm", "gemm_host", "gemm_fused", "gemm_w4a8", "gemm_w4a8_preshuffled", "w4a8_preshuffle",
           "w4a8_preshuffled_bytes", "gemm_mxfp4", "check", "make_layout", "Layout", "TmgError",
           "set_wait_budget_ns", "debug_wait_timeout", "launch_count", "version",
           "shutdown", "PATHS"]


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _layout_of(t: torch.Tensor, rows: int, cols: int) -> Layout:
    if t.dim() != 2 or tuple(t.shape) != (rows, cols):
        raise ValueError(f"tensor of shape {tuple(t.shape)} is not ({rows}, {cols}); "
                         "pass an explicit layout")
    return make_layout((rows, cols), (t.stride(0), t.stride(1)))


def _as_layout(spec, t: torch.Tensor, rows: int, cols: int):
    if spec is None:
        if t.dim() == 2 and t.shape[0] == rows and t.shape[1] == cols and t.is_contiguous():
            return None          # the library's default: row-major (rows, cols):(cols, 1)
        return _layout_of(t, rows, cols)
    if isinstance(spec, Layout):
        return spec
    shape, stride = spec
    return make_layout(shape, stride)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def gemm(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor | None = None, *,
         M: int | None = None, N: int | None = None, K: int | None = None,
         layoutA=None, layoutB=None, layoutD=None, path: str = "auto",
         stream=None) -> torch.Tensor:
    """D = A·Bᵀ on the GPU, fp32 accumulation.  A is (M,K), B is (N,K), D is
    (M,N); all three share dtype float32 or bfloat16 and live on the GPU.
    Returns D (allocated row-major if not given).  Asynchronous on `stream`
    (default: torch's current stream)."""
    if M is None:
        M = A.shape[0] if layoutA is None else None
    if K is None:
        K = A.shape[1] if layoutA is None else None
    if N is None:
        N = B.shape[0] if layoutB is None else None
    if M is None or N is None or K is None:
        raise ValueError("give M, N and K when passing explicit layouts")
    if D is None:
        D = torch.empty((M, N), dtype=A.dtype, device=A.device)
    dt = _dtype_code(A)
    if B.dtype != A.dtype or D.dtype != A.dtype:
        raise TypeError("A, B and D must share one dtype")
    if not (A.is_cuda and B.is_cuda and D.is_cuda):
        raise ValueError("A, B and D must be CUDA tensors")
    la = _as_layout(layoutA, A, M, K)
    lb = _as_layout(layoutB, B, N, K)
    ld = _as_layout(layoutD, D, M, N)
    L = _native.lib()
    st = L.tmg_gemm_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, dt,
                       la, lb, ld, PATHS[path], _stream_handle(stream))
    _native.raise_on(st)
    return D


def gemm_host(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor | None = None, *,
              stream=None) -> torch.Tensor:
    """D = A·Bᵀ from host memory: A (M,K) and B (N,K) contiguous CPU tensors
    (float32 or bfloat16, pinned for full speed), D (M,N) a CPU tensor of the
    same dtype (allocated pinned if not given).  The library moves the data
    and overlaps the transfers with the GEMM; the call returns once the work
    is queued on `stream` — synchronise it before reading D."""
    for name, t in (("A", A), ("B", B)):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D CPU tensor")
    if A.dtype != B.dtype or A.shape[1] != B.shape[1]:
        raise ValueError("A (M,K) and B (N,K) must share dtype and K")
    M, K = A.shape
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=A.dtype).pin_memory()
    if D.is_cuda or D.dtype != A.dtype or tuple(D.shape) != (M, N) or not D.is_contiguous():
        raise ValueError("D must be a contiguous CPU tensor of shape (M, N) and A's dtype")
    st = _native.lib().tmg_gemm_host(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, _dtype_code(A),
                                     _stream_handle(stream))
    _native.raise_on(st)
    return D


def _fp32_vec(v, n: int, name: str, dev):
    if v is None:
        return None
    if v.dtype != torch.float32 or tuple(v.shape) != (n,) or not v.is_contiguous() or v.device != dev:
        raise ValueError(f"{name} must be a contiguous float32 tensor of shape ({n},) on {dev}")
    return v.data_ptr()


def gemm_fused(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor | None = None, *,
               scale_a: torch.Tensor | None = None, scale_b: torch.Tensor | None = None,
               bias: torch.Tensor | None = None, epilogue: str = "none", stream=None) -> torch.Tensor:
    """D = bf16(act(A·Bᵀ · scale_a[m] · scale_b[n] + bias[n])), fp32 accumulation.

    A (M,K) and B (N,K): contiguous CUDA tensors of dtype bfloat16 or
    float8_e4m3fn (both the same).  scale_a (M,), scale_b (N,), bias (N,):
    float32 or None.  epilogue: "none", "bias", "bias_relu", "bias_silu",
    "bias_gelu" (GELU in its erf form).  D: bfloat16 (M,N), allocated if not
    given.  Asynchronous on `stream`."""
    if A.dtype != B.dtype:
        raise TypeError("A and B must share one dtype")
    if A.dtype == torch.bfloat16:
        dt = BF16
    elif A.dtype == torch.float8_e4m3fn:
        dt = E4M3
    else:
        raise TypeError(f"unsupported input dtype {A.dtype}: use bfloat16 or float8_e4m3fn")
    if epilogue not in EPILOGUES:
        raise ValueError(f"unknown epilogue {epilogue!r}; one of {sorted(EPILOGUES)}")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("A must be (M,K) and B (N,K)")
    M, K = A.shape
    N = B.shape[0]
    for name, t in (("A", A), ("B", B)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N) or not D.is_contiguous():
        raise ValueError("D must be a contiguous bfloat16 tensor of shape (M, N)")
    st = _native.lib().tmg_gemm_fused(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, dt,
                                      _fp32_vec(scale_a, M, "scale_a", A.device),
                                      _fp32_vec(scale_b, N, "scale_b", A.device),
                                      _fp32_vec(bias, N, "bias", A.device),
                                      EPILOGUES[epilogue], _stream_handle(stream))
    _native.raise_on(st)
    return D


def gemm_w4a8(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor | None = None, *,
              stream=None) -> torch.Tensor:
    """W4A8 GEMM, exact: A (M,K) int8, B (N, K/2) uint8 holding two signed
    int4 per byte (even k in the low nibble), D (M,N) int32.  All contiguous
    on the GPU."""
    if A.dtype != torch.int8 or A.dim() != 2 or not A.is_contiguous() or not A.is_cuda:
        raise ValueError("A must be a contiguous CUDA int8 tensor of shape (M, K)")
    M, K = A.shape
    if B.dtype != torch.uint8 or B.dim() != 2 or B.shape[1] * 2 != K or not B.is_contiguous() or not B.is_cuda:
        raise ValueError("B must be a contiguous CUDA uint8 tensor of shape (N, K/2)")
    N = B.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=torch.int32, device=A.device)
    if D.dtype != torch.int32 or tuple(D.shape) != (M, N) or not D.is_contiguous():
        raise ValueError("D must be a contiguous int32 tensor of shape (M, N)")
    _native.raise_on(_native.lib().tmg_gemm_w4a8(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                                  _stream_handle(stream)))
    return D


def w4a8_preshuffled_bytes(N: int, K: int) -> int:
    """Size of the pre-shuffled image of (N, K/2) packed int4 weights; 0
    unless N > 0, K > 0 and K is a multiple of 32."""
    return int(_native.lib().tmg_w4a8_preshuffled_bytes(N, K))


def w4a8_preshuffle(B: torch.Tensor, *, stream=None) -> torch.Tensor:
    """Pre-shuffle packed int4 weights B (N, K/2) uint8 into the decode
    kernel's tile order (16 KB blocks of 128 rows x 256 k, each contiguous);
    returns the 1-D uint8 image for gemm_w4a8_preshuffled.  K % 32 == 0."""
    if B.dtype != torch.uint8 or B.dim() != 2 or not B.is_contiguous() or not B.is_cuda:
        raise ValueError("B must be a contiguous CUDA uint8 tensor of shape (N, K/2)")
    N, K = B.shape[0], B.shape[1] * 2
    nbytes = w4a8_preshuffled_bytes(N, K)
    if nbytes == 0:
        raise ValueError(f"pre-shuffled weights need N > 0 and K a positive multiple of 32 (N={N}, K={K})")
    Bs = torch.empty(nbytes, dtype=torch.uint8, device=B.device)
    _native.raise_on(_native.lib().tmg_w4a8_preshuffle(B.data_ptr(), Bs.data_ptr(), N, K, _stream_handle(stream)))
    return Bs


def gemm_w4a8_preshuffled(A: torch.Tensor, Bs: torch.Tensor, N: int, D: torch.Tensor | None = None, *,
                          stream=None) -> torch.Tensor:
    """gemm_w4a8 with the weights given as w4a8_preshuffle's image Bs of an
    (N, K/2) matrix; same exact int32 result."""
    if A.dtype != torch.int8 or A.dim() != 2 or not A.is_contiguous() or not A.is_cuda:
        raise ValueError("A must be a contiguous CUDA int8 tensor of shape (M, K)")
    M, K = A.shape
    if Bs.dtype != torch.uint8 or not Bs.is_contiguous() or not Bs.is_cuda or \
            Bs.numel() != w4a8_preshuffled_bytes(N, K):
        raise ValueError("Bs must be the contiguous CUDA image w4a8_preshuffle made of (N, K/2) weights")
    if D is None:
        D = torch.empty((M, N), dtype=torch.int32, device=A.device)
    if D.dtype != torch.int32 or tuple(D.shape) != (M, N) or not D.is_contiguous():
        raise ValueError("D must be a contiguous int32 tensor of shape (M, N)")
    _native.raise_on(_native.lib().tmg_gemm_w4a8_preshuffled(A.data_ptr(), Bs.data_ptr(), D.data_ptr(), M, N, K,
                                                              _stream_handle(stream)))
    return D


def gemm_mxfp4(A: torch.Tensor, B: torch.Tensor, scaleA: torch.Tensor, scaleB: torch.Tensor,
               D: torch.Tensor | None = None, *, stream=None) -> torch.Tensor:
    """MXFP4 GEMM.  A: (M, K/2) uint8, two e2m1 codes per byte (even k in the
    low nibble); B: (N, K/2); scaleA: (M, K/32) uint8 e8m0; scaleB: (N, K/32).
    D: (M, N) bfloat16.  All contiguous on the GPU."""
    M, K2 = A.shape
    N = B.shape[0]
    K = 2 * K2
    for name, t, shape in (("A", A, (M, K2)), ("B", B, (N, K2)), ("scaleA", scaleA, (M, K // 32)),
                           ("scaleB", scaleB, (N, K // 32))):
        if t.dtype != torch.uint8 or tuple(t.shape) != shape or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor of shape {shape}")
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N) or not D.is_contiguous():
        raise ValueError("D must be a contiguous bfloat16 tensor of shape (M, N)")
    st = _native.lib().tmg_gemm_mxfp4(A.data_ptr(), B.data_ptr(), scaleA.data_ptr(),
                                      scaleB.data_ptr(), D.data_ptr(), M, N, K,
                                      _stream_handle(stream))
    _native.raise_on(st)
    return D


def check(stream=None) -> None:
    """Synchronise and raise TmgError if a kernel reported a timeout or a CUDA
    error occurred."""
    _native.raise_on(_native.lib().tmg_check(_stream_handle(stream)))


def set_wait_budget_ns(ns: int) -> None:
    _native.lib().tmg_set_wait_budget_ns(int(ns))


def debug_wait_timeout(budget_ns: int, stream=None) -> None:
    _native.raise_on(_native.lib().tmg_debug_wait_timeout(int(budget_ns), _stream_handle(stream)))


def launch_count() -> int:
    return int(_native.lib().tmg_launch_count())


def version() -> int:
    return int(_native.lib().tmg_version())


def shutdown() -> None:
    _native.lib().tmg_shutdown()
