"""Parity helpers shared by the GPU tests: run the CUDA path, run the oracle on
the same bits, compare within the stated bounds.

Bounds (stated once, used everywhere):
  * fp32 path: normwise max|D - D_ref| / max|D_ref| <= 1e-5.
  * bf16 / MXFP4 paths: per element |D - D_ref| <= 2e-2 * sqrt(K) *
    max|A| * max|B|, and relative Frobenius error ||D - D_ref|| / ||D_ref||
    <= 5e-3.  (max|A| of MXFP4 is the largest decoded magnitude.)
  * fused GEMM (scales, bias, activation): per element |D - D_ref| <=
    1.13 * 2e-2 * sqrt(K) * max|A| * max|B| * max|scale_a| * max|scale_b|
    + 2^-8 |D_ref| (1.13 bounds the slope of relu, silu and gelu; the last
    term is the bf16 rounding of the result), relative Frobenius <= 5e-3.
  * exact cases (integer-valued inputs, identity/permutation/all-ones B):
    D must equal the bf16 round-to-nearest-even of the exact result, bit for
    bit (fp32 for the fp32 path).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tiled_mma_atom_gb300 import inputs

FP32_NORMWISE = 1e-5
BF16_ELEM_FACTOR = 2e-2
BF16_FRO = 5e-3


def to_f64(D: torch.Tensor) -> np.ndarray:
    return D.detach().float().cpu().numpy().astype(np.float64)


def check_fp32(D: torch.Tensor, ref: np.ndarray) -> float:
    d = to_f64(D)
    rel = np.abs(d - ref).max() / max(np.abs(ref).max(), 1e-300)
    assert rel <= FP32_NORMWISE, f"fp32 normwise error {rel:.3e} > {FP32_NORMWISE}"
    return rel


def check_bf16_values(d: np.ndarray, ref: np.ndarray, K: int, amax: float, bmax: float) -> dict:
    """d, ref: float64 arrays of the same shape (full matrix or a sample)."""
    err = np.abs(d - ref)
    bound = BF16_ELEM_FACTOR * np.sqrt(K) * amax * bmax
    fro = np.linalg.norm(d - ref) / max(np.linalg.norm(ref), 1e-300)
    assert np.all(np.isfinite(d)), "non-finite output"
    assert err.max() <= bound, f"max |D-Dref| {err.max():.4g} > bound {bound:.4g}"
    assert fro <= BF16_FRO, f"relative Frobenius {fro:.3e} > {BF16_FRO}"
    return {"max_err": float(err.max()), "bound": float(bound), "fro": float(fro)}


ACT_SLOPE = 1.13      # max |d act / dy| of relu (1), silu (1.0998) and gelu (1.1289)


def check_fused_values(d: np.ndarray, ref: np.ndarray, K: int, amax: float, bmax: float,
                       samax: float = 1.0, sbmax: float = 1.0) -> dict:
    err = np.abs(d - ref)
    bound = ACT_SLOPE * BF16_ELEM_FACTOR * np.sqrt(K) * amax * bmax * samax * sbmax + 2.0 ** -8 * np.abs(ref)
    fro = np.linalg.norm(d - ref) / max(np.linalg.norm(ref), 1e-300)
    assert np.all(np.isfinite(d)), "non-finite output"
    worst = float((err - bound).max())
    assert worst <= 0, f"max excess over the bound {worst:.4g} (max err {err.max():.4g})"
    assert fro <= BF16_FRO, f"relative Frobenius {fro:.3e} > {BF16_FRO}"
    return {"max_err": float(err.max()), "fro": float(fro)}


def check_bf16(D: torch.Tensor, ref: np.ndarray, K: int, amax: float, bmax: float) -> dict:
    return check_bf16_values(to_f64(D), ref, K, amax, bmax)


def check_exact_bf16(D_bits: np.ndarray, ref_exact: np.ndarray) -> None:
    want = oracle.round_bf16_array(ref_exact)
    bad = np.count_nonzero(D_bits != want)
    assert bad == 0, f"{bad} of {want.size} outputs differ from RNE(exact)"


def bf16_bits(D: torch.Tensor) -> np.ndarray:
    return D.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def absmax(t: torch.Tensor) -> float:
    return float(t.float().abs().max())


def ref_full(A: torch.Tensor, B: torch.Tensor, dtype: int, layoutA=None, layoutB=None,
             M=None, N=None, K=None) -> np.ndarray:
    """Oracle D for CPU tensors A, B (row-major unless layouts are given)."""
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    la = layoutA or oracle.row_major(M, K)
    lb = layoutB or oracle.row_major(N, K)
    return oracle.gemm(inputs.bits_of(A), la, inputs.bits_of(B), lb, dtype, M, N, K)


def ref_entries(A: torch.Tensor, B: torch.Tensor, dtype: int, ms, ns) -> np.ndarray:
    M, K = A.shape
    N = B.shape[0]
    return oracle.gemm_entries(inputs.bits_of(A), oracle.row_major(M, K), inputs.bits_of(B),
                               oracle.row_major(N, K), dtype, K, ms, ns)


def sample_coords(M: int, N: int, count: int, seed: int = 0):
    """Random (m, n) pairs plus the four corners and the last row/column."""
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, count)
    ns = rng.integers(0, N, count)
    edge_m = np.array([0, 0, M - 1, M - 1] + [M - 1] * 8 + list(rng.integers(0, M, 8)))
    edge_n = np.array([0, N - 1, 0, N - 1] + list(rng.integers(0, N, 8)) + [N - 1] * 8)
    return np.concatenate([ms, edge_m]), np.concatenate([ns, edge_n])
