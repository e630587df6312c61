"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers and packs them into the storage
formats the library accepts; it holds none of the GEMM's arithmetic.  It is
shared by the tests, the benchmark and the oracle checks so that every side
reads bit-identical inputs.

Storage formats:
  * fp32 / bf16 matrices: torch tensors; bf16 values are fp32 draws rounded
    by torch's own float->bfloat16 conversion.
  * MXFP4: e2m1 codes packed two per byte, even k in the low nibble, rows
    K-contiguous, shape (rows, K/2) uint8; e8m0 scales (rows, K/32) uint8.

Seeds: 1000 * workload_index + {0: A, 1: B, 2: scale A, 3: scale B}.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    M: int
    N: int
    K: int
    dtype: str          # "f32", "bf16", "e4m3", "mxfp4" or "w4a8"
    a_dist: str         # description of the value distribution
    b_dist: str
    epilogue: str | None = None   # fused GEMM (tmg_gemm_fused) epilogue, or None
    a_mn_major: bool = False      # A stored MN-major: the buffer is Aᵀ, (K, M) row-major
    b_preshuffled: bool = False   # W4A8: B handed to the GEMM as its pre-shuffled image
    b_mn_major: bool = False      # B stored MN-major: the buffer is Bᵀ, (K, N) row-major (C = A·B)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    "fp32_128": Workload("fp32_128", 0, 128, 128, 128, "f32", "U[-1,1]", "U[-1,1]"),
    "bf16_1024": Workload("bf16_1024", 1, 1024, 1024, 1024, "bf16", "N(0,1)", "N(0,1)"),
    "bf16_4096": Workload("bf16_4096", 2, 4096, 4096, 4096, "bf16", "N(0,1)", "N(0,1)"),
    "skinny_16x28672x8192": Workload("skinny_16x28672x8192", 3, 16, 28672, 8192, "bf16",
                                     "N(0,1)", "N(0,0.02)"),
    "mxfp4_8192": Workload("mxfp4_8192", 4, 8192, 8192, 8192, "mxfp4",
                           "e2m1 codes U{0..15}, e8m0 exp U[-4,4]",
                           "e2m1 codes U{0..15}, e8m0 exp U[-4,4]"),
    # fused GEMMs: scale_a, scale_b ~ U[0.5, 1.5], bias ~ N(0,1), fp32
    "e4m3_8192_bias_gelu": Workload("e4m3_8192_bias_gelu", 5, 8192, 8192, 8192, "e4m3",
                                    "N(0,1) -> e4m3", "N(0,1) -> e4m3", "bias_gelu"),
    "bf16_4096_bias_silu": Workload("bf16_4096_bias_silu", 6, 4096, 4096, 4096, "bf16",
                                    "N(0,1)", "N(0,1)", "bias_silu"),
    # W4A8: int8 A x packed int4 B -> int32
    "w4a8_8192": Workload("w4a8_8192", 8, 8192, 8192, 8192, "w4a8", "int8 U[-128,127]",
                          "int4 U[-8,7], packed"),
    "w4a8_16x28672x8192": Workload("w4a8_16x28672x8192", 9, 16, 28672, 8192, "w4a8", "int8 U[-128,127]",
                                   "int4 U[-8,7], packed, pre-shuffled once before timing",
                                   b_preshuffled=True),
    # general layout: A given column-major, (M,K):(1,M)
    "bf16_4096_a_mn_major": Workload("bf16_4096_a_mn_major", 7, 4096, 4096, 4096, "bf16",
                                     "N(0,1), stored MN-major", "N(0,1)", None, True),
    # C = A·B with B stored (K, N) row-major: B is MN-major, (N,K):(1,N)
    "bf16_4096_b_kn": Workload("bf16_4096_b_kn", 10, 4096, 4096, 4096, "bf16",
                               "N(0,1)", "N(0,1), stored (K,N) row-major", b_mn_major=True),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def uniform_f32(rows: int, cols: int, seed: int, lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    g = _gen(seed)
    return torch.rand((rows, cols), generator=g, dtype=torch.float32) * (hi - lo) + lo


def normal_bf16(rows: int, cols: int, seed: int, std: float = 1.0) -> torch.Tensor:
    g = _gen(seed)
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def normal_e4m3(rows: int, cols: int, seed: int, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) draws converted to OCP E4M3 (torch.float8_e4m3fn)."""
    g = _gen(seed)
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.float8_e4m3fn)


def uniform_vec(n: int, seed: int, lo: float = 0.5, hi: float = 1.5) -> torch.Tensor:
    g = _gen(seed)
    return torch.rand((n,), generator=g, dtype=torch.float32) * (hi - lo) + lo


def normal_vec(n: int, seed: int, std: float = 1.0) -> torch.Tensor:
    g = _gen(seed)
    return torch.randn((n,), generator=g, dtype=torch.float32) * std


def integer_valued(rows: int, cols: int, seed: int, lo: int = -2, hi: int = 2,
                   dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """Integers uniform in [lo, hi], stored exactly in fp32, bf16 or E4M3
    (|value| <= 16 is exact in E4M3)."""
    g = _gen(seed)
    return torch.randint(lo, hi + 1, (rows, cols), generator=g, dtype=torch.int32).to(torch.float32).to(dtype)


def hashed_int(rows: int, cols: int, seed: int, row0: int = 0, device="cpu",
               dtype: torch.dtype = torch.bfloat16, lo: int = -2, hi: int = 2) -> torch.Tensor:
    """Integers in [lo, hi] given by an integer hash of (row0 + r, c, seed):
    the same values on any device and for any slice of rows, so a very large
    operand can be built on the GPU in pieces while a CPU check regenerates
    only the rows it samples."""
    r = torch.arange(row0, row0 + rows, device=device, dtype=torch.int64)[:, None]
    c = torch.arange(cols, device=device, dtype=torch.int64)[None, :]
    h = (r * 7919 + c * 104729 + seed * 15485863) % 1000003
    h = (h * h + 12345) % 999983
    return (h % (hi - lo + 1) + lo).to(torch.float32).to(dtype)


def hashed_int_device(rows: int, cols: int, seed: int, device, dtype: torch.dtype = torch.bfloat16,
                      chunk_rows: int = 4096) -> torch.Tensor:
    """hashed_int for the whole (rows, cols) matrix, built on `device` in row
    slices (bounded temporary memory)."""
    out = torch.empty((rows, cols), dtype=dtype, device=device)
    for r0 in range(0, rows, chunk_rows):
        n = min(chunk_rows, rows - r0)
        out[r0:r0 + n] = hashed_int(n, cols, seed, row0=r0, device=device, dtype=dtype)
    return out


def random_int8(rows: int, cols: int, seed: int) -> torch.Tensor:
    """Uniform int8 in [-128, 127]."""
    g = _gen(seed)
    return torch.randint(-128, 128, (rows, cols), generator=g, dtype=torch.int32).to(torch.int8)


def random_int4_packed(rows: int, K: int, seed: int) -> torch.Tensor:
    """(rows, K/2) bytes; each nibble an independent uniform 4-bit code
    (a two's complement int4 in [-8, 7])."""
    if K % 2:
        raise ValueError("K must be even for packed int4")
    g = _gen(seed)
    return torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)


def random_fp4_codes(rows: int, K: int, seed: int) -> torch.Tensor:
    """(rows, K/2) bytes; each nibble an independent uniform e2m1 code."""
    if K % 2:
        raise ValueError("K must be even for packed fp4")
    g = _gen(seed)
    return torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)


def random_e8m0(rows: int, K: int, seed: int, lo: int = -4, hi: int = 4) -> torch.Tensor:
    """(rows, K/32) bytes 127 + e, e uniform in [lo, hi]."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    g = _gen(seed)
    e = torch.randint(lo, hi + 1, (rows, K // 32), generator=g, dtype=torch.int32)
    return (e + 127).to(torch.uint8)


def pack_fp4(codes: torch.Tensor) -> torch.Tensor:
    """Pack a (rows, K) tensor of 4-bit codes, even k into the low nibble."""
    c = codes.to(torch.int32)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).to(torch.uint8)


def make_inputs(w: Workload):
    """Inputs of a workload on the CPU.

    Returns (A, B) for f32/bf16 (A as its (K, M) buffer when the workload
    stores it MN-major), (A, B, scaleA, scaleB) for mxfp4 and
    (A, B, scale_a, scale_b, bias) for a fused workload."""
    M = w.M
    s = 1000 * w.index
    if w.epilogue is not None:
        gen = normal_e4m3 if w.dtype == "e4m3" else normal_bf16
        return (gen(M, w.K, s + 0), gen(w.N, w.K, s + 1), uniform_vec(M, s + 2),
                uniform_vec(w.N, s + 3), normal_vec(w.N, s + 4))
    if w.dtype == "f32":
        return uniform_f32(M, w.K, s + 0), uniform_f32(w.N, w.K, s + 1)
    if w.dtype == "bf16":
        std_b = 0.02 if w.name.startswith("skinny") else 1.0
        A = normal_bf16(M, w.K, s + 0)
        if w.a_mn_major:
            A = A.t().contiguous()
        B = normal_bf16(w.N, w.K, s + 1, std=std_b)
        if w.b_mn_major:
            B = B.t().contiguous()
        return A, B
    if w.dtype == "w4a8":
        return random_int8(M, w.K, s + 0), random_int4_packed(w.N, w.K, s + 1)
    if w.dtype == "mxfp4":
        return (random_fp4_codes(M, w.K, s + 0), random_fp4_codes(w.N, w.K, s + 1),
                random_e8m0(M, w.K, s + 2), random_e8m0(w.N, w.K, s + 3))
    raise ValueError(w.dtype)


def bits_of(t: torch.Tensor):
    """numpy view of a CPU tensor's raw bits (uint32 for f32, uint16 for bf16)."""
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32).numpy().view("uint32")
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.uint8:
        return t.contiguous().numpy()
    if t.dtype == torch.float8_e4m3fn:
        return t.contiguous().view(torch.uint8).numpy()
    raise TypeError(t.dtype)
