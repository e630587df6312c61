"""The skinny entry point that allocates nothing, checked against the
ordinary (allocating) skinny entry point through the C ABI.

Some callers cannot allocate device memory when they call the GEMM — a
latency-critical loop that must not call cudaMalloc/cudaFree after start-up
(both can synchronise the device), or a plug-in whose host owns all device
memory and hands over only the operands.  tmg_gemm_skinny_noalloc serves
them from a fixed array in the library's static device memory.

This file is named to be collected last, so that a failure here cannot stop
a run before every other test has run.  It builds and loads the library on
its own, so it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from tests import parity
from tiled_mma_atom_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def native():
    import __graft_entry__
    __graft_entry__.build()
    from tiled_mma_atom_gb300 import _native
    return _native


def _existing(native, A, B, D, M, N, K, stream):
    L = native.lib()
    la = native.make_layout((M, K), (A.stride(0), 1))
    lb = native.make_layout((N, K), (B.stride(0), 1))
    ld = native.make_layout((M, N), (D.stride(0), 1))
    native.raise_on(L.tmg_gemm_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, native.BF16,
                                  la, lb, ld, native.PATHS["skinny"], stream))


def _noalloc(native, A, B, D, M, N, K, stream):
    L = native.lib()
    native.raise_on(L.tmg_gemm_skinny_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                              A.stride(0), B.stride(0), D.stride(0), stream))


def test_noalloc_matches_allocating_entry_point(native):
    torch.cuda.set_device(DEV)
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(16, 28672, 8192, 1), (40, 3000, 1000, 2), (5, 1000, 512, 3)]
    for M, N, K, seed in cases:
        A = inputs.normal_bf16(M, K, 500 + seed)
        B = inputs.normal_bf16(N, K, 600 + seed, std=0.02)
        dA, dB = A.to(DEV), B.to(DEV)
        ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        _existing(native, dA, dB, ref, M, N, K, stream)
        amax, bmax = parity.absmax(A), parity.absmax(B)
        # two calls in a row: the second sees whatever the first left in the
        # shared array
        for _ in range(2):
            D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
            _noalloc(native, dA, dB, D, M, N, K, stream)
            native.raise_on(native.lib().tmg_check(stream))
            parity.check_bf16_values(parity.to_f64(D), parity.to_f64(ref), K, amax, bmax)


def test_noalloc_rejects_sizes_beyond_its_scratch(native):
    L = native.lib()
    dummy = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    p = dummy.data_ptr()
    assert L.tmg_gemm_skinny_noalloc(p, p, p, 65, 8, 8, 8, 8, 8, None) == native.ERR_INVALID_ARG
    assert "64" in L.tmg_last_error().decode()
    assert L.tmg_gemm_skinny_noalloc(p, p, p, 16, 524288 + 128, 8, 8, 8, 524288 + 128,
                                     None) == native.ERR_INVALID_ARG
    assert "524288" in L.tmg_last_error().decode()
