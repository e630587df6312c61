"""GPU parity of the host-buffer GEMM (tmg_gemm_host): operands and result in
host memory, transfers pipelined with the GEMM by the library, compared with
the oracle on the same bits."""
import numpy as np
import pytest
import torch

import oracle
from tiled_mma_atom_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tmg():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as t
    yield t
    t.check()


def _sync(tmg):
    torch.cuda.current_stream().synchronize()
    tmg.check()


@pytest.mark.parametrize("M,N,K", [(3000, 1000, 512), (1, 256, 64), (4096, 768, 200)])
def test_host_bf16_vs_oracle(tmg, M, N, K):
    """Several row chunks (ragged last chunk), one chunk, K not a multiple of
    the K block."""
    A, B = inputs.normal_bf16(M, K, 501).pin_memory(), inputs.normal_bf16(N, K, 502).pin_memory()
    D = tmg.gemm_host(A, B)
    _sync(tmg)
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


def test_host_fp32_pageable(tmg):
    """fp32 (the CUDA-core path) from ordinary pageable memory."""
    M, N, K = 300, 200, 100
    A, B = inputs.uniform_f32(M, K, 511), inputs.uniform_f32(N, K, 512)
    D = torch.empty(M, N)
    tmg.gemm_host(A, B, D)
    _sync(tmg)
    parity.check_fp32(D, parity.ref_full(A, B, oracle.F32))


def test_host_integer_exact_back_to_back(tmg):
    """Two calls queued back to back on one stream reuse the workspace: both
    results are the bf16 rounding of the exact products, bit for bit."""
    M, N, K = 4096, 512, 256
    A1, B1 = inputs.integer_valued(M, K, 521).pin_memory(), inputs.integer_valued(N, K, 522).pin_memory()
    A2, B2 = inputs.integer_valued(M, K, 523).pin_memory(), inputs.integer_valued(N, K, 524).pin_memory()
    D1 = tmg.gemm_host(A1, B1)
    D2 = tmg.gemm_host(A2, B2)
    _sync(tmg)
    parity.check_exact_bf16(parity.bf16_bits(D1), parity.ref_full(A1, B1, oracle.BF16))
    parity.check_exact_bf16(parity.bf16_bits(D2), parity.ref_full(A2, B2, oracle.BF16))


def test_host_rejects_device_memory(tmg):
    from tiled_mma_atom_gb300 import _native
    A = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    Dh = torch.empty(8, 8, dtype=torch.bfloat16)
    st = _native.lib().tmg_gemm_host(A.data_ptr(), A.data_ptr(), Dh.data_ptr(), 8, 8, 8, _native.BF16, None)
    assert st == _native.ERR_INVALID_ARG
