"""Maximum-size edge cases: single operands of 2^31 elements (4 GB of bf16),
past the range of 32-bit element offsets, on the skinny and the CTA-pair
tensor-core paths.  Integer-valued inputs keep every partial sum exact, so
the sampled outputs must equal the bf16 rounding of the exact values bit for
bit.  The large operand is built on the GPU from a hash of (row, column) and
the oracle regenerates, on the CPU, only the rows it samples."""
import numpy as np
import pytest
import torch

import oracle
from tiled_mma_atom_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def tmg():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as t
    yield t
    t.check()


def _rows(idx, cols, seed):
    """Rows idx of the hashed matrix, regenerated on the CPU."""
    return torch.cat([inputs.hashed_int(1, cols, seed, row0=int(i)) for i in idx])


def test_skinny_b_with_2_pow_31_elements(tmg):
    M, N, K = 16, 131072, 16384                  # B: 2^31 elements
    B = inputs.hashed_int_device(N, K, 601, DEV)
    A = inputs.hashed_int(M, K, 602)
    D = tmg.gemm(A.to(DEV), B)
    tmg.check()
    rng = np.random.default_rng(7)
    ns = np.concatenate([rng.integers(0, N, 600), [0, N - 1, N - 2]])
    ms = rng.integers(0, M, ns.size)
    Bs = _rows(ns, K, 601)
    ref = oracle.gemm_entries(inputs.bits_of(A), oracle.row_major(M, K), inputs.bits_of(Bs),
                              oracle.row_major(ns.size, K), oracle.BF16, K, ms, np.arange(ns.size))
    got = parity.bf16_bits(D)[ms, ns]
    assert np.array_equal(got, oracle.round_bf16_array(ref))
    del B, D
    torch.cuda.empty_cache()


def test_pair_a_with_2_pow_31_elements(tmg):
    M, N, K = 65536, 512, 32768                  # A: 2^31 elements
    A = inputs.hashed_int_device(M, K, 611, DEV)
    B = inputs.hashed_int(N, K, 612)
    D = tmg.gemm(A, B.to(DEV), path="tc_pair")
    tmg.check()
    rng = np.random.default_rng(8)
    ms = np.concatenate([rng.integers(0, M, 600), [0, M - 1, M - 129]])
    ns = rng.integers(0, N, ms.size)
    As = _rows(ms, K, 611)
    ref = oracle.gemm_entries(inputs.bits_of(As), oracle.row_major(ms.size, K), inputs.bits_of(B),
                              oracle.row_major(N, K), oracle.BF16, K, np.arange(ms.size), ns)
    got = parity.bf16_bits(D)[ms, ns]
    assert np.array_equal(got, oracle.round_bf16_array(ref))
    del A, D
    torch.cuda.empty_cache()
