"""GPU parity of the W4A8 GEMM (int8 A x packed int4 B -> int32 D): the
result is exact, so it must equal the oracle's integer sums bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from tiled_mma_atom_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def tmg():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as t
    yield t
    t.check()


def _run(tmg, A, B):
    D = tmg.gemm_w4a8(A.to(DEV), B.to(DEV))
    tmg.check()
    return D.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (256, 384, 8448), (2048, 2560, 1024), (1, 40, 34), (17, 130, 4098)])
def test_w4a8_exact(tmg, M, N, K):
    """Ragged tiles, K not a multiple of 8 or of the 4096 segment, several
    segments, the stream-K tail (2048 x 2560), a single row."""
    A, B = inputs.random_int8(M, K, 701), inputs.random_int4_packed(N, K, 702)
    assert np.array_equal(_run(tmg, A, B), oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K))


def test_w4a8_extreme_values_exact(tmg):
    """Every product at its largest magnitude, (-128)(-8) = 1024, over K =
    12288 (three segments, each summing to 2^22): D = 12582912 everywhere;
    and the most negative mix."""
    M, N, K = 256, 256, 12288
    A = torch.full((M, K), -128, dtype=torch.int8)
    B = torch.full((N, K // 2), 0x88, dtype=torch.uint8)          # nibbles 8 -> -8
    D = _run(tmg, A, B)
    assert (D == 1024 * K).all()
    B2 = torch.full((N, K // 2), 0x77, dtype=torch.uint8)         # nibbles 7
    D2 = _run(tmg, A, B2)
    assert (D2 == -128 * 7 * K).all()


def test_w4a8_k0_writes_zeros(tmg):
    A = torch.empty((5, 0), dtype=torch.int8, device=DEV)
    B = torch.empty((7, 0), dtype=torch.uint8, device=DEV)
    D = torch.full((5, 7), 99, dtype=torch.int32, device=DEV)
    tmg.gemm_w4a8(A, B, D)
    tmg.check()
    assert torch.count_nonzero(D) == 0


def test_w4a8_workload_sampled(tmg):
    """The benchmark's W4A8 workload at full size, sampled outputs."""
    w = inputs.WORKLOADS["w4a8_8192"]
    A, B = inputs.make_inputs(w)
    D = tmg.gemm_w4a8(A.to(DEV), B.to(DEV))
    tmg.check()
    rng = np.random.default_rng(11)
    ms = np.concatenate([rng.integers(0, w.M, 3000), [0, w.M - 1]])
    ns = np.concatenate([rng.integers(0, w.N, 3000), [w.N - 1, 0]])
    ref = oracle.gemm_w4a8_entries(A.numpy(), B.numpy(), w.K, ms, ns)
    assert np.array_equal(D.cpu().numpy()[ms, ns].astype(np.int64), ref)
