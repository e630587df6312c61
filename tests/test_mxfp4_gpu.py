"""MXFP4 (e2m1 codes, one e8m0 scale per 32 K elements) tensor-core GEMM
against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tiled_mma_atom_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def tmg():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as t
    return t


# Kernel variants: one-CTA 128x128 tiles; CTA pairs with 256x128, 256x192
# and 256x256 tiles (selected through the library's testing variables).
VARIANTS = {"single": {"TMG_MXFP4_KERNEL": "single"},
            "pair128": {"TMG_MXFP4_KERNEL": "pair", "TMG_MXFP4_BN": "128"},
            "pair192": {"TMG_MXFP4_KERNEL": "pair", "TMG_MXFP4_BN": "192"},
            "pair256": {"TMG_MXFP4_KERNEL": "pair", "TMG_MXFP4_BN": "256"}}


@pytest.fixture(params=list(VARIANTS))
def variant(request, monkeypatch):
    for k, v in VARIANTS[request.param].items():
        monkeypatch.setenv(k, v)
    return request.param


def _run(tmg, A, B, sA, sB):
    D = tmg.gemm_mxfp4(*(t.to(DEV) for t in (A, B, sA, sB)))
    tmg.check()
    return D


def _ref(A, B, sA, sB, M, N, K):
    return oracle.gemm_mxfp4(A.numpy(), B.numpy(), sA.numpy(), sB.numpy(), M, N, K)


def _amax(X, S, K):
    return float(np.abs(oracle.read_mxfp4(X.numpy(), S.numpy(), X.shape[0], K)).max())


def test_mxfp4_unit_scales_bit_exact(tmg, variant):
    """Scales 2^0: every product is a multiple of 1/4 and |sum| < 2^15, so the
    fp32 accumulation is exact and D must be RNE_bf16(exact)."""
    M, N, K = 256, 384, 512
    A = inputs.random_fp4_codes(M, K, 1)
    B = inputs.random_fp4_codes(N, K, 2)
    sA = torch.full((M, K // 32), 127, dtype=torch.uint8)
    sB = torch.full((N, K // 32), 127, dtype=torch.uint8)
    D = _run(tmg, A, B, sA, sB)
    parity.check_exact_bf16(parity.bf16_bits(D), _ref(A, B, sA, sB, M, N, K))


def test_mxfp4_per_block_scales_bit_exact(tmg, variant):
    """Scales 2^-1..2^1 varying per row and per 32-element block: products
    are multiples of 2^-4 below 2^8 and sums stay below 2^17, so the result
    is still exact — any misplaced scale (wrong row, block or half-word)
    changes it."""
    M, N, K = 384, 256, 1024
    A = inputs.random_fp4_codes(M, K, 3)
    B = inputs.random_fp4_codes(N, K, 4)
    sA = inputs.random_e8m0(M, K, 5, lo=-1, hi=1)
    sB = inputs.random_e8m0(N, K, 6, lo=-1, hi=1)
    D = _run(tmg, A, B, sA, sB)
    parity.check_exact_bf16(parity.bf16_bits(D), _ref(A, B, sA, sB, M, N, K))


def test_mxfp4_per_block_scales_partial_scale_group(tmg, variant):
    """K = 2560 is ten K blocks of 256: the pair kernel copies raw scales four
    K blocks at a time, so the last copy of each tile holds two.  Per-block
    scales 2^-1..2^1 keep the result exact (as above); ragged M and N put
    rows past the end of both operands into the last tiles."""
    M, N, K = 392, 328, 2560
    A = inputs.random_fp4_codes(M, K, 13)
    B = inputs.random_fp4_codes(N, K, 14)
    sA = inputs.random_e8m0(M, K, 15, lo=-1, hi=1)
    sB = inputs.random_e8m0(N, K, 16, lo=-1, hi=1)
    D = _run(tmg, A, B, sA, sB)
    parity.check_exact_bf16(parity.bf16_bits(D), _ref(A, B, sA, sB, M, N, K))


@pytest.mark.parametrize("M,N,K", [(2048, 2304, 4096), (512, 640, 8192)])
def test_mxfp4_partial_wave_exact(tmg, variant, M, N, K):
    """Problems whose tiles do not fill whole waves of CTA pairs (fewer tiles
    than pairs; a long K at 512 x 640 x 8192).  Unit scales keep every sum
    exact (multiples of 1/4 of magnitude at most 36 K < 2^19), so D must
    equal RNE_bf16 of the exact sum bit for bit, and a second call must give
    the same bits."""
    A = inputs.random_fp4_codes(M, K, 17)
    B = inputs.random_fp4_codes(N, K, 18)
    sA = torch.full((M, K // 32), 127, dtype=torch.uint8)
    sB = torch.full((N, K // 32), 127, dtype=torch.uint8)
    D = _run(tmg, A, B, sA, sB)
    parity.check_exact_bf16(parity.bf16_bits(D), _ref(A, B, sA, sB, M, N, K))
    D2 = _run(tmg, A, B, sA, sB)
    assert torch.equal(D, D2)


def test_mxfp4_one_hot_scale_locates_each_block(tmg, variant):
    """All codes 1.0; one row of A (or of B) gets scale 2^1 on a single K
    block.  Each output of that row (column) must be K + 32, all others K."""
    M, N, K = 256, 320, 512
    one = torch.full((max(M, N), K), 2, dtype=torch.int32)    # code 2 = 1.0
    A = inputs.pack_fp4(one[:M])
    B = inputs.pack_fp4(one[:N])
    for side, idx, blk in [("a", 0, 0), ("a", 37, 5), ("a", 127, 15), ("a", 200, 9), ("a", 255, 3),
                           ("b", 0, 1), ("b", 95, 7), ("b", 130, 12), ("b", 191, 14), ("b", 300, 2)]:
        sA = torch.full((M, K // 32), 127, dtype=torch.uint8)
        sB = torch.full((N, K // 32), 127, dtype=torch.uint8)
        (sA if side == "a" else sB)[idx, blk] = 128
        D = _run(tmg, A, B, sA, sB).float().cpu()
        want = torch.full((M, N), float(K))
        if side == "a":
            want[idx, :] = K + 32
        else:
            want[:, idx] = K + 32
        assert torch.equal(D, want), (side, idx, blk)


@pytest.mark.parametrize("M,N,K", [(300, 200, 1024), (256, 640, 256), (520, 392, 768), (512, 384, 1536)])
def test_mxfp4_random_vs_oracle(tmg, variant, M, N, K):
    A = inputs.random_fp4_codes(M, K, 7)
    B = inputs.random_fp4_codes(N, K, 8)
    sA = inputs.random_e8m0(M, K, 9)
    sB = inputs.random_e8m0(N, K, 10)
    D = _run(tmg, A, B, sA, sB)
    parity.check_bf16(D, _ref(A, B, sA, sB, M, N, K), K, _amax(A, sA, K), _amax(B, sB, K))


def test_mxfp4_workload_8192_sampled(tmg):
    """8192³ MXFP4 (codes U{0..15}, scale exponents U[-4,4]), the benchmark's
    launch (automatic kernel choice): sampled outputs vs the oracle."""
    w = inputs.WORKLOADS["mxfp4_8192"]
    A, B, sA, sB = inputs.make_inputs(w)
    D = _run(tmg, A, B, sA, sB)
    ms, ns = parity.sample_coords(w.M, w.N, 4000, seed=4)
    ref = oracle.gemm_mxfp4_entries(A.numpy(), B.numpy(), sA.numpy(), sB.numpy(), w.K, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, w.K, 6.0 * 16, 6.0 * 16)


def test_mxfp4_rejects_unaligned_k(tmg):
    A = torch.zeros((4, 24), dtype=torch.uint8, device=DEV)       # K = 48
    s = torch.zeros((4, 1), dtype=torch.uint8, device=DEV)
    with pytest.raises(tmg.TmgError) as ei:
        tmg.gemm_mxfp4(A, A, s, s)
    assert ei.value.status == 1


def test_mxfp4_small_m_uses_one_cta_kernel(tmg):
    """M < 256 cannot fill a CTA pair; the automatic choice must still be
    exact (integer-valued case: unit scales)."""
    M, N, K = 100, 200, 256
    A = inputs.random_fp4_codes(M, K, 11)
    B = inputs.random_fp4_codes(N, K, 12)
    sA = torch.full((M, K // 32), 127, dtype=torch.uint8)
    sB = torch.full((N, K // 32), 127, dtype=torch.uint8)
    D = _run(tmg, A, B, sA, sB)
    parity.check_exact_bf16(parity.bf16_bits(D), _ref(A, B, sA, sB, M, N, K))
