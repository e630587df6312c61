"""GPU parity of the general-layout tensor-core path (PACKED_TC): bf16
operands in any (Shape, Stride) layout are gathered through crd2idx into
K-major copies, multiplied on tcgen05, and a general D is scattered back
through its layout.  Compared with the oracle, which reads the same buffers
through the same layouts.
"""
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


def _ref(Abuf, la, Bbuf, lb, M, N, K):
    return oracle.gemm(inputs.bits_of(Abuf), oracle.make_layout(*la), inputs.bits_of(Bbuf),
                       oracle.make_layout(*lb), oracle.BF16, M, N, K)


def _perm_rows_nested(X, a):
    """Store the rows of X (R, K) so that row r = r0 + a*r1 sits at buffer row
    r0*(R/a) + r1: the nested row mode (a, R/a):(K*R/a, K)."""
    R, K = X.shape
    b = R // a
    buf = torch.empty_like(X)
    for r in range(R):
        buf[(r % a) * b + r // a] = X[r]
    return buf, ((a, b), K), ((K * b, K), 1)


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (256, 384, 203), (1000, 700, 136)])
def test_mn_major_operands(tmg, M, N, K):
    """A column-major (M,K):(1,M) and B stored (K,N) row-major, i.e.
    (N,K):(1,N): both gathered, ragged tiles, K not a multiple of 8."""
    A, B = inputs.normal_bf16(M, K, 401), inputs.normal_bf16(N, K, 402)
    At, Bt = A.t().contiguous(), B.t().contiguous()
    D = tmg.gemm(At.to(DEV), Bt.to(DEV), M=M, N=N, K=K, layoutA=((M, K), (1, M)),
                 layoutB=((N, K), (1, N)), path="packed_tc")
    tmg.check()
    ref = _ref(At, ((M, K), (1, M)), Bt, ((N, K), (1, N)), M, N, K)
    parity.check_bf16(D, ref, K, parity.absmax(A), parity.absmax(B))


def test_integer_exact_nested_strided_broadcast(tmg):
    """Integer inputs (every order of summation exact): A with a nested row
    mode, B broadcast along n (stride 0) on alternate calls, and a strided K
    mode; bit-exact against RNE of the exact result."""
    M, N, K = 512, 640, 256
    A = inputs.integer_valued(M, K, 411)
    Abuf, sa, da = _perm_rows_nested(A, 4)
    B = inputs.integer_valued(N, K, 412)
    Bwide = torch.zeros(N, 2 * K, dtype=torch.bfloat16)
    Bwide[:, ::2] = B                                     # K stride 2
    D = tmg.gemm(Abuf.to(DEV), Bwide.to(DEV), M=M, N=N, K=K, layoutA=(sa, da), layoutB=((N, K), (2 * K, 2)),
                 path="packed_tc")
    tmg.check()
    ref = _ref(Abuf, (sa, da), Bwide, ((N, K), (2 * K, 2)), M, N, K)
    parity.check_exact_bf16(parity.bf16_bits(D), ref)
    brow = inputs.integer_valued(1, K, 413)
    D2 = tmg.gemm(Abuf.to(DEV), brow.to(DEV), M=M, N=N, K=K, layoutA=(sa, da), layoutB=((N, K), (0, 1)),
                  path="packed_tc")
    tmg.check()
    ref2 = _ref(Abuf, (sa, da), brow, ((N, K), (0, 1)), M, N, K)
    parity.check_exact_bf16(parity.bf16_bits(D2), ref2)


def test_general_output_layout_scatter(tmg):
    """D with a nested column mode (4, N/4):(N/4, 1)... permuted columns: the
    result is computed densely and scattered through D's layout; padding
    around it stays untouched."""
    M, N, K = 384, 512, 128
    A, B = inputs.integer_valued(M, K, 421), inputs.integer_valued(N, K, 422)
    ref = _ref(A, ((M, K), (K, 1)), B, ((N, K), (K, 1)), M, N, K)
    ld = N + 8
    Dbuf = torch.full((M, ld), float("nan"), dtype=torch.bfloat16, device=DEV)
    b = N // 4
    # column n = n0 + 4 n1 stored at n0 * b + n1 within the padded row
    tmg.gemm(A.to(DEV), B.to(DEV), Dbuf, M=M, N=N, K=K, layoutD=((M, (4, b)), (ld, (b, 1))), path="packed_tc")
    tmg.check()
    got = parity.bf16_bits(Dbuf)
    n = np.arange(N)
    cols = (n % 4) * b + n // 4
    parity.check_exact_bf16(got[:, cols], ref)
    assert torch.isnan(Dbuf[:, N:].float()).all(), "padding of D was written"


def test_auto_takes_packed_path_for_large_general_layouts(tmg):
    """AUTO sends a large MN-major bf16 problem to the packed tensor-core
    path (kernel launches: pack A, GEMM) and a small one to FFMA (one)."""
    M = N = K = 1024
    A, B = inputs.normal_bf16(M, K, 431), inputs.normal_bf16(N, K, 432)
    At = A.t().contiguous().to(DEV)
    dB = B.to(DEV)
    n0 = tmg.launch_count()
    D = tmg.gemm(At, dB, M=M, N=N, K=K, layoutA=((M, K), (1, M)))
    tmg.check()
    assert tmg.launch_count() - n0 == 2
    ms, ns = parity.sample_coords(M, N, 4000, seed=3)
    ref = oracle.gemm_entries(inputs.bits_of(A.t().contiguous()), oracle.make_layout((M, K), (1, M)),
                              inputs.bits_of(B), oracle.row_major(N, K), oracle.BF16, K, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, K, parity.absmax(A), parity.absmax(B))
    n0 = tmg.launch_count()
    tmg.gemm(At[:64, :64].contiguous(), dB[:64, :64].contiguous(), M=64, N=64, K=64, layoutA=((64, 64), (1, 64)))
    tmg.check()
    assert tmg.launch_count() - n0 == 1


def test_mn_major_workload_size_sampled(tmg):
    """The general-layout workload of the benchmark (bf16 4096³, A
    column-major) at full size, sampled against the oracle."""
    w = inputs.WORKLOADS["bf16_4096_a_mn_major"]
    A, B = inputs.make_inputs(w)
    D = tmg.gemm(A.to(DEV), B.to(DEV), M=w.M, N=w.N, K=w.K, layoutA=((w.M, w.K), (1, w.M)))
    tmg.check()
    ms, ns = parity.sample_coords(w.M, w.N, 3000, seed=5)
    ref = oracle.gemm_entries(inputs.bits_of(A), oracle.make_layout((w.M, w.K), (1, w.M)), inputs.bits_of(B),
                              oracle.row_major(w.N, w.K), oracle.BF16, w.K, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, w.K, parity.absmax(A), parity.absmax(B))


@pytest.mark.parametrize("maj", [1, 2, 3])
@pytest.mark.parametrize("M,N,K", [(2048, 2560, 320), (2000, 2600, 136)])
def test_mn_major_read_in_place(tmg, monkeypatch, maj, M, N, K):
    """Large enough for CTA pairs: MN-major A (bit 0) and/or B (bit 1) are
    read in place by the pair kernel (64 x 64 boxes, MN-major MMA
    descriptors) instead of being gathered; ragged M, N and K.  The result
    meets the oracle bound and equals the gathered path's bit for bit (the
    same MMAs in the same order: the tile width and schedule are pinned, as
    the two paths choose among different widths when B is MN-major)."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", "256")
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", "sk")
    A, B = inputs.normal_bf16(M, K, 411), inputs.normal_bf16(N, K, 412)
    la = ((M, K), (1, M)) if maj & 1 else ((M, K), (K, 1))
    lb = ((N, K), (1, N)) if maj & 2 else ((N, K), (K, 1))
    Ab = A.t().contiguous() if maj & 1 else A
    Bb = B.t().contiguous() if maj & 2 else B
    Ad, Bd = Ab.to(DEV), Bb.to(DEV)
    n0 = tmg.launch_count()
    D = tmg.gemm(Ad, Bd, M=M, N=N, K=K, layoutA=la, layoutB=lb)
    tmg.check()
    assert tmg.launch_count() - n0 == 1                  # the pair kernel alone: no gather
    ref = _ref(Ab, la, Bb, lb, M, N, K)
    parity.check_bf16(D, ref, K, parity.absmax(A), parity.absmax(B))
    monkeypatch.setenv("TMG_NO_INPLACE_MN", "1")
    n0 = tmg.launch_count()
    D2 = tmg.gemm(Ad, Bd, M=M, N=N, K=K, layoutA=la, layoutB=lb)
    tmg.check()
    assert tmg.launch_count() - n0 >= 2                  # gathered, then the GEMM
    assert torch.equal(D, D2)


@pytest.mark.parametrize("width", [128, 192, 224, 256])
def test_mn_major_a_in_place_every_width(tmg, monkeypatch, width):
    """A column-major read in place at every pair-tile width (its boxes do
    not depend on the width), data-parallel with a partial last wave:
    equal to the gathered path at the same width and schedule."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", str(width))
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", "dp")
    M, N, K = 2048, 2600, 200
    A, B = inputs.normal_bf16(M, K, 431), inputs.normal_bf16(N, K, 432)
    la = ((M, K), (1, M))
    Ad, Bd = A.t().contiguous().to(DEV), B.to(DEV)
    n0 = tmg.launch_count()
    D = tmg.gemm(Ad, Bd, M=M, N=N, K=K, layoutA=la)
    tmg.check()
    assert tmg.launch_count() - n0 == 1
    parity.check_bf16(D, _ref(A.t().contiguous(), la, B, ((N, K), (K, 1)), M, N, K), K, parity.absmax(A),
                      parity.absmax(B))
    monkeypatch.setenv("TMG_NO_INPLACE_MN", "1")
    D2 = tmg.gemm(Ad, Bd, M=M, N=N, K=K, layoutA=la)
    tmg.check()
    assert torch.equal(D, D2)


def test_b_kn_workload_size_sampled(tmg):
    """The benchmark's C = A·B workload (bf16 4096³, B stored K×N row-major,
    i.e. MN-major) at full size, sampled against the oracle."""
    w = inputs.WORKLOADS["bf16_4096_b_kn"]
    A, B = inputs.make_inputs(w)
    n0 = tmg.launch_count()
    D = tmg.gemm(A.to(DEV), B.to(DEV), M=w.M, N=w.N, K=w.K, layoutB=((w.N, w.K), (1, w.N)))
    tmg.check()
    assert tmg.launch_count() - n0 == 1
    ms, ns = parity.sample_coords(w.M, w.N, 3000, seed=6)
    ref = oracle.gemm_entries(inputs.bits_of(A), oracle.row_major(w.M, w.K), inputs.bits_of(B),
                              oracle.make_layout((w.N, w.K), (1, w.N)), oracle.BF16, w.K, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, w.K, parity.absmax(A), parity.absmax(B))


def test_mn_major_in_place_padded_leading_dimension(tmg):
    """Column-major A inside a wider buffer (lda = M + 8) and B (K,N)
    row-major inside one with ldb = N + 24: still read in place."""
    M, N, K = 2048, 2560, 192
    A, B = inputs.normal_bf16(M, K, 421), inputs.normal_bf16(N, K, 422)
    Abuf = torch.zeros(K, M + 8, dtype=torch.bfloat16)
    Abuf[:, :M] = A.t()
    Bbuf = torch.zeros(K, N + 24, dtype=torch.bfloat16)
    Bbuf[:, :N] = B.t()
    la, lb = ((M, K), (1, M + 8)), ((N, K), (1, N + 24))
    n0 = tmg.launch_count()
    D = tmg.gemm(Abuf.to(DEV), Bbuf.to(DEV), M=M, N=N, K=K, layoutA=la, layoutB=lb)
    tmg.check()
    assert tmg.launch_count() - n0 == 1
    parity.check_bf16(D, _ref(Abuf, la, Bbuf, lb, M, N, K), K, parity.absmax(A), parity.absmax(B))
