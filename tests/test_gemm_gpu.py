"""GPU parity tests: every kernel family against the CPU oracle, through the
C ABI (tiled_mma_atom_gb300 is ctypes marshalling over libtmg.so).

Small cases are compared element by element with the full oracle result;
the full-size workloads are compared on sampled outputs that the oracle
computes one by one, in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_mma_atom_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as tmg
    yield tmg
    tmg.check()


@pytest.fixture
def tmg(built):
    return built


def _gpu(*ts):
    return [t.to(DEV) for t in ts]


# ------------------------------------------------------------- FFMA / fp32

def test_ffma_fp32_workload_128(tmg):
    """fp32 128³, U[-1,1] (the fp32 workload), full oracle comparison."""
    w = inputs.WORKLOADS["fp32_128"]
    A, B = inputs.make_inputs(w)
    dA, dB = _gpu(A, B)
    D = tmg.gemm(dA, dB)
    tmg.check()
    parity.check_fp32(D, parity.ref_full(A, B, oracle.F32))


def test_ffma_fp32_ragged_and_general_layouts(tmg):
    """Ragged sizes and non-row-major layouts: A column-major, B stored
    (K, N) row-major, D column-major with padding, and a nested K mode."""
    M, N, K = 37, 53, 72
    A = inputs.uniform_f32(M, K, 11)
    B = inputs.uniform_f32(N, K, 12)
    ref = parity.ref_full(A, B, oracle.F32)
    # A column-major: buffer holds Aᵀ contiguous
    At = A.t().contiguous()
    Bkn = B.t().contiguous()                                  # (K, N) row-major
    Dbuf = torch.full((N, M + 3), float("nan"), device=DEV)   # D col-major, ld = M + 3
    tmg.gemm(At.to(DEV), Bkn.to(DEV), Dbuf, M=M, N=N, K=K,
             layoutA=((M, K), (1, M)), layoutB=((N, K), (1, N)), layoutD=((M, N), (1, M + 3)))
    tmg.check()
    D = Dbuf[:, :M].t()
    parity.check_fp32(D, ref)
    assert torch.isnan(Dbuf[:, M:]).all(), "padding of D was written"
    # nested K mode: k = k0 + 8 k1 stored at k0 * 9 + k1 inside each row
    Anest = torch.empty(M, K)
    for k in range(K):
        Anest[:, (k % 8) * 9 + k // 8] = A[:, k]
    D2 = tmg.gemm(Anest.to(DEV), B.to(DEV), M=M, N=N, K=K,
                  layoutA=((M, (8, 9)), (K, (9, 1))), layoutB=((N, K), (K, 1)))
    tmg.check()
    parity.check_fp32(D2, ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 700, 264), (1000, 900, 200), (70, 33, 136)])
def test_ffma_dense_and_general_kernels_agree(tmg, dtype, M, N, K):
    """Row-major operands with 16-byte rows take the dense CUDA-core kernel;
    the same values read through a padded row stride (K + 1, not a multiple
    of the vector), or from a pointer 4 bytes past a 16-byte boundary, take
    the general crd2idx kernel.  Both use the same tiles
    and k order, so they agree bit for bit; both match the oracle.  The
    shapes cover the three tile configurations (16x16 with 128-deep K
    slices, 32x32, 64x64) and ragged edges."""
    if dtype == "f32":
        A, B = inputs.uniform_f32(M, K, 41), inputs.uniform_f32(N, K, 42)
    else:
        A, B = inputs.normal_bf16(M, K, 43), inputs.normal_bf16(N, K, 44)
    Apad = torch.zeros(M, K + 1, dtype=A.dtype)
    Apad[:, :K] = A
    dA, dB, dApad = _gpu(A, B, Apad)
    D1 = tmg.gemm(dA, dB, path="ffma").clone()
    D2 = tmg.gemm(dApad, dB, M=M, N=N, K=K, layoutA=((M, K), (K + 1, 1)), path="ffma")
    tmg.check()
    assert torch.equal(D1, D2)
    # the same row-major values four bytes past a 16-byte boundary: general kernel
    flat = torch.zeros(M * K + 8, dtype=A.dtype, device=DEV)
    Aoff = flat[4 // A.element_size():][:M * K].view(M, K)
    Aoff.copy_(dA)
    D3 = tmg.gemm(Aoff, dB, path="ffma")
    tmg.check()
    assert torch.equal(D1, D3)
    if dtype == "f32":
        parity.check_fp32(D1, parity.ref_full(A, B, oracle.F32))
    else:
        parity.check_bf16(D1, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


def test_ffma_broadcast_operand(tmg):
    """A zero stride broadcasts one row of B to every n."""
    M, N, K = 20, 30, 40
    A = inputs.uniform_f32(M, K, 21)
    brow = inputs.uniform_f32(1, K, 22)
    D = tmg.gemm(A.to(DEV), brow.to(DEV), M=M, N=N, K=K, layoutB=((N, K), (0, 1)))
    tmg.check()
    ref = parity.ref_full(A, brow.expand(N, K).contiguous(), oracle.F32)
    parity.check_fp32(D, ref)


def test_ffma_bf16_general_layout(tmg):
    """bf16 with an MN-major A goes to the CUDA-core path (crd2idx loads)."""
    M, N, K = 70, 90, 100
    A = inputs.normal_bf16(M, K, 31)
    B = inputs.normal_bf16(N, K, 32)
    At = A.t().contiguous()
    D = tmg.gemm(At.to(DEV), B.to(DEV), M=M, N=N, K=K, layoutA=((M, K), (1, M)))
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


def test_zero_k_writes_zeros(tmg):
    D = torch.full((5, 7), float("nan"), device=DEV)
    A = torch.empty((5, 0), device=DEV)
    B = torch.empty((7, 0), device=DEV)
    tmg.gemm(A, B, D)
    tmg.check()
    assert (D == 0).all()


# --------------------------------------------------------- tcgen05 bf16

@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (200, 300, 136), (129, 257, 72),
                                   (1000, 1000, 1000), (64, 512, 4096)])
def test_tc_random_vs_oracle(tmg, M, N, K):
    A = inputs.normal_bf16(M, K, M + 1)
    B = inputs.normal_bf16(N, K, N + 2)
    D = tmg.gemm(*_gpu(A, B), path="tc")
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


def test_tc_identity_b_is_exact(tmg):
    """B = I: every output equals the matching A element exactly."""
    M, K = 256, 512
    A = inputs.normal_bf16(M, K, 41)
    I = torch.eye(K, dtype=torch.bfloat16)
    D = tmg.gemm(*_gpu(A, I), path="tc")
    tmg.check()
    assert torch.equal(D.cpu(), A)


def test_tc_permutation_b_is_exact(tmg):
    M, K = 384, 256
    A = inputs.normal_bf16(M, K, 42)
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(7))
    P = torch.zeros(K, K, dtype=torch.bfloat16)
    P[torch.arange(K), perm] = 1
    D = tmg.gemm(*_gpu(A, P), path="tc")
    tmg.check()
    assert torch.equal(D.cpu(), A[:, perm])


def test_tc_all_ones_is_k(tmg):
    M, N, K = 256, 384, 4096
    D = tmg.gemm(torch.ones(M, K, dtype=torch.bfloat16, device=DEV),
                 torch.ones(N, K, dtype=torch.bfloat16, device=DEV), path="tc")
    tmg.check()
    assert (D == K).all()


@pytest.mark.parametrize("M,N,K", [(512, 512, 1024), (300, 700, 264)])
def test_tc_integer_inputs_bit_exact(tmg, M, N, K):
    A = inputs.integer_valued(M, K, 51)
    B = inputs.integer_valued(N, K, 52)
    D = tmg.gemm(*_gpu(A, B), path="tc")
    tmg.check()
    parity.check_exact_bf16(parity.bf16_bits(D), parity.ref_full(A, B, oracle.BF16))


def test_tc_column_major_d_swaps_operands(tmg):
    """D column-major is computed as Dᵀ = B·Aᵀ on the tensor cores."""
    M, N, K = 300, 200, 128
    A = inputs.normal_bf16(M, K, 61)
    B = inputs.normal_bf16(N, K, 62)
    Dt = torch.empty((N, M), dtype=torch.bfloat16, device=DEV)
    tmg.gemm(*_gpu(A, B), Dt, M=M, N=N, K=K, layoutD=((M, N), (1, M)), path="tc")
    tmg.check()
    parity.check_bf16(Dt.t(), parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


@pytest.mark.parametrize("path", ["tc_single", "tc_pair"])
def test_tc_wide_tiles_sampled(tmg, path):
    """Many tiles: the one-CTA kernel takes 128x256 tiles, the pair kernel
    its widest tiles."""
    M, N, K = 4096, 2560, 512
    A = inputs.normal_bf16(M, K, 71)
    B = inputs.normal_bf16(N, K, 72)
    D = tmg.gemm(*_gpu(A, B), path=path)
    tmg.check()
    ms, ns = parity.sample_coords(M, N, 20000, seed=1)
    ref = parity.ref_entries(A, B, oracle.BF16, ms, ns)
    d = parity.to_f64(D)[ms, ns]
    parity.check_bf16_values(d, ref, K, parity.absmax(A), parity.absmax(B))
    # integer inputs at the same shape: sampled outputs exact
    Ai = inputs.integer_valued(M, K, 73)
    Bi = inputs.integer_valued(N, K, 74)
    Di = tmg.gemm(*_gpu(Ai, Bi), path=path)
    tmg.check()
    refi = parity.ref_entries(Ai, Bi, oracle.BF16, ms, ns)
    parity.check_exact_bf16(parity.bf16_bits(Di)[ms, ns], refi)


# Shapes for which the pair kernel picks each tile width on 152 SMs
# (76 pairs): (M, N) -> width.
PAIR_SHAPES = [((512, 512), 128), ((2048, 1536), 192), ((2048, 1792), 224), ((2048, 2048), 256)]


@pytest.mark.parametrize("shape,width", PAIR_SHAPES)
def test_tc_pair_each_tile_width_vs_oracle(tmg, shape, width):
    M, N = shape
    K = 256
    A = inputs.normal_bf16(M, K, 130 + width)
    B = inputs.normal_bf16(N, K, 131 + width)
    D = tmg.gemm(*_gpu(A, B), path="tc_pair")
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


@pytest.mark.parametrize("sched", ["sk", "dp"])
@pytest.mark.parametrize("width", [128, 192, 224, 256])
def test_tc_pair_stream_k_tail_exact(tmg, width, sched, monkeypatch):
    """2048 x 2560 leaves a partial last wave for every pair tile width: with
    a stream-K tail the last tiles are summed from fp32 partials, data-parallel
    the last wave leaves pairs idle.  Integer inputs: bit-exact; twice in a row
    (the tile counters reset themselves)."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", str(width))
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", sched)
    M, N, K = 2048, 2560, 1024
    A = inputs.integer_valued(M, K, 200 + width)
    B = inputs.integer_valued(N, K, 201 + width)
    dA, dB = _gpu(A, B)
    D1 = tmg.gemm(dA, dB, path="tc_pair").clone()
    D2 = tmg.gemm(dA, dB, path="tc_pair")
    tmg.check()
    assert torch.equal(D1, D2)
    parity.check_exact_bf16(parity.bf16_bits(D2), parity.ref_full(A, B, oracle.BF16))


@pytest.mark.parametrize("width", [128, 224, 256])
def test_tc_pair_fewer_tiles_than_pairs_exact(tmg, width, monkeypatch):
    """Data-parallel with fewer tiles than CTA pairs (1024 x 2048: 32 tiles
    at width 256, 36 at 224, 64 at 128, on 76 pairs): only that many pairs
    are launched.  Ragged N and K; integer inputs, bit-exact."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", str(width))
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", "dp")
    M, N, K = 1024, 2000, 520
    A = inputs.integer_valued(M, K, 220 + width)
    B = inputs.integer_valued(N, K, 221 + width)
    D = tmg.gemm(*_gpu(A, B), path="tc_pair")
    tmg.check()
    parity.check_exact_bf16(parity.bf16_bits(D), parity.ref_full(A, B, oracle.BF16))


def test_tc_pair_stream_k_random_vs_oracle(tmg, monkeypatch):
    """Random inputs through the stream-K tail (4096 x 4096 has 256 tiles of
    256 columns over 76 pairs); sampled outputs in the split tiles' region."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", "256")
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", "sk")
    M, N, K = 4096, 4096, 512
    A = inputs.normal_bf16(M, K, 211)
    B = inputs.normal_bf16(N, K, 212)
    D = tmg.gemm(*_gpu(A, B), path="tc_pair")
    tmg.check()
    ms, ns = parity.sample_coords(M, N, 30000, seed=9)
    ref = parity.ref_entries(A, B, oracle.BF16, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, K, parity.absmax(A), parity.absmax(B))


@pytest.mark.parametrize("M,N,K", [(300, 333, 200), (640, 1000, 520), (256, 16, 64)])
def test_tc_pair_ragged_integer_exact(tmg, M, N, K):
    """Ragged pair tiles (row half of the second CTA partly or wholly out of
    range, ragged N and K) with integer inputs: bit-exact."""
    A = inputs.integer_valued(M, K, 140 + M)
    B = inputs.integer_valued(N, K, 141 + N)
    D = tmg.gemm(*_gpu(A, B), path="tc_pair")
    tmg.check()
    parity.check_exact_bf16(parity.bf16_bits(D), parity.ref_full(A, B, oracle.BF16))


@pytest.mark.parametrize("M,N,K", [(4648, 600, 256), (2856, 300, 4160)])
def test_tc_pair_ragged_tile_groups_exact(tmg, M, N, K):
    """The pair kernel's tile order runs groups of 16 M-tiles at K = 256
    (19 M-tiles: one group of 16 and a ragged group of 3) and groups of 8
    at K = 4160 (12 M-tiles: 8 and a ragged 4).  Integer inputs: bit-exact."""
    A = inputs.integer_valued(M, K, 160 + M)
    B = inputs.integer_valued(N, K, 161 + N)
    D = tmg.gemm(*_gpu(A, B), path="tc_pair")
    tmg.check()
    parity.check_exact_bf16(parity.bf16_bits(D), parity.ref_full(A, B, oracle.BF16))


def test_tc_single_and_pair_agree(tmg):
    """One-CTA and CTA-pair kernels on the same inputs: integer inputs make
    both exact, so they must agree bit for bit."""
    M, N, K = 768, 896, 384
    A = inputs.integer_valued(M, K, 150)
    B = inputs.integer_valued(N, K, 151)
    dA, dB = _gpu(A, B)
    D1 = tmg.gemm(dA, dB, path="tc_single").clone()
    D2 = tmg.gemm(dA, dB, path="tc_pair")
    tmg.check()
    assert torch.equal(D1, D2)


def test_auto_dispatch_random_shapes(tmg):
    """Shapes drawn at random (seeded) through the auto dispatch, which picks
    one-CTA or pair kernels, tile widths and schedules from its cost model:
    every choice it makes on them must give the oracle's values (sampled
    entries, including the corners and the last row and column)."""
    rng = np.random.default_rng(2024)
    for i in range(16):
        M = int(rng.integers(65, 3200))
        N = int(rng.integers(16, 5200))
        K = 8 * int(rng.integers(1, 320))
        A = inputs.normal_bf16(M, K, 600 + 2 * i)
        B = inputs.normal_bf16(N, K, 601 + 2 * i)
        D = tmg.gemm(*_gpu(A, B))
        tmg.check()
        ms, ns = parity.sample_coords(M, N, 600, seed=i)
        ref = parity.ref_entries(A, B, oracle.BF16, ms, ns)
        parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, K, parity.absmax(A), parity.absmax(B))


def test_tc_deterministic(tmg):
    A = inputs.normal_bf16(512, 768, 81)
    B = inputs.normal_bf16(640, 768, 82)
    dA, dB = _gpu(A, B)
    D1 = tmg.gemm(dA, dB, path="tc").clone()
    D2 = tmg.gemm(dA, dB, path="tc")
    tmg.check()
    assert torch.equal(D1, D2)


def test_workload_bf16_1024_full(tmg):
    """bf16 1024³ N(0,1): full oracle comparison, auto path (tcgen05)."""
    w = inputs.WORKLOADS["bf16_1024"]
    A, B = inputs.make_inputs(w)
    D = tmg.gemm(*_gpu(A, B))
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), w.K, parity.absmax(A), parity.absmax(B))


def test_workload_bf16_4096_sampled(tmg):
    """bf16 4096³ N(0,1), the benchmark's launch: sampled outputs vs oracle."""
    w = inputs.WORKLOADS["bf16_4096"]
    A, B = inputs.make_inputs(w)
    D = tmg.gemm(*_gpu(A, B))
    tmg.check()
    ms, ns = parity.sample_coords(w.M, w.N, 6000, seed=2)
    ref = parity.ref_entries(A, B, oracle.BF16, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, w.K, parity.absmax(A), parity.absmax(B))


# ------------------------------------------------------------- skinny

@pytest.mark.parametrize("M", [1, 7, 16, 17, 40, 64])
def test_skinny_tc_vs_oracle(tmg, M):
    N, K = 1000, 1000
    A = inputs.normal_bf16(M, K, 90 + M)
    B = inputs.normal_bf16(N, K, 91, std=0.02)
    D = tmg.gemm(*_gpu(A, B), path="skinny")
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


def test_skinny_tc_integer_exact_and_repeatable(tmg):
    """Split-K partial sums of integers are exact; two calls in a row agree
    bit for bit (the per-tile counters reset themselves)."""
    M, N, K = 16, 4096, 8192
    A = inputs.integer_valued(M, K, 101)
    B = inputs.integer_valued(N, K, 102)
    dA, dB = _gpu(A, B)
    D1 = tmg.gemm(dA, dB, path="skinny").clone()
    D2 = tmg.gemm(dA, dB, path="skinny")
    tmg.check()
    assert torch.equal(D1, D2)
    ref = parity.ref_full(A, B, oracle.BF16)
    parity.check_exact_bf16(parity.bf16_bits(D2), ref)


@pytest.mark.parametrize("N", [19456, 25600, 38952])
def test_skinny_tc_whole_and_split_tiles_exact(tmg, N):
    """The skinny kernel's schedule: tiles // G whole tiles per CTA and the
    remaining tiles shared out as stream-K runs.  On 152 SMs: 152 tiles (all
    whole, nothing split), 200 tiles (one whole tile each, 48 split), and
    305 tiles with a ragged last one (two whole tiles each, one tile split
    over more CTAs than it has K blocks, so most CTAs have no stream-K
    units).  Integer inputs: bit-exact, twice in a row."""
    M, K = 16, 1024
    A = inputs.integer_valued(M, K, 111)
    B = inputs.integer_valued(N, K, 112 + N)
    dA, dB = _gpu(A, B)
    D1 = tmg.gemm(dA, dB, path="skinny").clone()
    D2 = tmg.gemm(dA, dB, path="skinny")
    tmg.check()
    assert torch.equal(D1, D2)
    parity.check_exact_bf16(parity.bf16_bits(D2), parity.ref_full(A, B, oracle.BF16))


def test_workload_skinny_sampled(tmg):
    """16x28672x8192 decode GEMM, the benchmark's launch (auto -> skinny)."""
    w = inputs.WORKLOADS["skinny_16x28672x8192"]
    A, B = inputs.make_inputs(w)
    dA, dB = _gpu(A, B)
    D = tmg.gemm(dA, dB)
    tmg.check()
    rng = np.random.default_rng(3)
    ns = np.concatenate([rng.integers(0, w.N, 3000), [0, w.N - 1]])
    ms = np.repeat(np.arange(w.M), ns.size)
    ns = np.tile(ns, w.M)
    ref = parity.ref_entries(A, B, oracle.BF16, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, w.K, parity.absmax(A), parity.absmax(B))
    # the CUDA-core split-K variant on the same launch shape
    D2 = tmg.gemm(dA, dB, path="skinny_ffma")
    tmg.check()
    parity.check_bf16_values(parity.to_f64(D2)[ms, ns], ref, w.K, parity.absmax(A), parity.absmax(B))


@pytest.mark.parametrize("M", [1, 5, 16])
def test_skinny_ffma_vs_oracle(tmg, M):
    N, K = 999, 1032
    A = inputs.normal_bf16(M, K, 110 + M)
    B = inputs.normal_bf16(N, K, 111, std=0.02)
    D = tmg.gemm(*_gpu(A, B), path="skinny_ffma")
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


# ------------------------------------------------------ failure handling

def test_bounded_wait_reports_timeout_and_gpu_stays_usable(tmg):
    tmg.debug_wait_timeout(2_000_000)         # 2 ms budget, nothing ever arrives
    with pytest.raises(tmg.TmgError) as ei:
        tmg.check()
    assert ei.value.status == 4
    tmg.check()                               # the error word was cleared
    A = inputs.normal_bf16(128, 64, 5)
    D = tmg.gemm(*_gpu(A, A), path="tc")
    tmg.check()
    parity.check_bf16(D, parity.ref_full(A, A, oracle.BF16), 64, parity.absmax(A), parity.absmax(A))


def test_forced_path_rejects_what_it_cannot_take(tmg):
    A = torch.ones(8, 16, device=DEV)
    with pytest.raises(tmg.TmgError) as ei:
        tmg.gemm(A, A, path="tc")             # fp32 has no tensor-core path
    assert ei.value.status == 2


def test_launch_count_increments(tmg):
    before = tmg.launch_count()
    A = inputs.normal_bf16(128, 64, 6)
    tmg.gemm(*_gpu(A, A))
    tmg.check()
    assert tmg.launch_count() == before + 1


# ------------------------------------------------------------ edge cases

def test_tc_padded_leading_dimensions(tmg):
    """A, B with padded rows (ld = K + 8) and D with an odd row stride (no
    16-byte stores possible: the scalar store path)."""
    M, N, K, ldd = 200, 100, 136, 101
    A = inputs.normal_bf16(M, K + 8, 161)
    B = inputs.normal_bf16(N, K + 8, 162)
    Dbuf = torch.full((M, ldd), float("nan"), dtype=torch.bfloat16, device=DEV)
    tmg.gemm(*_gpu(A, B), Dbuf, M=M, N=N, K=K, layoutA=((M, K), (K + 8, 1)), layoutB=((N, K), (K + 8, 1)),
             layoutD=((M, N), (ldd, 1)), path="tc")
    tmg.check()
    ref = parity.ref_full(A[:, :K].contiguous(), B[:, :K].contiguous(), oracle.BF16)
    parity.check_bf16(Dbuf[:, :N], ref, K, parity.absmax(A), parity.absmax(B))
    assert torch.isnan(Dbuf[:, N:].float()).all(), "padding of D was written"


@pytest.mark.parametrize("M,N,K", [(300, 1, 64), (1, 300, 64), (1, 1, 8), (257, 3, 8), (5, 7, 0)])
def test_degenerate_shapes_auto_path(tmg, M, N, K):
    """One-row / one-column outputs, the smallest K, and K = 0, on the
    automatic path (bf16)."""
    A = inputs.integer_valued(M, K, 170 + M)
    B = inputs.integer_valued(N, K, 171 + N)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    tmg.gemm(*_gpu(A, B), D, M=M, N=N, K=K)
    tmg.check()
    if K == 0:
        assert (D == 0).all()
        return
    parity.check_exact_bf16(parity.bf16_bits(D), parity.ref_full(A, B, oracle.BF16))


def test_skinny_long_k_integer_exact(tmg):
    """K = 65536 on the skinny path: each tile's K run spans many CTAs."""
    M, N, K = 4, 256, 65536
    A = inputs.integer_valued(M, K, 181, lo=-1, hi=1)
    B = inputs.integer_valued(N, K, 182, lo=-1, hi=1)
    D = tmg.gemm(*_gpu(A, B), path="skinny")
    tmg.check()
    parity.check_exact_bf16(parity.bf16_bits(D), parity.ref_full(A, B, oracle.BF16))


def test_ffma_nested_output_layout(tmg):
    """D written through a nested column mode: n = n0 + 4 n1 at n0 * 16 + n1
    inside each row."""
    M, N, K = 9, 16, 33
    A = inputs.uniform_f32(M, K, 191)
    B = inputs.uniform_f32(N, K, 192)
    Dbuf = torch.full((M, N), float("nan"), device=DEV)
    tmg.gemm(A.to(DEV), B.to(DEV), Dbuf, M=M, N=N, K=K, layoutD=((M, (4, 4)), (N, (4, 1))))
    tmg.check()
    ref = parity.ref_full(A, B, oracle.F32)
    d = Dbuf.cpu()
    got = torch.empty(M, N)
    for n in range(N):
        got[:, n] = d[:, (n % 4) * 4 + n // 4]
    parity.check_fp32(got, ref)
