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
def test_w4a8_exact(tmg, M, N, K, monkeypatch):
    """Ragged tiles, K not a multiple of 8 or of the 4096 segment, several
    segments, the stream-K tail (2048 x 2560), a single row."""
    if (M, N) == (2048, 2560):
        monkeypatch.setenv("TMG_TC_PAIR_SCHED", "sk")
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


@pytest.mark.parametrize("M,N,K", [(1, 1000, 128), (16, 1024, 4096), (17, 777, 1280), (64, 2048, 2048),
                                   (5, 300, 1056), (33, 129, 32)])
def test_w4a8_decode_exact(tmg, M, N, K):
    """Decode shapes (M <= 64, K a multiple of 32): the weights stay 4-bit
    until the kernel; ragged N, a ragged last K block of 256, several
    partial (stream-K) tiles."""
    A, B = inputs.random_int8(M, K, 711), inputs.random_int4_packed(N, K, 712)
    assert np.array_equal(_run(tmg, A, B), oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K))


@pytest.mark.parametrize("M", [16, 17, 40])
def test_w4a8_decode_several_units_per_cta(tmg, M):
    """512 (tile, K block) units on 152 CTAs: each CTA's run of 3-4 units
    crosses tile boundaries, so runs split into segments of 1 to 4 units.
    With M <= 32 two MMA issuers take alternate units (a segment of one
    unit leaves one of them out); with M = 40 one issuer takes all.  Exact
    against the oracle, pre-shuffled and row-major weights alike."""
    N, K = 2048, 8192
    A, B = inputs.random_int8(M, K, 741), inputs.random_int4_packed(N, K, 742)
    ref = oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K)
    assert np.array_equal(_run(tmg, A, B), ref)
    Bs = tmg.w4a8_preshuffle(B.to(DEV))
    D = tmg.gemm_w4a8_preshuffled(A.to(DEV), Bs, N)
    tmg.check()
    assert np.array_equal(D.cpu().numpy(), ref)


@pytest.mark.parametrize("shuffled", [False, True])
@pytest.mark.parametrize("N,K", [(25600, 2048), (38952, 1024), (19496, 2048)])
def test_w4a8_decode_many_tiles_exact(tmg, N, K, shuffled):
    """Decode shapes with more 128-row tiles than SMs (200, 153 and 305
    tiles, the last ragged), so every CTA's stream-K run spans whole and
    shared tiles (red.adds into zeroed D).  Row-major and pre-shuffled
    weights; bit-exact."""
    M = 16
    A, B = inputs.random_int8(M, K, 751), inputs.random_int4_packed(N, K, 752)
    ref = oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K)
    got = _run_shuffled(tmg, A, B) if shuffled else _run(tmg, A, B)
    assert np.array_equal(got, ref)


def test_w4a8_decode_extreme_values_at_max_k(tmg):
    """K = 32768, the decode kernel's limit, with the values that drive its
    fp32 column sums furthest from zero: the kernel splits a = 16 hi + lo
    (hi = (a + 8) >> 4, lo in [-8, 7]) and offsets b by 8 (u = b + 8 in
    0..15), so hi = +-8 or lo = -8 against u = 15 give |sum| = 120 K, just
    below 2^22; a = -128 against b = -8 (u = 0) puts all of D = 2^25 in the
    row-sum correction."""
    M, N, K = 16, 384, 32768
    for a, byte, b in [(-128, 0x88, -8), (127, 0x77, 7), (-128, 0x77, 7), (8, 0x77, 7)]:
        A = torch.full((M, K), a, dtype=torch.int8)
        B = torch.full((N, K // 2), byte, dtype=torch.uint8)
        assert (_run(tmg, A, B) == a * b * K).all(), (a, b)


def test_w4a8_decode_and_general_paths_agree(tmg, monkeypatch):
    """The same decode-shaped problem through both paths: identical int32."""
    M, N, K = 32, 1536, 2048
    A, B = inputs.random_int8(M, K, 721), inputs.random_int4_packed(N, K, 722)
    d1 = _run(tmg, A, B)
    monkeypatch.setenv("TMG_W4A8_PATH", "general")
    d2 = _run(tmg, A, B)
    assert np.array_equal(d1, d2)
    assert np.array_equal(d1, oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K))


def test_w4a8_decode_workload_sampled(tmg):
    w = inputs.WORKLOADS["w4a8_16x28672x8192"]
    A, B = inputs.make_inputs(w)
    D = tmg.gemm_w4a8(A.to(DEV), B.to(DEV))
    tmg.check()
    rng = np.random.default_rng(12)
    ms = rng.integers(0, w.M, 4000)
    ns = np.concatenate([rng.integers(0, w.N, 3998), [0, w.N - 1]])
    ref = oracle.gemm_w4a8_entries(A.numpy(), B.numpy(), w.K, ms, ns)
    assert np.array_equal(D.cpu().numpy()[ms, ns].astype(np.int64), ref)


def _preshuffle_reference(B: np.ndarray, N: int, K: int) -> np.ndarray:
    """The pre-shuffled image, restated from its definition: 16 KB blocks
    (t, kb) of 128 rows x 256 k in order t * KB + kb; inside a block row r's
    16-byte chunk c at r * 128 + 16 * (c ^ (r % 8)); zero padding."""
    T, KB = -(-N // 128), -(-K // 256)
    padded = np.zeros((T * 128, KB * 128), np.uint8)
    padded[:N, :K // 2] = B
    blocks = padded.reshape(T, 128, KB, 8, 16).transpose(0, 2, 1, 3, 4)   # (t, kb, r, c, byte)
    out = np.zeros_like(blocks)
    for r in range(128):
        for c in range(8):
            out[:, :, r, c ^ (r % 8)] = blocks[:, :, r, c]
    return out.reshape(-1)


@pytest.mark.parametrize("N,K", [(128, 256), (300, 1056), (1000, 32)])
def test_w4a8_preshuffle_layout(tmg, N, K):
    B = inputs.random_int4_packed(N, K, 731)
    Bs = tmg.w4a8_preshuffle(B.to(DEV))
    tmg.check()
    assert Bs.numel() == tmg.w4a8_preshuffled_bytes(N, K)
    assert np.array_equal(Bs.cpu().numpy(), _preshuffle_reference(B.numpy(), N, K))


def _run_shuffled(tmg, A, B):
    N = B.shape[0]
    Bs = tmg.w4a8_preshuffle(B.to(DEV))
    D = tmg.gemm_w4a8_preshuffled(A.to(DEV), Bs, N)
    tmg.check()
    return D.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("M,N,K", [(1, 1000, 128), (16, 1024, 4096), (17, 777, 1280), (64, 2048, 2048),
                                   (5, 300, 1056), (200, 330, 544), (1, 40, 32)])
def test_w4a8_preshuffled_exact(tmg, M, N, K):
    """Pre-shuffled weights: decode shapes (the contiguous-stream kernel) and
    a larger M (the general path unpacking from the image), bit-exact."""
    A, B = inputs.random_int8(M, K, 741), inputs.random_int4_packed(N, K, 742)
    assert np.array_equal(_run_shuffled(tmg, A, B), oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K))


def test_w4a8_preshuffled_extreme_values_at_max_k(tmg):
    M, N, K = 16, 256, 32768
    for a, byte, b in [(127, 0x77, 7), (8, 0x77, 7), (-128, 0x88, -8)]:
        A = torch.full((M, K), a, dtype=torch.int8)
        B = torch.full((N, K // 2), byte, dtype=torch.uint8)
        assert (_run_shuffled(tmg, A, B) == a * b * K).all(), (a, b)


def test_w4a8_preshuffled_decode_workload_sampled(tmg):
    w = inputs.WORKLOADS["w4a8_16x28672x8192"]
    A, B = inputs.make_inputs(w)
    Bs = tmg.w4a8_preshuffle(B.to(DEV))
    D = tmg.gemm_w4a8_preshuffled(A.to(DEV), Bs, w.N)
    tmg.check()
    rng = np.random.default_rng(13)
    ms = rng.integers(0, w.M, 4000)
    ns = np.concatenate([rng.integers(0, w.N, 3998), [0, w.N - 1]])
    ref = oracle.gemm_w4a8_entries(A.numpy(), B.numpy(), w.K, ms, ns)
    assert np.array_equal(D.cpu().numpy()[ms, ns].astype(np.int64), ref)


def _biased_operands(M, N, K, a_lo, a_hi, b_lo, b_hi, seed):
    """int8 A uniform in [a_lo, a_hi] and int4 B uniform in [b_lo, b_hi],
    packed two per byte (even k low): inputs whose products all share a
    sign and a size, so the kernels' fp32 column sums grow to millions while
    keeping random low-order bits."""
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(a_lo, a_hi + 1, (M, K), generator=g, dtype=torch.int32).to(torch.int8)
    v = torch.randint(b_lo, b_hi + 1, (N, K), generator=g, dtype=torch.int32) & 15
    B = (v[:, 0::2] | (v[:, 1::2] << 4)).to(torch.uint8)
    return A, B


@pytest.mark.parametrize("path", ["decode", "general"])
def test_w4a8_large_sums_keep_low_bits(tmg, monkeypatch, path):
    """Exactness where it is hardest: column sums near the kernels' bound
    (about 2^22 for the decode kernel, just under 2^23 for the general path's
    8192-deep K segments) with random low-order bits.  A tensor core that
    dropped accumulator bits would fail here although the uniform-value
    tests pass (their partial sums are multiples of large powers of two)."""
    if path == "general":
        monkeypatch.setenv("TMG_W4A8_PATH", "general")
        M, N, K = 64, 256, 8192
    else:
        M, N, K = 16, 256, 32768
    for a_lo, a_hi, b_lo, b_hi in [(120, 127, 6, 7), (-128, -100, -8, -6), (-128, 127, -8, 7),
                                   (-128, -126, -8, -7)]:
        A, B = _biased_operands(M, N, K, a_lo, a_hi, b_lo, b_hi, 751 + a_lo)
        ref = oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K)
        assert np.array_equal(_run(tmg, A, B), ref), (path, a_lo, b_lo)


@pytest.mark.parametrize("path", ["decode", "general"])
def test_w4a8_misaligned_activations(tmg, monkeypatch, path):
    """A contiguous but starting one byte past an aligned address: the
    kernels' vector loads of A fall back to byte loads, same exact result."""
    if path == "general":
        monkeypatch.setenv("TMG_W4A8_PATH", "general")
    M, N, K = 9, 300, 1056
    A, B = inputs.random_int8(M, K, 761), inputs.random_int4_packed(N, K, 762)
    buf = torch.empty(M * K + 16, dtype=torch.int8, device=DEV)
    Ad = buf[1:1 + M * K].view(M, K)
    Ad.copy_(A.to(DEV))
    assert Ad.data_ptr() % 8 == 1
    D = tmg.gemm_w4a8(Ad, B.to(DEV))
    tmg.check()
    assert np.array_equal(D.cpu().numpy().astype(np.int64), oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K))
