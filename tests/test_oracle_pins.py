"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one part of the oracle to something it cannot agree with by
construction: a value the pages print, a closed form, an exact special case,
brute-force enumeration, or an independent library (numpy float64 matmul,
torch's own bf16 conversions).  A plausible mistake — a dropped term, a
transposed operand, a wrong nibble or scale index, a wrong rounding — fails at
least one of them (see the comment on each test).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tiled_mma_atom_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ layouts

def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = [int(v) for v in vals]
    return rows


def test_crd2idx_worked_example():
    """The page's worked example: (3,5) on (8,16):(1,8) -> 43 and back."""
    g = _read_golden("crd2idx_example.txt")
    L = oracle.make_layout(tuple(g["layout_shape"]), tuple(g["layout_stride"]))
    r, c, idx = g["crd2idx"]
    assert oracle.crd2idx(r, c, L) == idx
    i, r2, c2 = g["idx2crd"]
    assert oracle.idx2crd(i, L) == (r2, c2)


def test_8x16_colmajor_is_bijection_i_plus_8j():
    """(8,16):(1,8) maps (i,j) -> i + 8j, a bijection onto 0..127;
    idx2crd inverts it.  A swapped stride or mode fails here."""
    L = oracle.make_layout((8, 16), (1, 8))
    seen = set()
    for i in range(8):
        for j in range(16):
            idx = oracle.crd2idx(i, j, L)
            assert idx == i + 8 * j
            seen.add(idx)
            assert oracle.idx2crd(idx, L) == (i, j)
    assert seen == set(range(128))
    assert oracle.mode_size(L, 0) == 8 and oracle.mode_size(L, 1) == 16


def test_nested_mode_brute_force():
    """A nested mode (s0,s1):(d0,d1) takes its scalar coordinate apart
    colexicographically.  Enumerate the sub-coordinates directly and compare
    (catches a lexicographic split or swapped sub-strides)."""
    s0, s1, d0, d1 = 4, 8, 9, 36
    L = oracle.make_layout((9, (s0, s1)), (1, (d0, d1)))
    linear = 0
    for c1, c0 in itertools.product(range(s1), range(s0)):  # c0 fastest
        for m in range(9):
            assert oracle.crd2idx(m, linear, L) == m + c0 * d0 + c1 * d1
        linear += 1
    assert oracle.mode_size(L, 1) == 32
    # an irregular nested stride, nested row mode
    L2 = oracle.make_layout(((3, 5), 7), ((7, 21 * 2), 1))
    linear = 0
    for c1, c0 in itertools.product(range(5), range(3)):
        for k in range(7):
            assert oracle.crd2idx(linear, k, L2) == c0 * 7 + c1 * 42 + k
        linear += 1


def test_nested_layout_reads_like_flat_equivalent():
    """(9,(4,8)):(1,(9,36)) is the compact colex layout of (9,32):(1,9):
    decoding one buffer through either gives the same matrix."""
    buf = np.arange(9 * 32, dtype=np.float32)
    nested = oracle.make_layout((9, (4, 8)), (1, (9, 36)))
    flat = oracle.make_layout((9, 32), (1, 9))
    a = oracle.read_matrix(buf, nested, oracle.F32, 9, 32)
    b = oracle.read_matrix(buf, flat, oracle.F32, 9, 32)
    assert np.array_equal(a, b)
    # and the column-major reading of an arange is i + 9j
    i, j = np.meshgrid(np.arange(9), np.arange(32), indexing="ij")
    assert np.array_equal(a, i + 9 * j)


# ---------------------------------------------------------------- decoders

def test_bf16_decode_all_patterns_vs_torch():
    """Every one of the 65536 bf16 bit patterns widens exactly like torch's
    bfloat16 -> float32 conversion (an independent implementation)."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    got = oracle.read_matrix(pats, oracle.row_major(1, 65536), oracle.BF16, 1, 65536)[0]
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    # spot values
    assert oracle.decode_bf16(0x3F80) == 1.0
    assert oracle.decode_bf16(0xC000) == -2.0
    assert oracle.decode_bf16(0x0001) == 2.0 ** -133
    assert math.isinf(oracle.decode_bf16(0x7F80))


def test_round_bf16_vs_torch():
    """RNE to bf16 agrees with torch's float32 -> bfloat16 conversion on
    float32 inputs across the whole exponent range, subnormals included."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # add exact ties and near-ties around 1.0
    extra = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 - 2 ** -9, -(1 + 2 ** -8),
                      2.0 ** -126, 2.0 ** -133, 1.5 * 2.0 ** -133, 2.0 ** -134,
                      3.3895313892515355e38, 3.4e38, 0.0, -0.0], dtype=np.float32)
    x = np.concatenate([x, extra])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16_array(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_single_rounding_from_double():
    """A value just above a bf16 tie rounds up; rounding through float32 first
    would fall onto the tie and round down to even."""
    assert oracle.round_bf16(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.round_bf16(1 + 2 ** -8) == 0x3F80          # tie -> even
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 0x3F82      # tie -> even (up)
    assert oracle.round_bf16(-3.0) == 0xC040
    assert oracle.round_bf16(1e39) == 0x7F80                 # overflow
    assert oracle.round_bf16(float("nan")) & 0x7F80 == 0x7F80


OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
            -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_table():
    """All 16 E2M1 codes against the OCP MX table of values."""
    for code, v in enumerate(OCP_E2M1):
        got = oracle.decode_e2m1(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), code


def test_e8m0():
    assert oracle.decode_e8m0(127) == 1.0
    assert oracle.decode_e8m0(128) == 2.0
    assert oracle.decode_e8m0(126) == 0.5
    assert oracle.decode_e8m0(0) == 2.0 ** -127
    assert oracle.decode_e8m0(254) == 2.0 ** 127
    assert math.isnan(oracle.decode_e8m0(255))


def test_mxfp4_nibble_order_and_scale_block():
    """Even k in the low nibble; element k takes scale k // 32."""
    K = 64
    X = np.zeros((1, K // 2), np.uint8)
    X[0, 0] = 0x21          # k=0 -> code 1 (0.5), k=1 -> code 2 (1.0)
    X[0, 16] = 0x0F         # k=32 -> code 15 (-6), k=33 -> code 0
    S = np.array([[127, 129]], np.uint8)   # block 0 x1, block 1 x4
    d = oracle.read_mxfp4(X, S, 1, K)[0]
    assert d[0] == 0.5 and d[1] == 1.0
    assert d[32] == -24.0 and d[33] == 0.0
    assert np.count_nonzero(d) == 3


# --------------------------------------------------------------- contraction

def test_contraction_2x2x2_by_hand():
    """A = [[1,2],[3,4]], B (N x K) = [[5,6],[7,8]] -> A·Bᵀ = [[17,23],[39,53]]
    (A·B would be [[19,22],[43,50]])."""
    A = np.array([[1, 2], [3, 4]], np.float32)
    B = np.array([[5, 6], [7, 8]], np.float32)
    D = oracle.gemm(A, oracle.row_major(2, 2), B, oracle.row_major(2, 2), oracle.F32, 2, 2, 2)
    assert D.tolist() == [[17.0, 23.0], [39.0, 53.0]]


@pytest.mark.parametrize("M,N,K", [(5, 7, 11), (33, 17, 64), (1, 9, 3)])
def test_gemm_vs_numpy_float64(M, N, K):
    """Non-square random fp32 operands vs numpy's float64 a @ b.T."""
    rng = np.random.default_rng(M * 100 + N)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (N, K)).astype(np.float32)
    D = oracle.gemm(A, oracle.row_major(M, K), B, oracle.row_major(N, K), oracle.F32, M, N, K)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.allclose(D, ref, rtol=1e-13, atol=1e-13)


def test_gemm_layouts_give_same_logical_result():
    """The same logical A and B stored row-major, column-major, with padded
    leading dimensions, or as a (K,N) row-major B, read identically."""
    M, N, K = 6, 5, 7
    rng = np.random.default_rng(3)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (N, K)).astype(np.float32)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    # A column-major: buffer is A^T contiguous; layout (M,K):(1,M)
    At = np.ascontiguousarray(A.T)
    # B stored as (K, N) row-major, the naive-GEMM orientation: layout (N,K):(1,N)
    Bkn = np.ascontiguousarray(B.T)
    D1 = oracle.gemm(At, oracle.col_major(M, K), Bkn, oracle.col_major(N, K), oracle.F32, M, N, K)
    assert np.allclose(D1, ref, rtol=1e-13, atol=1e-13)
    # padded leading dimension 9 on A
    Ap = np.zeros((M, 9), np.float32)
    Ap[:, :K] = A
    D2 = oracle.gemm(Ap, oracle.row_major(M, K, ld=9), B, oracle.row_major(N, K), oracle.F32, M, N, K)
    assert np.array_equal(D2, oracle.gemm(A, oracle.row_major(M, K), B, oracle.row_major(N, K),
                                          oracle.F32, M, N, K))


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
def test_exact_all_ones(dtype):
    """All-ones operands: every entry equals K."""
    M, N, K = 3, 4, 1024
    tdt = torch.float32 if dtype == oracle.F32 else torch.bfloat16
    A = inputs.bits_of(torch.ones(M, K, dtype=tdt))
    B = inputs.bits_of(torch.ones(N, K, dtype=tdt))
    D = oracle.gemm(A, oracle.row_major(M, K), B, oracle.row_major(N, K), dtype, M, N, K)
    assert np.all(D == K)


def test_exact_identity_and_permutation():
    """B = I gives D = A; B = a permutation matrix P gives D[:, n] = A[:, p(n)]."""
    M, K = 8, 16
    A_t = inputs.normal_bf16(M, K, 11)
    A = inputs.bits_of(A_t)
    Avals = A_t.float().numpy().astype(np.float64)
    I = inputs.bits_of(torch.eye(K, dtype=torch.bfloat16))
    D = oracle.gemm(A, oracle.row_major(M, K), I, oracle.row_major(K, K), oracle.BF16, M, K, K)
    assert np.array_equal(D, Avals)
    perm = np.random.default_rng(5).permutation(K)
    P = torch.zeros(K, K, dtype=torch.bfloat16)
    P[np.arange(K), perm] = 1          # row n of B selects k = perm[n]
    D = oracle.gemm(A, oracle.row_major(M, K), inputs.bits_of(P), oracle.row_major(K, K),
                    oracle.BF16, M, K, K)
    assert np.array_equal(D, Avals[:, perm])


def test_exact_integer_valued():
    """Integers in [-2, 2]: the fp64 sums are exact; compare with an int64
    matmul."""
    M, N, K = 9, 13, 300
    A = inputs.integer_valued(M, K, 21)
    B = inputs.integer_valued(N, K, 22)
    D = oracle.gemm(inputs.bits_of(A), oracle.row_major(M, K), inputs.bits_of(B),
                    oracle.row_major(N, K), oracle.BF16, M, N, K)
    ref = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    assert np.array_equal(D, ref.astype(np.float64))


def test_transpose_symmetry_bit_exact():
    """gemm(A, B) == gemm(B, A)ᵀ exactly (same products, same k order)."""
    M, N, K = 7, 5, 40
    A = inputs.bits_of(inputs.normal_bf16(M, K, 1))
    B = inputs.bits_of(inputs.normal_bf16(N, K, 2))
    D1 = oracle.gemm(A, oracle.row_major(M, K), B, oracle.row_major(N, K), oracle.BF16, M, N, K)
    D2 = oracle.gemm(B, oracle.row_major(N, K), A, oracle.row_major(M, K), oracle.BF16, N, M, K)
    assert np.array_equal(D1, D2.T)


def test_entries_agree_with_full():
    """The per-entry path (direct from encoded operands, through layouts)
    agrees exactly with the decode-then-contract path."""
    M, N, K = 12, 10, 96
    A_t = inputs.normal_bf16(K, M, 31)                   # stored (K, M): A col-major
    B = inputs.bits_of(inputs.normal_bf16(N, K, 32))
    LA = oracle.col_major(M, K)
    LB = oracle.row_major(N, K)
    A = inputs.bits_of(A_t)
    D = oracle.gemm(A, LA, B, LB, oracle.BF16, M, N, K)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    E = oracle.gemm_entries(A, LA, B, LB, oracle.BF16, K, ms.ravel(), ns.ravel())
    assert np.array_equal(E.reshape(M, N), D)


# -------------------------------------------------------------------- MXFP4

def _decode_mx_independent(X, S, K):
    """Decode via the OCP table above and numpy indexing (not the oracle)."""
    tab = np.array(OCP_E2M1)
    lo, hi = X & 0xF, X >> 4
    codes = np.empty((X.shape[0], K), np.int64)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    scale = np.repeat(np.exp2(S.astype(np.float64) - 127), 32, axis=1)
    return tab[codes] * scale


def test_mxfp4_gemm_vs_independent_decode():
    M, N, K = 9, 6, 128
    A = inputs.random_fp4_codes(M, K, 41).numpy()
    B = inputs.random_fp4_codes(N, K, 42).numpy()
    sA = inputs.random_e8m0(M, K, 43).numpy()
    sB = inputs.random_e8m0(N, K, 44).numpy()
    D = oracle.gemm_mxfp4(A, B, sA, sB, M, N, K)
    ref = _decode_mx_independent(A, sA, K) @ _decode_mx_independent(B, sB, K).T
    # every product is a short dyadic number: both sums are exact
    assert np.array_equal(D, ref)
    E = oracle.gemm_mxfp4_entries(A, B, sA, sB, K, [0, 8, 3], [0, 5, 2])
    assert np.array_equal(E, D[[0, 8, 3], [0, 5, 2]])


def test_mxfp4_scale_doubling():
    """Raising every scale of A by one exponent step doubles D exactly."""
    M, N, K = 4, 5, 96
    A = inputs.random_fp4_codes(M, K, 51).numpy()
    B = inputs.random_fp4_codes(N, K, 52).numpy()
    sA = inputs.random_e8m0(M, K, 53).numpy()
    sB = inputs.random_e8m0(N, K, 54).numpy()
    D1 = oracle.gemm_mxfp4(A, B, sA, sB, M, N, K)
    D2 = oracle.gemm_mxfp4(A, B, sA + 1, sB, M, N, K)
    assert np.array_equal(D2, 2 * D1)


def test_mxfp4_unit_scales_all_codes():
    """Scale byte 127 (x1): row of all 16 codes dotted with a one-hot row
    reproduces each code's value; with all-ones codes (1.0 = code 2) every
    entry equals K."""
    K = 32
    codes = np.tile(np.arange(16), 2)[None, :]
    A = inputs.pack_fp4(torch.from_numpy(codes)).numpy()
    sA = np.full((1, 1), 127, np.uint8)
    for k in range(K):
        onehot = np.zeros((1, K), np.int64)
        onehot[0, k] = 2                               # code 2 = 1.0
        B = inputs.pack_fp4(torch.from_numpy(onehot)).numpy()
        d = oracle.gemm_mxfp4(A, B, sA, sA, 1, 1, K)[0, 0]
        assert d == OCP_E2M1[k % 16]
    ones = inputs.pack_fp4(torch.full((3, 64), 2)).numpy()
    s1 = np.full((3, 2), 127, np.uint8)
    assert np.all(oracle.gemm_mxfp4(ones, ones, s1, s1, 3, 3, 64) == 64)


# ------------------------------------------------------- fp8 and epilogues

def test_e4m3_spec_values():
    """OFP8 E4M3 table values (min/max subnormal and normal, 1.0, 448, NaN).
    A wrong bias (8 as in FNUZ) or a missing subnormal branch fails here."""
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for code, val in rows:
        got = oracle.decode_e4m3(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val), (code, got, val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val)), code


def test_e4m3_all_codes_match_torch():
    """Every one of the 256 codes against torch's float8_e4m3fn decode (an
    independent implementation of the same OCP format)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.decode_e4m3(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_activation_closed_forms():
    """Textbook values: sigma(1) = 0.7310585786300049 (silu(1) = sigma(1)),
    Phi(1) = 0.8413447460685429 (gelu(1) = Phi(1), gelu(-1) = -(1 - Phi(1)));
    relu, and none/bias are the identity."""
    act = oracle.activation
    assert act(1.0, "bias_silu") == pytest.approx(0.7310585786300049, abs=1e-15)
    assert act(1.0, "bias_gelu") == pytest.approx(0.8413447460685429, abs=1e-15)
    assert act(-1.0, "bias_gelu") == pytest.approx(-0.15865525393145707, abs=1e-15)
    assert act(-3.5, "bias_relu") == 0.0 and act(2.25, "bias_relu") == 2.25
    for e in ("none", "bias"):
        assert act(-7.5, e) == -7.5
    assert act(0.0, "bias_silu") == 0.0 and act(0.0, "bias_gelu") == 0.0


@pytest.mark.parametrize("epi", ["bias_silu", "bias_gelu"])
def test_activation_odd_identity(epi):
    """x*s(x) - (-x)*s(-x) = x for s = sigma and s = Phi (s(x) + s(-x) = 1):
    a sign error or a wrong argument scale inside the activation fails."""
    for x in np.linspace(-9, 9, 73):
        assert oracle.activation(x, epi) - oracle.activation(-x, epi) == pytest.approx(x, abs=1e-12)


@pytest.mark.parametrize("epi,fn", [("bias_silu", torch.nn.functional.silu),
                                    ("bias_gelu", torch.nn.functional.gelu)])
def test_activation_matches_torch_fp64(epi, fn):
    """Against torch's fp64 silu and exact (erf) gelu, an independent library."""
    x = torch.linspace(-12, 12, 241, dtype=torch.float64)
    ref = fn(x).numpy()
    got = np.array([oracle.activation(v, epi) for v in x.numpy()])
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_fused_epilogue_hand_example():
    """A = [[1,2],[3,4]], B = [[1,0],[1,1]] -> acc = [[1,3],[3,7]];
    scale_a = [2, .5] (by row of D), scale_b = [1, 3] (by column), bias =
    [10, -20] (by column): y = [[12, -2], [11.5, -9.5]].  Swapping which
    vector indexes rows or columns, or adding bias before scaling, fails."""
    A = inputs.bits_of(torch.tensor([[1.0, 2.0], [3.0, 4.0]]).to(torch.bfloat16))
    B = inputs.bits_of(torch.tensor([[1.0, 0.0], [1.0, 1.0]]).to(torch.bfloat16))
    kw = dict(scale_a=[2.0, 0.5], scale_b=[1.0, 3.0], bias=[10.0, -20.0])
    y = oracle.gemm_fused(A, B, oracle.BF16, 2, 2, 2, epilogue="bias", **kw)
    assert np.array_equal(y, [[12.0, -2.0], [11.5, -9.5]])
    r = oracle.gemm_fused(A, B, oracle.BF16, 2, 2, 2, epilogue="bias_relu", **kw)
    assert np.array_equal(r, [[12.0, 0.0], [11.5, 0.0]])
    n = oracle.gemm_fused(A, B, oracle.BF16, 2, 2, 2, epilogue="none", scale_a=[2.0, 0.5])
    assert np.array_equal(n, [[2.0, 6.0], [1.5, 3.5]])
    # the same product with E4M3 codes 1 = 0x38, 2 = 0x40, 3 = 0x44, 4 = 0x48
    A8 = np.array([[0x38, 0x40], [0x44, 0x48]], dtype=np.uint8)
    B8 = np.array([[0x38, 0x00], [0x38, 0x38]], dtype=np.uint8)
    assert np.array_equal(oracle.gemm_fused(A8, B8, oracle.E4M3, 2, 2, 2, epilogue="bias", **kw), y)


def test_fused_matches_numpy_and_entries():
    """The fused oracle against numpy's fp64 matmul of the decoded operands
    followed by the epilogue written with numpy/scipy (an independent
    evaluation), and its sampled-entry form against the full one."""
    from scipy.special import erf
    M, N, K = 37, 29, 70
    g = torch.Generator().manual_seed(5)
    A = torch.randn(M, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    B = torch.randn(N, K, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sa = torch.rand(M, generator=g).numpy() + 0.5
    sb = torch.rand(N, generator=g).numpy() + 0.5
    bias = torch.randn(N, generator=g).numpy()
    a = torch.from_numpy(A).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    b = torch.from_numpy(B).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    y = (a @ b.T) * sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :] + bias.astype(np.float64)
    ref = 0.5 * y * (1 + erf(y / np.sqrt(2)))
    got = oracle.gemm_fused(A, B, oracle.E4M3, M, N, K, sa, sb, bias, "bias_gelu")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    ms, ns = np.array([0, 36, 5, 17]), np.array([0, 28, 11, 3])
    ent = oracle.gemm_fused_entries(A, B, oracle.E4M3, M, N, K, ms, ns, sa, sb, bias, "bias_gelu")
    np.testing.assert_allclose(ent, got[ms, ns], rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------- W4A8

def test_int4_decode_matches_arithmetic_shift():
    """A nibble placed in the top half of an int8 and shifted right
    arithmetically (numpy) gives the two's complement value."""
    ref = (np.arange(16, dtype=np.uint8) << 4).view(np.int8) >> 4
    assert [oracle.decode_int4(n) for n in range(16)] == ref.tolist()


def test_w4a8_hand_example():
    """A = [[1,-2],[127,-128]], B = [[3,-1],[-8,7]] packed even-k-low:
    bytes 0xF3 and 0x78; D = [[5,-22],[509,-1912]].  A swapped nibble order
    or an unsigned decode fails."""
    A = np.array([[1, -2], [127, -128]], dtype=np.int8)
    B = np.array([[0xF3], [0x78]], dtype=np.uint8)
    assert oracle.gemm_w4a8(A, B, 2, 2, 2).tolist() == [[5, -22], [509, -1912]]


def test_w4a8_matches_numpy_int64():
    """Random int8 x packed int4 against numpy's int64 matmul of an
    independently unpacked B; the entry form against the full form."""
    M, N, K = 23, 31, 66
    A = inputs.random_int8(M, K, 91).numpy()
    Bp = inputs.random_int4_packed(N, K, 92).numpy()
    lo = (Bp << 4).view(np.int8) >> 4
    hi = Bp.view(np.int8) >> 4
    Bk = np.empty((N, K), dtype=np.int64)
    Bk[:, 0::2], Bk[:, 1::2] = lo, hi
    ref = A.astype(np.int64) @ Bk.T
    got = oracle.gemm_w4a8(A, Bp, M, N, K)
    assert np.array_equal(got, ref)
    ms, ns = np.array([0, 22, 7]), np.array([30, 0, 11])
    assert np.array_equal(oracle.gemm_w4a8_entries(A, Bp, K, ms, ns), ref[ms, ns])
