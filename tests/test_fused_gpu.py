"""GPU parity of the fused GEMM (tmg_gemm_fused): bf16 and E4M3 inputs,
per-row / per-column scales, bias and the relu / silu / gelu epilogues,
against the CPU oracle's fp64 evaluation of
y = act(acc * scale_a[m] * scale_b[n] + bias[n]), through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_mma_atom_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
EPIS = ["none", "bias", "bias_relu", "bias_silu", "bias_gelu"]
KINDS = {"bf16": (inputs.normal_bf16, torch.bfloat16, oracle.BF16),
         "e4m3": (inputs.normal_e4m3, torch.float8_e4m3fn, oracle.E4M3)}


@pytest.fixture(scope="module")
def tmg():
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as t
    yield t
    t.check()


def _vecs(M, N, seed, epi):
    sa = inputs.uniform_vec(M, seed)
    sb = inputs.uniform_vec(N, seed + 1)
    bias = inputs.normal_vec(N, seed + 2) if epi != "none" else None
    return sa, sb, bias


def _run(tmg, A, B, sa, sb, bias, epi):
    d = lambda t: None if t is None else t.to(DEV)
    D = tmg.gemm_fused(A.to(DEV), B.to(DEV), scale_a=d(sa), scale_b=d(sb), bias=d(bias), epilogue=epi)
    tmg.check()
    return D


def _np(t):
    return None if t is None else t.numpy()


@pytest.mark.parametrize("kind", sorted(KINDS))
@pytest.mark.parametrize("epi", EPIS)
def test_fused_vs_oracle(tmg, kind, epi):
    """Ragged M and N (several 256 x 256 pair tiles and partial ones) and a K
    that is not a whole number of K blocks."""
    gen, _, odt = KINDS[kind]
    M, N, K = 300, 520, 320
    A, B = gen(M, K, 301), gen(N, K, 302)
    sa, sb, bias = _vecs(M, N, 303, epi)
    D = _run(tmg, A, B, sa, sb, bias, epi)
    ref = oracle.gemm_fused(inputs.bits_of(A), inputs.bits_of(B), odt, M, N, K, _np(sa), _np(sb), _np(bias), epi)
    parity.check_fused_values(parity.to_f64(D), ref, K, parity.absmax(A), parity.absmax(B),
                              float(sa.max()), float(sb.max()))


@pytest.mark.parametrize("width", [128, 192, 224, 256])
@pytest.mark.parametrize("kind", sorted(KINDS))
def test_fused_integer_exact_through_stream_k(tmg, kind, width, monkeypatch):
    """Integer inputs, power-of-two scales, integer bias, relu: every step is
    exact in fp32, so D must be the bf16 rounding of the exact value, bit for
    bit.  2048 x 2560 leaves a partial last wave: its tiles are summed from
    stream-K partials before the epilogue (224-wide tiles: the epilogue warps
    of a lane quarter split 7 column chunks 4 + 3).  Twice: the counters
    reset."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", str(width))
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", "sk")
    _, dt, odt = KINDS[kind]
    M, N, K = 2048, 2560, 1024
    A = inputs.integer_valued(M, K, 311, dtype=dt)
    B = inputs.integer_valued(N, K, 312, dtype=dt)
    g = torch.Generator().manual_seed(313)
    sa = 2.0 ** torch.randint(-1, 2, (M,), generator=g).float()
    sb = 2.0 ** torch.randint(-1, 2, (N,), generator=g).float()
    bias = torch.randint(-8, 9, (N,), generator=g).float()
    D1 = _run(tmg, A, B, sa, sb, bias, "bias_relu").clone()
    D2 = _run(tmg, A, B, sa, sb, bias, "bias_relu")
    assert torch.equal(D1, D2)
    ref = oracle.gemm_fused(inputs.bits_of(A), inputs.bits_of(B), odt, M, N, K, sa.numpy(), sb.numpy(),
                            bias.numpy(), "bias_relu")
    got = parity.bf16_bits(D2) & 0x7FFF | (parity.bf16_bits(D2) & 0x8000) * (parity.to_f64(D2) != 0)
    want = oracle.round_bf16_array(ref + 0.0)
    assert np.count_nonzero(got != want) == 0


@pytest.mark.parametrize("M", [1, 17, 130])
def test_fused_small_m(tmg, M):
    """Fewer rows than one pair tile (the second CTA's rows all out of range
    when M <= 128)."""
    N, K = 384, 256
    A, B = inputs.normal_e4m3(M, K, 321), inputs.normal_e4m3(N, K, 322)
    sa, sb, bias = _vecs(M, N, 323, "bias_gelu")
    D = _run(tmg, A, B, sa, sb, bias, "bias_gelu")
    ref = oracle.gemm_fused(inputs.bits_of(A), inputs.bits_of(B), oracle.E4M3, M, N, K, _np(sa), _np(sb),
                            _np(bias), "bias_gelu")
    parity.check_fused_values(parity.to_f64(D), ref, K, parity.absmax(A), parity.absmax(B),
                              float(sa.max()), float(sb.max()))


@pytest.mark.parametrize("epi", ["none", "bias_silu"])
def test_fused_k0(tmg, epi):
    """K = 0: the sum is empty, D = act(bias) (zeros without a bias)."""
    M, N = 33, 70
    A = torch.empty((M, 0), dtype=torch.bfloat16)
    B = torch.empty((N, 0), dtype=torch.bfloat16)
    bias = inputs.normal_vec(N, 331) if epi != "none" else None
    D = tmg.gemm_fused(A.to(DEV), B.to(DEV), bias=None if bias is None else bias.to(DEV), epilogue=epi)
    tmg.check()
    if bias is None:
        assert torch.count_nonzero(D) == 0
        return
    ref = np.array([[oracle.activation(b, epi) for b in bias.numpy().astype(np.float64)]] * M)
    np.testing.assert_allclose(parity.to_f64(D), ref, rtol=2.0 ** -8, atol=1e-6)


def test_fused_none_matches_plain_pair_gemm(tmg, monkeypatch):
    """With no scales, no bias and no activation, the fused kernel is the
    plain pair kernel at the same tile width: identical bits."""
    monkeypatch.setenv("TMG_TC_PAIR_BN", "256")
    M, N, K = 1024, 2304, 512
    A, B = inputs.normal_bf16(M, K, 341), inputs.normal_bf16(N, K, 342)
    dA, dB = A.to(DEV), B.to(DEV)
    D1 = tmg.gemm(dA, dB, path="tc_pair")
    D2 = tmg.gemm_fused(dA, dB)
    tmg.check()
    assert torch.equal(D1, D2)


def test_fused_missing_bias_raises(tmg):
    A = inputs.normal_bf16(8, 64, 351).to(DEV)
    with pytest.raises(tmg.TmgError):
        tmg.gemm_fused(A, A, epilogue="bias")


@pytest.mark.parametrize("name", [n for n, w in inputs.WORKLOADS.items() if w.epilogue])
def test_fused_workload_sampled(tmg, name):
    """The benchmark's fused workloads at full size, in the launch
    configuration it times; sampled outputs against the oracle."""
    w = inputs.WORKLOADS[name]
    A, B, sa, sb, bias = inputs.make_inputs(w)
    D = _run(tmg, A, B, sa, sb, bias, w.epilogue)
    ms, ns = parity.sample_coords(w.M, w.N, 4000, seed=17)
    odt = oracle.E4M3 if w.dtype == "e4m3" else oracle.BF16
    ref = oracle.gemm_fused_entries(inputs.bits_of(A), inputs.bits_of(B), odt, w.M, w.N, w.K, ms, ns,
                                    sa.numpy(), sb.numpy(), bias.numpy(), w.epilogue)
    parity.check_fused_values(parity.to_f64(D)[ms, ns], ref, w.K, parity.absmax(A), parity.absmax(B),
                              float(sa.max()), float(sb.max()))
