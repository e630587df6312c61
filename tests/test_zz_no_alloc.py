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

import oracle
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
    """Same kernel, same launch: for M up to 48 the fixed array holds partial
    sums for every SM, so both calls split K over the same grid and add the
    split tiles in the same fixed order: the results are equal bit for bit.
    Checked twice in a row — the second call sees whatever the first left in
    the shared array — and against sampled outputs of the oracle."""
    torch.cuda.set_device(DEV)
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(16, 28672, 8192, 1), (40, 3000, 1000, 2), (5, 1000, 512, 3)]
    for M, N, K, seed in cases:
        A = inputs.normal_bf16(M, K, 500 + seed)
        B = inputs.normal_bf16(N, K, 600 + seed, std=0.02)
        dA, dB = A.to(DEV), B.to(DEV)
        ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        _existing(native, dA, dB, ref, M, N, K, stream)
        for _ in range(2):
            D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
            _noalloc(native, dA, dB, D, M, N, K, stream)
            native.raise_on(native.lib().tmg_check(stream))
            assert torch.equal(D, ref), (M, N, K)
        _check_oracle_samples(A, B, D, M, N, K, seed)


def test_noalloc_m64_runs_on_fewer_ctas(native):
    """For M from 49 to 64 the array holds partial sums for 127 CTAs, so the
    call runs on 127 of the 152 SMs: a different stream-K split of the same
    sums, so it agrees with the allocating call within the bf16 bound (not
    bit for bit) and with the oracle on sampled outputs, on two calls in a
    row."""
    torch.cuda.set_device(DEV)
    stream = torch.cuda.current_stream().cuda_stream
    M, N, K, seed = 64, 28672, 8192, 4
    A = inputs.normal_bf16(M, K, 500 + seed)
    B = inputs.normal_bf16(N, K, 600 + seed, std=0.02)
    dA, dB = A.to(DEV), B.to(DEV)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    _existing(native, dA, dB, ref, M, N, K, stream)
    amax, bmax = parity.absmax(A), parity.absmax(B)
    first = None
    for _ in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        _noalloc(native, dA, dB, D, M, N, K, stream)
        native.raise_on(native.lib().tmg_check(stream))
        parity.check_bf16_values(parity.to_f64(D), parity.to_f64(ref), K, amax, bmax)
        if first is None:
            first = D.clone()
        else:
            assert torch.equal(D, first)       # the fix-up order does not depend on timing
    _check_oracle_samples(A, B, D, M, N, K, seed)


def _check_oracle_samples(A, B, D, M, N, K, seed):
    rng = np.random.default_rng(seed)
    ns = np.concatenate([rng.integers(0, N, 600), [0, N - 1]])
    ms = np.repeat(np.arange(M), ns.size)
    ns = np.tile(ns, M)
    ref = parity.ref_entries(A, B, oracle.BF16, ms, ns)
    parity.check_bf16_values(parity.to_f64(D)[ms, ns], ref, K, parity.absmax(A), parity.absmax(B))


def test_noalloc_rejects_sizes_beyond_its_scratch(native):
    L = native.lib()
    dummy = torch.empty(16, dtype=torch.bfloat16, device=DEV)
    p = dummy.data_ptr()
    assert L.tmg_gemm_skinny_noalloc(p, p, p, 65, 8, 8, 8, 8, 8, None) == native.ERR_INVALID_ARG
    assert "64" in L.tmg_last_error().decode()
    assert L.tmg_gemm_skinny_noalloc(p, p, p, 16, 524288 + 128, 8, 8, 8, 524288 + 128,
                                     None) == native.ERR_INVALID_ARG
    assert "524288" in L.tmg_last_error().decode()
