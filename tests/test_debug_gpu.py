"""The debug aids, on the GPU.

* The bounds-checked build (libtmg_debug.so, same ABI): small parity cases of
  every kernel family run through it, match the oracle, and report no
  out-of-range offset; its probe entry point shows that a caught offset
  reaches tmg_check as TMG_ERR_BOUNDS while the GPU stays usable.
* TMG_LOG=1: every call names the kernel family and schedule it chose.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tiled_mma_atom_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dbg():
    """The package bound to the debug build for this module, the normal
    build restored afterwards."""
    import __graft_entry__
    __graft_entry__.build()
    from tiled_mma_atom_gb300 import _native, build
    build.build(debug_bounds=True)
    import tiled_mma_atom_gb300 as t
    _native.use_library(_native.DEBUG_LIB_PATH)
    try:
        assert _native.lib().tmg_debug_build() == 1
        yield t
    finally:
        _native.use_library(os.path.join(_native.HERE, "libtmg.so"))


def _bf16_case(t, M, N, K, seed, **kw):
    A, B = inputs.normal_bf16(M, K, seed), inputs.normal_bf16(N, K, seed + 1)
    D = t.gemm(A.to(DEV), B.to(DEV), **kw)
    t.check()
    parity.check_bf16(D, parity.ref_full(A, B, oracle.BF16), K, parity.absmax(A), parity.absmax(B))


def test_debug_build_runs_every_family_clean(dbg, monkeypatch):
    t = dbg
    # fp32 on the CUDA cores, through a general (column-major) layout of A
    M, N, K = 129, 130, 72
    A, B = inputs.uniform_f32(K, M, 1), inputs.uniform_f32(N, K, 2)
    la = ((M, K), (1, M))
    D = t.gemm(A.to(DEV), B.to(DEV), M=M, N=N, K=K, layoutA=la)
    t.check()
    ref = oracle.gemm(inputs.bits_of(A), oracle.make_layout((M, K), (1, M)), inputs.bits_of(B),
                      oracle.row_major(N, K), oracle.F32, M, N, K)
    parity.check_fp32(D, ref)
    # bf16 tensor cores: one CTA, CTA pairs with a stream-K tail, skinny
    _bf16_case(t, 200, 300, 136, 3, path="tc_single")
    monkeypatch.setenv("TMG_TC_PAIR_BN", "128")
    monkeypatch.setenv("TMG_TC_PAIR_SCHED", "sk")
    _bf16_case(t, 520, 600, 256, 5, path="tc_pair")
    monkeypatch.delenv("TMG_TC_PAIR_BN")
    monkeypatch.delenv("TMG_TC_PAIR_SCHED")
    _bf16_case(t, 24, 3000, 1000, 7, path="skinny")
    # MXFP4 on CTA pairs and on one CTA
    for kernel in ("pair", "single"):
        monkeypatch.setenv("TMG_MXFP4_KERNEL", kernel)
        M, N, K = 300, 392, 1024
        A, B = inputs.random_fp4_codes(M, K, 9), inputs.random_fp4_codes(N, K, 10)
        sA, sB = inputs.random_e8m0(M, K, 11), inputs.random_e8m0(N, K, 12)
        D = t.gemm_mxfp4(*(x.to(DEV) for x in (A, B, sA, sB)))
        t.check()
        ref = oracle.gemm_mxfp4(A.numpy(), B.numpy(), sA.numpy(), sB.numpy(), M, N, K)
        amax = float(np.abs(oracle.read_mxfp4(A.numpy(), sA.numpy(), M, K)).max())
        bmax = float(np.abs(oracle.read_mxfp4(B.numpy(), sB.numpy(), N, K)).max())
        parity.check_bf16(D, ref, K, amax, bmax)
    monkeypatch.delenv("TMG_MXFP4_KERNEL")
    # fused E4M3 with scales, bias and GELU
    M, N, K = 600, 520, 512
    A, B = inputs.normal_e4m3(M, K, 13), inputs.normal_e4m3(N, K, 14)
    sa, sb, bias = inputs.uniform_vec(M, 15), inputs.uniform_vec(N, 16), inputs.normal_vec(N, 17)
    D = t.gemm_fused(A.to(DEV), B.to(DEV), scale_a=sa.to(DEV), scale_b=sb.to(DEV), bias=bias.to(DEV),
                     epilogue="bias_gelu")
    t.check()
    ref = oracle.gemm_fused(inputs.bits_of(A), inputs.bits_of(B), oracle.E4M3, M, N, K, sa.numpy(), sb.numpy(),
                            bias.numpy(), "bias_gelu")
    parity.check_fused_values(parity.to_f64(D), ref, K, parity.absmax(A), parity.absmax(B),
                              sa.max().item(), sb.max().item())
    # W4A8: the decode kernel and the general (unpack + pair) path, exact
    for M, N, K in ((16, 1000, 1024), (300, 260, 512)):
        A, B = inputs.random_int8(M, K, 18), inputs.random_int4_packed(N, K, 19)
        D = t.gemm_w4a8(A.to(DEV), B.to(DEV))
        t.check()
        assert np.array_equal(D.cpu().numpy().astype(np.int64), oracle.gemm_w4a8(A.numpy(), B.numpy(), M, N, K))


def test_debug_bounds_probe_reports_and_gpu_stays_usable(dbg):
    t = dbg
    from tiled_mma_atom_gb300 import _native
    _native.raise_on(_native.lib().tmg_debug_bounds_probe(None))
    with pytest.raises(t.TmgError) as ei:
        t.check()
    assert ei.value.status == _native.ERR_BOUNDS
    assert "outside its buffer" in str(ei.value)
    _bf16_case(t, 130, 200, 64, 21)          # the next GEMM is clean and correct
    t.check()


def test_log_names_the_chosen_kernel():
    code = ("import torch, tiled_mma_atom_gb300 as t;"
            "A = torch.randn(512, 256, dtype=torch.bfloat16, device='cuda');"
            "B = torch.randn(768, 256, dtype=torch.bfloat16, device='cuda');"
            "t.gemm(A, B); t.gemm(A[:16], B); t.check()")
    env = dict(os.environ, TMG_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("tmg: ")]
    assert len(lines) == 2, r.stderr
    assert "bf16 512x768x256 -> " in lines[0] and "tiles" in lines[0]
    assert "skinny_tc_kernel" in lines[1]
    quiet = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT,
                           env=dict(os.environ, TMG_LOG="0"))
    assert quiet.returncode == 0 and "tmg: " not in quiet.stderr


def test_log_shows_the_cost_model_choices():
    """The cost model's choices for three shapes, as TMG_LOG reports them:
    bf16 4096^3 on 224-wide pair tiles in four whole data-parallel waves
    (16 x 19 = 304 tiles on 76 pairs), 1024^3 on one-CTA 128x64 tiles, and
    2048^3 at K = 4096 on 256-wide pair tiles in one partial wave (64 of the
    76 pairs) rather than one-CTA tiles in two waves.  The pair tiles run in
    groups of 16 M-tiles while sixteen 256-row A panels take at most 32 MB
    (K = 4096 bf16: 2 MB each) and in groups of 8 beyond (K = 8192)."""
    code = ("import torch, tiled_mma_atom_gb300 as t\n"
            "for (M, N, K) in ((4096, 4096, 4096), (1024, 1024, 1024), (2048, 2048, 4096), (2048, 2048, 8192)):\n"
            "    A = torch.randn(M, K, dtype=torch.bfloat16, device='cuda')\n"
            "    B = torch.randn(N, K, dtype=torch.bfloat16, device='cuda')\n"
            "    t.gemm(A, B)\n"
            "t.check()\n")
    env = dict(os.environ, TMG_LOG="1")
    env.pop("TMG_TC_PAIR_BN", None)
    env.pop("TMG_TC_PAIR_SCHED", None)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("tmg: ")]
    assert len(lines) == 4, r.stderr
    assert "tc2_gemm_kernel" in lines[0] and "256x224 tiles" in lines[0] and "304 data-parallel + 0 stream-K" in lines[0]
    assert "groups of 16 M-tiles" in lines[0]
    assert "tc_bf16_kernel" in lines[1] and "128x64 tiles" in lines[1]
    assert "tc2_gemm_kernel" in lines[2] and "256x256 tiles" in lines[2] and "+ 0 stream-K" in lines[2]
    assert "groups of 16 M-tiles" in lines[2]
    assert "tc2_gemm_kernel" in lines[3] and "groups of 8 M-tiles" in lines[3]

