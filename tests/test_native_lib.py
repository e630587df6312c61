"""Host-side checks of the C-ABI library (no GPU needed).

The library is compiled here (nvcc cross-compiles sm_103a), loaded through
ctypes, and every function include/tmg.h declares must be exported.  Calls
whose arguments are rejected before any device work are exercised too.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from tiled_mma_atom_gb300 import build
    build.build()
    from tiled_mma_atom_gb300 import _native
    return _native


def _header_functions():
    text = open(os.path.join(ROOT, "include", "tmg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tmg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_functions(native):
    assert _header_functions() == sorted(native.EXPORTS)


def test_every_declared_symbol_is_exported(native):
    out = subprocess.run(["nm", "-D", "--defined-only", native.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (tmg_\w+)", out))
    missing = [f for f in _header_functions() if f not in exported]
    assert not missing, missing
    lib = native.lib()
    for f in _header_functions():
        assert hasattr(lib, f)


def test_version_and_launch_count(native):
    lib = native.lib()
    assert lib.tmg_version() == 100
    assert lib.tmg_launch_count() == 0


def _call(native, M, N, K, dtype=1, path=0, la=None, lb=None, ld=None, ptr=16):
    lib = native.lib()
    return lib.tmg_gemm_ex(ptr, ptr, ptr, M, N, K, dtype, la, lb, ld, path, None)


def test_rejects_bad_arguments_before_device_work(native):
    assert _call(native, -1, 4, 4) == native.ERR_INVALID_ARG
    assert "negative" in native.lib().tmg_last_error().decode()
    assert _call(native, 4, 4, 4, dtype=7) == native.ERR_INVALID_ARG
    assert _call(native, 4, 4, 4, path=9) == native.ERR_INVALID_ARG
    lib = native.lib()
    assert lib.tmg_gemm_ex(None, None, 16, 4, 4, 4, 1, None, None, None, 0, None) == native.ERR_INVALID_ARG
    bad = native.make_layout((4, 5), (5, 1))          # wrong K extent
    assert _call(native, 4, 4, 4, la=bad) == native.ERR_INVALID_ARG
    assert "layoutA" in lib.tmg_last_error().decode()
    neg = native.make_layout((4, 4), (-4, 1))
    assert _call(native, 4, 4, 4, lb=neg) == native.ERR_INVALID_ARG
    zero_d = native.make_layout((4, 4), (0, 1))       # D rows would alias
    assert _call(native, 4, 4, 4, ld=zero_d) == native.ERR_INVALID_ARG
    deep = native.make_layout((4, 4), (4, 1))
    deep.depth[0] = 3
    assert _call(native, 4, 4, 4, la=deep) == native.ERR_INVALID_ARG
    nested_bad = native.make_layout(((2, 3), 4), ((1, 2), 6))   # 2*3 != 4
    assert _call(native, 4, 4, 4, la=nested_bad) == native.ERR_INVALID_ARG


def test_empty_problems_are_noops(native):
    assert _call(native, 0, 4, 4) == native.OK
    assert _call(native, 4, 0, 4) == native.OK
    lib = native.lib()
    assert lib.tmg_gemm_mxfp4(16, 16, 16, 16, 16, 0, 8, 64, None) == native.OK


def test_mxfp4_rejects_k_not_multiple_of_32(native):
    lib = native.lib()
    assert lib.tmg_gemm_mxfp4(16, 16, 16, 16, 16, 4, 4, 48, None) == native.ERR_INVALID_ARG
    assert "multiple of 32" in lib.tmg_last_error().decode()


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from tiled_mma_atom_gb300 import _native
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(_native.TmgError):
        _native.lib()


def test_fused_rejects_bad_arguments_before_device_work(native):
    lib = native.lib()
    # fp32 inputs have no tensor-core path
    assert lib.tmg_gemm_fused(16, 16, 16, 4, 4, 64, native.F32, None, None, None, 0, None) == native.ERR_UNSUPPORTED
    # an unknown input type or epilogue
    assert lib.tmg_gemm_fused(16, 16, 16, 4, 4, 64, 9, None, None, None, 0, None) == native.ERR_INVALID_ARG
    assert lib.tmg_gemm_fused(16, 16, 16, 4, 4, 64, native.BF16, None, None, None, 7, None) == native.ERR_INVALID_ARG
    # a bias epilogue without a bias
    for epi in (1, 2, 3, 4):
        assert lib.tmg_gemm_fused(16, 16, 16, 4, 4, 64, native.E4M3, None, None, None, epi,
                                  None) == native.ERR_INVALID_ARG
    assert "bias" in lib.tmg_last_error().decode()
    # negative extents, empty problems
    assert lib.tmg_gemm_fused(16, 16, 16, -1, 4, 64, native.BF16, None, None, None, 0, None) == native.ERR_INVALID_ARG
    assert lib.tmg_gemm_fused(16, 16, 16, 0, 4, 64, native.BF16, None, None, None, 0, None) == native.OK
    # E4M3 is not an element type of tmg_gemm (its D would be E4M3)
    assert _call(native, 4, 4, 4, dtype=native.E4M3) == native.ERR_INVALID_ARG


def test_w4a8_rejects_bad_arguments_before_device_work(native):
    lib = native.lib()
    assert lib.tmg_gemm_w4a8(16, 16, 16, 4, 4, 7, None) == native.ERR_INVALID_ARG      # odd K
    assert "odd" in lib.tmg_last_error().decode()
    assert lib.tmg_gemm_w4a8(16, 16, 16, -1, 4, 8, None) == native.ERR_INVALID_ARG
    assert lib.tmg_gemm_w4a8(16, 16, 16, 0, 4, 8, None) == native.OK
    assert lib.tmg_gemm_w4a8(None, None, 16, 4, 4, 8, None) == native.ERR_INVALID_ARG


def test_w4a8_preshuffled_bytes_is_host_arithmetic(native):
    """One 16 KB block per (128 weight rows, 256 k), ragged edges rounded up;
    0 for shapes the pre-shuffled layout does not take."""
    lib = native.lib()
    assert lib.tmg_w4a8_preshuffled_bytes(28672, 8192) == 28672 * 8192 // 2
    assert lib.tmg_w4a8_preshuffled_bytes(129, 288) == 2 * 2 * 16384
    assert lib.tmg_w4a8_preshuffled_bytes(1, 32) == 16384
    assert lib.tmg_w4a8_preshuffled_bytes(128, 48) == 0          # K not a multiple of 32
    assert lib.tmg_w4a8_preshuffled_bytes(0, 256) == 0
    assert lib.tmg_w4a8_preshuffled_bytes(128, 0) == 0


def test_w4a8_preshuffle_rejects_bad_arguments_before_device_work(native):
    lib = native.lib()
    assert lib.tmg_w4a8_preshuffle(16, 16, 4, 48, None) == native.ERR_INVALID_ARG      # K % 32
    assert "multiple of 32" in lib.tmg_last_error().decode()
    assert lib.tmg_w4a8_preshuffle(16, 16, -1, 64, None) == native.ERR_INVALID_ARG
    assert lib.tmg_w4a8_preshuffle(None, None, 0, 64, None) == native.OK               # empty
    assert lib.tmg_w4a8_preshuffle(None, 16, 4, 64, None) == native.ERR_INVALID_ARG
    assert lib.tmg_w4a8_preshuffle(8, 16, 4, 64, None) == native.ERR_INVALID_ARG        # misaligned
    assert lib.tmg_gemm_w4a8_preshuffled(16, 16, 16, 4, 4, 48, None) == native.ERR_INVALID_ARG
    assert lib.tmg_gemm_w4a8_preshuffled(16, 24, 16, 4, 4, 64, None) == native.ERR_INVALID_ARG
    assert lib.tmg_gemm_w4a8_preshuffled(16, 16, 16, 0, 4, 64, None) == native.OK


def test_normal_build_has_no_bounds_checks(native):
    """The normal build compiles the bounds checks out: it says so, and its
    probe entry point refuses (without touching a GPU)."""
    L = native.lib()
    assert L.tmg_debug_build() == 0
    assert L.tmg_debug_bounds_probe(None) == native.ERR_UNSUPPORTED
    assert "debug build" in L.tmg_last_error().decode()
