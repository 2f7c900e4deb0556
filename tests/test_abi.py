"""The C-ABI library builds, loads, exports every declared symbol, and rejects
bad arguments before touching the GPU.  No GPU needed."""
import ctypes as ct
import os
import re

import pytest

import rns_emulated_fp64_gb300 as os2
from rns_emulated_fp64_gb300 import binding

HDR = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "os2.h")


def declared_functions():
    src = open(HDR).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(os2_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = os2.load()
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), f"{name} missing from {binding.lib_path()}"
    assert set(names) == set(binding.EXPORTS)


def test_library_is_in_tree():
    p = os.path.realpath(binding.lib_path())
    root = os.path.realpath(os.path.dirname(os.path.dirname(__file__)))
    assert p.startswith(root)


def test_moduli_and_status_strings():
    assert os2.moduli(20) == [256, 255, 253, 251, 247, 241, 239, 233, 229, 227, 223, 217, 211,
                              199, 197, 193, 191, 181, 179, 173]
    lib = os2.load()
    assert lib.os2_moduli(0, (ct.c_int32 * 20)()) == 0
    assert lib.os2_moduli(21, (ct.c_int32 * 21)()) == 0
    for s in range(8):
        assert os2.status_string(s)
    assert os2.status_string(99) == "unknown status"


def test_workspace_sizes():
    # N*(m+n)*ceil64(k)*2 bytes of planes plus N*m*ceil16(n) bytes of product residues
    w = os2.workspace_size(8192, 8192, 8192, 16, "fast")
    assert w >= 16 * (8192 + 8192) * 8192 * 2 + 16 * 8192 * 8192
    assert w < 1.01 * (16 * (8192 + 8192) * 8192 * 2 + 16 * 8192 * 8192) + 4096
    assert os2.workspace_size(100, 37, 65, 14, "accurate") > os2.workspace_size(100, 37, 65, 14, "fast")
    assert os2.workspace_size(-1, 4, 4, 14, "fast") == 0
    assert os2.workspace_size(4, 4, 4, 0, "fast") == 0
    assert os2.workspace_size(4, 4, 4, 21, "fast") == 0
    assert os2.workspace_size(4, 4, 4, 14, 7) == 0
    h = os2.host_workspace_size(64, 64, 64, 14)
    assert h >= os2.workspace_size(64, 64, 64, 14) + 3 * 64 * 64 * 8
    assert os2.launch_count(64, 64, 64, 14, "fast") == 4
    assert os2.launch_count(64, 64, 64, 14, "accurate") == 7
    # default (and CUDA-core CRT): row panels of about 2048 rows for m >= 4096
    for v in (os2.CRT_AUTO, os2.CRT_SIMT):
        os2.set_crt_variant(v)
        assert os2.launch_count(4095, 64, 64, 14, "fast") == 4          # one row panel
        assert os2.launch_count(8192, 64, 64, 14, "fast") == 1 + 3 * 4   # four row panels
        assert os2.launch_count(8192, 64, 64, 14, "accurate") == 4 + 3 * 4
        assert os2.launch_count(8192, 64, 8192, 14, "accurate") == 3 + 2 + 3 * 4
    # tensor-core CRT: one pass whatever m
    os2.set_crt_variant(os2.CRT_TC)
    try:
        assert os2.launch_count(4095, 64, 64, 14, "fast") == 4
        assert os2.launch_count(8192, 64, 64, 14, "fast") == 4
        assert os2.launch_count(8192, 64, 64, 14, "accurate") == 7
        assert os2.launch_count(8192, 64, 8192, 14, "accurate") == 3 + 2 + 3   # 2 bound segments
    finally:
        os2.set_crt_variant(os2.CRT_AUTO)
    assert os2.load().os2_set_crt_variant(3) == 1


def test_argument_errors_are_synchronous():
    lib = os2.load()
    P = ct.c_void_p(0x1000)      # never dereferenced: every case fails validation first
    g = lib.os2_gemm
    assert g(-1, 4, 4, P, 4, P, 4, P, 4, 14, 0, None, 0, None) == binding.ERR_INVALID_ARG
    assert g(4, 4, 4, P, 3, P, 4, P, 4, 14, 0, None, 0, None) == binding.ERR_INVALID_ARG   # lda < k
    assert g(4, 4, 4, P, 4, P, 3, P, 4, 14, 0, None, 0, None) == binding.ERR_INVALID_ARG   # ldb < k
    assert g(4, 5, 4, P, 4, P, 4, P, 4, 14, 0, None, 0, None) == binding.ERR_INVALID_ARG   # ldc < n
    assert g(4, 4, 4, P, 4, P, 4, P, 4, 0, 0, None, 0, None) == binding.ERR_INVALID_ARG    # N
    assert g(4, 4, 4, P, 4, P, 4, P, 4, 21, 0, None, 0, None) == binding.ERR_INVALID_ARG
    assert g(4, 4, 4, P, 4, P, 4, P, 4, 14, 2, None, 0, None) == binding.ERR_INVALID_ARG   # mode
    assert g(4, 4, 4, None, 4, P, 4, P, 4, 14, 0, None, 0, None) == binding.ERR_INVALID_ARG
    assert g(4, 4, 1 << 24, P, 1 << 24, P, 1 << 24, P, 4, 14, 0, None, 0, None) == binding.ERR_UNSUPPORTED
    assert g(4, 4, 1 << 19, P, 1 << 19, P, 1 << 19, P, 4, 14, 1, None, 0, None) == binding.ERR_UNSUPPORTED
    assert g(4, 4, 1 << 19, P, 1 << 19, P, 1 << 19, P, 4, 14, 0, None, 0, None) == binding.ERR_WORKSPACE
    assert g(4, 4, 4, P, 4, P, 4, P, 4, 14, 0, None, 0, None) == binding.ERR_WORKSPACE
    assert g(4, 4, 4, P, 4, P, 4, P, 4, 14, 0, ct.c_void_p(0x1001), 1 << 20, None) == binding.ERR_WORKSPACE
    assert g(4, 4, 4, ct.c_void_p(0x1004), 4, P, 4, P, 4, 14, 0, None, 0, None) == binding.ERR_INVALID_ARG
    r = lib.os2_residues
    assert r(4, 10, P, 10, P, 14, P, 32, None) == binding.ERR_INVALID_ARG    # ldp % 64
    assert r(4, 100, P, 100, P, 14, P, 64, None) == binding.ERR_INVALID_ARG  # ldp < k
    gr = lib.os2_gemm_residues
    assert gr(4, 4, 4, P, P, 64, 14, 0, P, 8, 0, None) == binding.ERR_INVALID_ARG   # ldo % 16 for int8
    assert gr(4, 4, 4, P, P, 64, 14, 2, P, 16, 0, None) == binding.ERR_INVALID_ARG  # out kind
    assert gr(4, 4, 4, P, P, 64, 14, 0, P, 16, 5, None) == binding.ERR_INVALID_ARG  # variant
    assert gr(4, 4, 4, P, P, 64, 14, 0, P, 16, binding.GEMM_TC_I8, None) == binding.ERR_INVALID_ARG
    big = 1 << 17
    assert gr(4, 4, big, P, P, big, 14, 1, P, 4, 0, None) == binding.ERR_UNSUPPORTED  # raw int32 k limit
    c = lib.os2_crt
    assert c(4, 4, P, 2, 14, P, P, P, 4, None, None) == binding.ERR_INVALID_ARG     # ldcres < n
    assert lib.os2_set_gemm_variant(5) == binding.ERR_INVALID_ARG
    assert lib.os2_set_gemm_variant(binding.GEMM_TC_I8) == binding.OK
    assert lib.os2_set_gemm_variant(binding.GEMM_S8_SYNC) == binding.OK
    assert lib.os2_set_gemm_variant(binding.GEMM_TC) == binding.OK
    w = lib.os2_wait_selftest
    assert w(0, None, None) == binding.ERR_INVALID_ARG                 # limit < 1
    assert w((1 << 34) + 1, None, None) == binding.ERR_INVALID_ARG     # limit > 2^34


def test_binding_raises_without_fallback(monkeypatch):
    """The product path never routes around libos2."""
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding._build, "LIB", "/nonexistent/libos2.so")
    with pytest.raises(RuntimeError):
        binding.load(build_if_missing=False)


def test_gemm_residues_checks_plane_dtype():
    """The int8-plane variant takes int8 planes, the others FP16 ones; a
    mismatch is refused before any call into the library."""
    import torch
    f16 = torch.zeros((1, 4, 64), dtype=torch.float16)
    i8 = torch.zeros((1, 4, 64), dtype=torch.int8)
    with pytest.raises(TypeError):
        binding.gemm_residues(f16, f16, 64, variant=binding.GEMM_S8_SYNC)
    with pytest.raises(TypeError):
        binding.gemm_residues(i8, i8, 64, variant=binding.GEMM_TC)
