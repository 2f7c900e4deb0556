"""Seeded randomized parity sweep of the whole path.

Each case draws a shape (1..260 in every dimension), a number of moduli (1..20),
a mode, an input family and exponent spread, a step-3 kernel and a CRT kernel,
and adds zero rows and columns and subnormal entries now and then.  Every entry
of C, through os2_gemm and through os2_gemm_host, must equal the oracle's bits
([Q] 行列積への当てはめ方: the five steps; the oracle restates them exactly).
"""
import numpy as np
import pytest
import torch

import rns_emulated_fp64_gb300 as os2
import workloads
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

VARIANTS = [os2.GEMM_TC, os2.GEMM_TC_1SM, os2.GEMM_TC_I8, os2.GEMM_S8_SYNC, os2.GEMM_SIMT]
CRTS = [os2.CRT_TC, os2.CRT_SIMT, os2.CRT_AUTO]


def _cases(count=80, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        m, n, k = (int(x) for x in rng.integers(1, 261, 3))
        N = int(rng.integers(1, 21))
        mode = "fast" if rng.random() < 0.5 else "accurate"
        kind = str(rng.choice(["normal", "spread", "spread", "int"]))
        if kind == "spread":
            phi = float(rng.choice([0.5, 2.0, 6.0]))
        elif kind == "int":
            phi = float(rng.choice([3.0, 1000.0]))
        else:
            phi = 0.0
        variant = VARIANTS[int(rng.integers(len(VARIANTS)))]
        crt = CRTS[int(rng.integers(len(CRTS)))]
        out.append((i, m, n, k, N, mode, kind, phi, variant, crt))
    return out


def _bits_equal(a, b):
    a = np.ascontiguousarray(a, np.float64)
    b = np.ascontiguousarray(b, np.float64)
    return np.array_equal(a.view(np.uint64), b.view(np.uint64))


@pytest.mark.parametrize("case", _cases(), ids=lambda c: "c%d_%dx%dx%d_N%d_%s_%s_v%d_crt%d"
                         % (c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[8], c[9]))
def test_random_configuration_bit_exact(case):
    i, m, n, k, N, mode, kind, phi, variant, crt = case
    A, Bt = workloads.make_pair(kind, m, n, k, seed=100 + i, phi=phi)
    rng = np.random.default_rng(i)
    if m > 2 and rng.random() < 0.3:
        A[int(rng.integers(m))] = 0.0
    if n > 2 and rng.random() < 0.3:
        Bt[int(rng.integers(n))] = 0.0
    if rng.random() < 0.3:
        A[int(rng.integers(m)), int(rng.integers(k))] = 5e-324
    os2.set_gemm_variant(variant)
    os2.set_crt_variant(crt)
    try:
        C = os2.gemm(torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda(), N, mode).cpu().numpy()
        st = os2.get_status()
        assert st == 0, os2.status_string(st)
        Ch = torch.full((m, n), np.nan, dtype=torch.float64).pin_memory()
        os2.gemm_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(Bt).pin_memory(), Ch, N,
                      mode)
        torch.cuda.current_stream().synchronize()
        st = os2.get_status()
        assert st == 0, os2.status_string(st)
    finally:
        os2.set_gemm_variant(os2.GEMM_TC)
        os2.set_crt_variant(os2.CRT_AUTO)
    ref = orc.gemm_entries(A, Bt, N, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0
    assert _bits_equal(C, ref.C), f"os2_gemm: {np.count_nonzero(C != ref.C)} entries differ"
    assert _bits_equal(Ch.numpy(), ref.C), "os2_gemm_host differs from the oracle"


def _cases_other(count=40, seed=3031):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        m, n, k = (int(x) for x in rng.integers(1, 161, 3))
        what = str(rng.choice(["sgemm", "zgemm", "cgemm"]))
        N = int(rng.integers(1, 21))
        mode = "fast" if rng.random() < 0.5 else "accurate"
        phi = float(rng.choice([0.5, 2.0, 4.0]))
        variant = VARIANTS[int(rng.integers(len(VARIANTS)))]
        out.append((i, what, m, n, k, N, mode, phi, variant))
    return out


@pytest.mark.parametrize("case", _cases_other(), ids=lambda c: "c%d_%s_%dx%dx%d_N%d_%s_v%d"
                         % (c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[8]))
def test_random_sgemm_complex_bit_exact(case):
    """The same sweep for the SGEMM and complex products ([G] Ergebnisse and
    Bedeutung), against the oracle's binary32 rounding and its real block form."""
    i, what, m, n, k, N, mode, phi, variant = case
    omode = orc.FAST if mode == "fast" else orc.ACCURATE
    A, Bt = workloads.make_pair("spread", m, n, k, seed=300 + i, phi=phi)
    os2.set_gemm_variant(variant)
    try:
        if what == "sgemm":
            A32, B32 = A.astype(np.float32), Bt.astype(np.float32)
            C = os2.sgemm(torch.from_numpy(A32).cuda(), torch.from_numpy(B32).cuda(), N,
                          mode).cpu().numpy()
        else:
            Ai, Bi = workloads.make_pair("spread", m, n, k, seed=400 + i, phi=phi)
            dt = np.complex64 if what == "cgemm" else np.complex128
            Z, W = (A + 1j * Ai).astype(dt), (Bt + 1j * Bi).astype(dt)
            C = os2.zgemm(torch.from_numpy(Z).cuda(), torch.from_numpy(W).cuda(), N,
                          mode).cpu().numpy()
        st = os2.get_status()
        assert st == 0, os2.status_string(st)
    finally:
        os2.set_gemm_variant(os2.GEMM_TC)
    if what == "sgemm":
        ref = orc.gemm_entries(A32, B32, N, mode=omode, want_X=False, want_c=False, want_G=False,
                               out_f32=True)
        assert ref.mismatches == 0
        assert np.array_equal(C.view(np.uint32), ref.C.view(np.uint32))
    else:
        ref, r = orc.complex_gemm_entries(Z, W, N, mode=omode, single=what == "cgemm")
        assert r.mismatches == 0
        view = np.uint32 if what == "cgemm" else np.uint64
        assert np.array_equal(C.view(view), ref.view(view))
