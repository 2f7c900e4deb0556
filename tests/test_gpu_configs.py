"""The five workload configurations, at their full sizes, in the launch
configuration the benchmark times (os2_gemm, default 2-SM tensor-core step 3).

Every run is compared with the CPU oracle on a seeded grid of output entries
(64 rows x 64 columns, always including the last row and column): bit-exact
FP64 results (which implies |dC_ij| <= 2^-50 (|A||B|)_ij, also checked), the
oracle's own CRT value equal to its direct exact product (|A'B'| < P/2), and
bit-exact exponents on every row and column in fast mode."""
import numpy as np
import pytest
import torch

import rns_emulated_fp64_gb300 as os2
import workloads
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
TOL = 2.0 ** -50


def run(A, Bt, N, mode, ws=None):
    Ad = torch.from_numpy(A).cuda()
    Bd = torch.from_numpy(Bt).cuda()
    C = os2.gemm(Ad, Bd, N, mode, workspace=ws)
    st = os2.get_status()
    assert st == 0, os2.status_string(st)
    return Ad, Bd, C


def check_sample(A, Bt, C, N, mode, count=64, seed=1):
    rows, cols = workloads.sample_grid(A.shape[0], Bt.shape[0], count, seed)
    ref = orc.gemm_entries(A, Bt, N, rows, cols, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0, "oracle: CRT value differs from the exact integer product"
    got = C[torch.from_numpy(rows).long().cuda()][:, torch.from_numpy(cols).long().cuda()].cpu().numpy()
    bad = np.flatnonzero(got.view(np.uint64) != ref.C.view(np.uint64))
    assert bad.size == 0, f"{bad.size} sampled entries differ from the oracle"
    absprod = np.abs(A[rows]) @ np.abs(Bt[cols]).T
    assert np.all(np.abs(got - ref.C) <= TOL * absprod)
    return ref


def test_config_64cube_normal_N14_fast_full():
    A, Bt = workloads.make_pair("normal", 64, 64, 64, seed=0)
    _, _, C = run(A, Bt, 14, "fast")
    ref = orc.gemm_entries(A, Bt, 14, want_X=False, want_c=False, want_G=False)
    assert np.array_equal(C.cpu().numpy().view(np.uint64), ref.C.view(np.uint64))


@pytest.mark.parametrize("phi", [0.5, 2.0, 4.0])
def test_config_1024cube_spread(phi):
    """1024^3, (U-0.5) exp(phi N(0,1)), N in {12,...,20}, fast and accurate."""
    A, Bt = workloads.make_pair("spread", 1024, 1024, 1024, seed=0, phi=phi)
    for N in (12, 14, 16, 18, 20):
        for mode in ("fast", "accurate"):
            Ad, Bd, C = run(A, Bt, N, mode)
            check_sample(A, Bt, C, N, mode, count=48)
            if mode == "fast":
                e, f = os2.scale(Ad, Bd, N, "fast")
                assert np.array_equal(e.cpu().numpy(), orc.scale_fast(A, N))
                assert np.array_equal(f.cpu().numpy(), orc.scale_fast(Bt, N))


@pytest.mark.parametrize("mode", ["fast", "accurate"])
def test_config_4096cube_scale_sweep(mode):
    """4096^3, all-ones and N(0,1), each times 2^s for s in {-200,...,200},
    N = 16: C scales by 2^s exactly (A scaled) and 2^2s (A and B scaled); the
    all-ones product is k 2^s on every entry (the CRT never wraps)."""
    n = 4096
    N = 16
    ws = os2.alloc_workspace(os2.workspace_size(n, n, n, N, mode))
    ones = np.ones((n, n))
    _, _, C1 = run(ones, ones, N, mode, ws)
    assert torch.all(C1 == n)
    A, Bt = workloads.make_pair("normal", n, n, n, seed=0)
    _, _, C0 = run(A, Bt, N, mode, ws)
    check_sample(A, Bt, C0, N, mode, count=32)
    C0h = C0.cpu().numpy()
    for s in (-200, -100, -50, 50, 100, 200):
        a = 2.0 ** s
        _, _, Co = run(ones * a, ones, N, mode, ws)
        assert torch.all(Co == n * a)
        _, _, Coo = run(ones * a, ones * a, N, mode, ws)
        assert torch.all(Coo == n * a * a)
        _, _, Cs = run(np.ldexp(A, s), Bt, N, mode, ws)
        assert np.array_equal(Cs.cpu().numpy().view(np.uint64), np.ldexp(C0h, s).view(np.uint64))
        _, _, Css = run(np.ldexp(A, s), np.ldexp(Bt, s), N, mode, ws)
        assert np.array_equal(Css.cpu().numpy().view(np.uint64), np.ldexp(C0h, 2 * s).view(np.uint64))


@pytest.mark.parametrize("mode", ["fast", "accurate"])
def test_config_8192cube_spread(mode):
    """8192^3, (U-0.5) exp(0.5 N(0,1)), N in {14, 16, 18}: the benchmark's
    workload, 4096 sampled entries against the oracle."""
    A, Bt = workloads.make_pair("spread", 8192, 8192, 8192, seed=0, phi=0.5)
    for N in (14, 16, 18):
        _, _, C = run(A, Bt, N, mode)
        check_sample(A, Bt, C, N, mode, count=64)
        del C
        torch.cuda.empty_cache()


def test_config_8192cube_int8_tensor_path():
    """The benchmark's workload (8192^3, 16 moduli, fast) with step 3 on the INT8
    tensor path (mma.sync s8 on int8 residue planes): 4096 sampled entries
    against the oracle, and every entry equal to the default path's."""
    A, Bt = workloads.make_pair("spread", 8192, 8192, 8192, seed=0, phi=0.5)
    Ad, Bd, C = run(A, Bt, 16, "fast")
    os2.set_gemm_variant(os2.GEMM_S8_SYNC)
    try:
        C8 = os2.gemm(Ad, Bd, 16, "fast")
        assert os2.get_status() == 0
    finally:
        os2.set_gemm_variant(os2.GEMM_TC)
    assert torch.equal(C8, C)
    check_sample(A, Bt, C8, 16, "fast", count=64)


def test_config_16384sq_k32768_spread():
    """m = n = 16384, k = 32768, (U-0.5) exp(N(0,1)), 18 moduli, fast mode."""
    A, Bt = workloads.make_pair("spread", 16384, 16384, 32768, seed=0, phi=1.0)
    _, _, C = run(A, Bt, 18, "fast")
    check_sample(A, Bt, C, 18, "fast", count=64)
