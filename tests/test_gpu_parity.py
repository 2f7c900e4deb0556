"""Parity of every step of the CUDA path against the CPU oracle, through the
C ABI.  Integer results (exponents, residue planes, raw products, residue
products, CRT integers) must be bit-exact; FP64 results must be bit-identical
to the oracle's correctly rounded values, which implies the stated bound
|dC_ij| <= 2^-50 (|A||B|)_ij (checked as well)."""
import numpy as np
import pytest
import torch

import rns_emulated_fp64_gb300 as os2
import workloads
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2.0 ** -50


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def status_ok():
    st = os2.get_status()
    assert st == 0, os2.status_string(st)


def assert_bits_equal(got, want, what):
    got = np.ascontiguousarray(got, np.float64)
    want = np.ascontiguousarray(want, np.float64)
    bad = np.flatnonzero(got.view(np.uint64) != want.view(np.uint64))
    assert bad.size == 0, f"{what}: {bad.size} entries differ, first {bad[:5]}: " \
                          f"{got.ravel()[bad[:5]]} vs {want.ravel()[bad[:5]]}"


def check_tolerance(C, A, Bt, rows, cols, ref):
    absprod = np.abs(A[rows]) @ np.abs(Bt[cols]).T
    assert np.all(np.abs(C - ref) <= TOL * absprod)


@pytest.fixture(params=[os2.CRT_TC, os2.CRT_SIMT, os2.CRT_AUTO],
                ids=["crt_tc", "crt_simt", "crt_auto"])
def crt_variant(request):
    """Runs a test with each choice of the kernel of steps 4 + 5 (tensor-core
    limb sums, CUDA-core multiply-adds, and the default mix of the two); all
    must give the oracle's bits."""
    os2.set_crt_variant(request.param)
    yield request.param
    os2.set_crt_variant(os2.CRT_AUTO)


SHAPES = [(64, 64, 64), (1, 1, 1), (3, 5, 7), (129, 257, 65), (300, 520, 1000), (128, 256, 960),
          (130, 140, 1921)]


# ------------------------------------------------------------------ step 1 --
@pytest.mark.parametrize("kind,phi", [("normal", 0.0), ("spread", 0.5), ("spread", 4.0)])
@pytest.mark.parametrize("N", [2, 12, 16, 20])
@pytest.mark.parametrize("k", [777, 778, 9216, 9218])
def test_scale_fast_parity(kind, phi, N, k):
    """Rows of 256-thread (k <= 8192) and 512-thread CTAs, odd k (rows that
    alternate between 16-byte aligned and not, so both the two-entry vector
    loads and the scalar loads run) and even k.  Zero rows, subnormal-only
    rows and entries."""
    A, Bt = workloads.make_pair(kind, 257, 130, k, seed=N, phi=phi)
    A[5] = 0.0
    A[7, ::3] = 5e-324
    A[9] = 5e-324
    e, f = os2.scale(dev(A), dev(Bt), N, "fast")
    status_ok()
    assert np.array_equal(e.cpu().numpy(), orc.scale_fast(A, N))
    assert np.array_equal(f.cpu().numpy(), orc.scale_fast(Bt, N))


def test_scale_fast_nonfinite_sets_status():
    """Inf in a row of A, then NaN in a column of B, set the status word."""
    A, Bt = workloads.make_pair("normal", 40, 30, 1024, seed=1)
    A[3, 17] = np.inf
    os2.scale(dev(A), dev(Bt), 16, "fast")
    assert os2.get_status() == os2.binding.ERR_NONFINITE
    Bt[2, 5] = np.nan
    A[3, 17] = 1.0
    os2.scale(dev(A), dev(Bt), 16, "fast")
    assert os2.get_status() == os2.binding.ERR_NONFINITE


@pytest.mark.parametrize("N", [4, 14, 20])
def test_scale_accurate_parity(N):
    A, Bt = workloads.make_pair("spread", 200, 150, 333, seed=N, phi=2.0)
    Bt[3] = 0.0
    e, f = os2.scale(dev(A), dev(Bt), N, "accurate")
    status_ok()
    ee, ff = orc.scale_accu(A, Bt, N)
    assert np.array_equal(e.cpu().numpy(), ee)
    assert np.array_equal(f.cpu().numpy(), ff)


# ------------------------------------------------------------------ step 2 --
@pytest.mark.parametrize("N", [1, 7, 16, 20])
@pytest.mark.parametrize("kind,phi", [("spread", 4.0), ("normal", 0.0)])
def test_residue_planes_parity(N, kind, phi):
    A, _ = workloads.make_pair(kind, 67, 1, 301, seed=3, phi=phi)
    A[2, 0] = -2.0 ** 1000
    A[4, :] = 0.0
    e = orc.scale_fast(A, N)
    planes = os2.residues(dev(A), dev(e), N)
    status_ok()
    got = planes.cpu().numpy()
    assert got.shape == (N, 67, 320)
    want = orc.residues(A, e, N)
    assert np.array_equal(got[:, :, :301].astype(np.int64), want.astype(np.int64))
    assert np.all(got[:, :, 301:] == 0)


def test_residues_extreme_exponents():
    """Exponents far from the fast-mode choice exercise every word count of
    the integer split: integers just below and just above 2^59 and 2^74 (the
    limits of four and five 15-bit words), up to just below 2^89, and deep
    right shifts."""
    rng = np.random.default_rng(11)
    X = rng.standard_normal((40, 64))
    X[7, 5] = -X[7, 5]
    E = int(np.frexp(np.abs(X).max())[1])          # |x| < 2^E
    for N in (5, 18, 20):
        for e_val in (-60, -1, 0, 30, 59 - E, 60 - E, 74 - E, 75 - E, 83 - E, 89 - E):
            e = np.full(40, e_val, np.int32)
            planes = os2.residues(dev(X), dev(e), N)
            status_ok()
            want = orc.residues(X, e, N)
            assert np.array_equal(planes.cpu().numpy()[:, :, :64].astype(np.int64),
                                  want.astype(np.int64)), (N, e_val)


def test_residues_integer_too_wide_is_reported():
    """An exponent that makes |trunc(x 2^e)| reach 2^89 (beyond every
    exponent step 1 produces) sets the range status instead of writing wrong
    residues."""
    X = np.full((2, 64), 0.75)                     # |x| < 2^0
    e = np.array([90, 88], np.int32)               # row 0: 0.75 * 2^90 >= 2^89
    planes = os2.residues(dev(X), dev(e), 3)
    assert os2.get_status() == os2.binding.ERR_RANGE
    status_ok()                                    # get_status cleared it
    want = orc.residues(X[1:], e[1:], 3)
    assert np.array_equal(planes.cpu().numpy()[:, 1, :64].astype(np.int64),
                          want[:, 0].astype(np.int64))


# ------------------------------------------------------------------ step 3 --
def _planes_pair(m, n, k, N, seed=0, kind="spread", phi=1.0):
    A, Bt = workloads.make_pair(kind, m, n, k, seed=seed, phi=phi)
    e = orc.scale_fast(A, N)
    f = orc.scale_fast(Bt, N)
    return A, Bt, e, f, os2.residues(dev(A), dev(e), N), os2.residues(dev(Bt), dev(f), N)


def _step3(RA, RB, k, out_kind, variant):
    """os2_gemm_residues on the FP16 planes, or on int8 copies of them for the
    variant that reads int8 planes."""
    if variant == os2.GEMM_S8_SYNC:
        RA, RB = RA.to(torch.int8), RB.to(torch.int8)
    return os2.gemm_residues(RA, RB, k, out_kind, variant)


def _int_product(RA, RB, k):
    a = RA.float().cpu().numpy().astype(np.int64)[:, :, :k]
    b = RB.float().cpu().numpy().astype(np.int64)[:, :, :k]
    return np.einsum("lik,ljk->lij", a, b)


@pytest.mark.parametrize("variant", [os2.GEMM_TC, os2.GEMM_SIMT, os2.GEMM_S8_SYNC])
@pytest.mark.parametrize("m,n,k", [(128, 128, 64), (129, 257, 65), (300, 200, 1100), (64, 64, 4097)])
def test_raw_int32_products_bit_exact(variant, m, n, k):
    N = 3
    A, Bt, e, f, RA, RB = _planes_pair(m, n, k, N)
    G = _step3(RA, RB, k, os2.OUT_RAW_INT32, variant)
    status_ok()
    want = _int_product(RA, RB, k)
    assert np.array_equal(G.cpu().numpy()[:, :, :n].astype(np.int64), want)


@pytest.mark.parametrize("variant", [os2.GEMM_TC, os2.GEMM_TC_1SM, os2.GEMM_SIMT, os2.GEMM_S8_SYNC])
@pytest.mark.parametrize("m,n,k,N", [(128, 256, 64, 2), (513, 700, 3000, 16), (256, 256, 961, 5), (129, 257, 65, 14), (300, 520, 1000, 16),
                                     (256, 512, 2000, 20), (70, 33, 3000, 9)])
def test_modp_products_bit_exact(variant, m, n, k, N):
    A, Bt, e, f, RA, RB = _planes_pair(m, n, k, N, seed=m)
    c = _step3(RA, RB, k, os2.OUT_MODP_INT8, variant)
    status_ok()
    rows = np.arange(m, dtype=np.int32)
    cols = np.arange(n, dtype=np.int32)
    ref = orc.gemm_entries(A, Bt, N, rows, cols, want_X=False, want_G=False)
    got = np.transpose(c.cpu().numpy()[:, :, :n], (1, 2, 0))
    assert np.array_equal(got, ref.c)


def test_int32_accumulation_worst_case():
    """[Q] 手順3: all residues -128 with the inner dimension just below 2^17
    gives 2^14 (2^17 - 64) < 2^31, exact."""
    k = (1 << 17) - 64
    RA = torch.full((1, 128, k), -128.0, dtype=torch.float16, device=DEV)
    RB = torch.full((1, 128, k), -128.0, dtype=torch.float16, device=DEV)
    for variant in (os2.GEMM_TC, os2.GEMM_S8_SYNC):
        G = _step3(RA, RB, k, os2.OUT_RAW_INT32, variant)
        status_ok()
        assert torch.all(G[:, :, :128] == 16384 * k), variant
    for variant in (os2.GEMM_TC, os2.GEMM_TC_1SM, os2.GEMM_S8_SYNC):
        c = _step3(RA, RB, k, os2.OUT_MODP_INT8, variant)
        status_ok()
        assert torch.all(c[:, :, :128] == 0)   # 2^14 k is a multiple of 256


def test_modp_alternating_extremes():
    """Residues at the ends of every modulus range, products of alternating
    sign: the in-TMEM reduction keeps every partial sum exact."""
    N, m, n, k = 20, 128, 256, 4096
    mods = os2.moduli(N)
    rng = np.random.default_rng(5)
    ra = np.zeros((N, m, k), np.float16)
    rb = np.zeros((N, n, k), np.float16)
    for l, p in enumerate(mods):
        lo, hi = -(p // 2), (p + 1) // 2 - 1
        ra[l] = rng.choice([lo, hi], size=(m, k))
        rb[l] = rng.choice([lo, hi], size=(n, k))
    RA, RB = dev(ra), dev(rb)
    c = os2.gemm_residues(RA, RB, k, os2.OUT_MODP_INT8, os2.GEMM_TC).cpu().numpy()[:, :, :n]
    c1 = os2.gemm_residues(RA, RB, k, os2.OUT_MODP_INT8, os2.GEMM_TC_1SM).cpu().numpy()[:, :, :n]
    c8 = _step3(RA, RB, k, os2.OUT_MODP_INT8, os2.GEMM_S8_SYNC).cpu().numpy()[:, :, :n]
    status_ok()
    assert np.array_equal(c, c1)
    assert np.array_equal(c, c8)
    G = np.einsum("lik,ljk->lij", ra.astype(np.int64), rb.astype(np.int64))
    for l, p in enumerate(mods):
        r = np.mod(G[l], p)
        r = np.where(r >= (p + 1) // 2, r - p, r)
        assert np.array_equal(c[l].astype(np.int64), r)


# --------------------------------------------------------------- steps 4-5 --
@pytest.mark.parametrize("N", [1, 2, 4, 5, 8, 9, 12, 13, 14, 16, 17, 20])
def test_crt_parity_from_oracle_residues(N, crt_variant):
    A, Bt = workloads.make_pair("spread", 37, 45, 90, seed=N, phi=2.0)
    ref = orc.gemm_entries(A, Bt, N)
    cres = np.zeros((N, 37, 48), np.int8)
    cres[:, :, :45] = np.transpose(ref.c, (2, 0, 1))
    C, X = os2.crt(dev(cres), 45, dev(ref.e), dev(ref.f), want_X=True)
    status_ok()
    assert np.array_equal(X.cpu().numpy().view(np.uint32), ref.X)
    assert_bits_equal(C.cpu().numpy(), ref.C, "C")


@pytest.mark.parametrize("ldcres", [48, 52, 45])
def test_crt_unaligned_rows_fall_back(ldcres):
    """Rows of c that are not 16-byte multiples take the CUDA-core kernel
    (the tensor-core one reads 16-byte vectors): same bits."""
    N, m, n = 16, 21, 45
    A, Bt = workloads.make_pair("spread", m, n, 70, seed=ldcres, phi=2.0)
    ref = orc.gemm_entries(A, Bt, N)
    cres = np.zeros((N, m, ldcres), np.int8)
    cres[:, :, :n] = np.transpose(ref.c, (2, 0, 1))
    if ldcres % 4:
        with pytest.raises(os2.Os2Error):
            os2.crt(dev(cres), n, dev(ref.e), dev(ref.f))
        return
    C = os2.crt(dev(cres), n, dev(ref.e), dev(ref.f))
    status_ok()
    assert_bits_equal(C.cpu().numpy(), ref.C, f"ldcres={ldcres}")


@pytest.mark.parametrize("N", [1, 2])
def test_crt_exhaustive_small_moduli_sets(N, crt_variant):
    """Every residue vector for N = 1 (256 values) and N = 2 (256 x 255):
    X is the unique value in [-P/2, P/2) with those residues (brute force),
    including X = -P/2 itself; with e = f = 0 the result is X exactly."""
    mods = os2.moduli(N)
    P = int(np.prod(mods))
    grids = np.meshgrid(*[np.arange(-(p // 2), (p + 1) // 2) for p in mods], indexing="ij")
    res = np.stack([g.reshape(-1) for g in grids])          # N x P residue vectors
    vals = np.arange(-P // 2, P // 2)                          # brute force: residues of each X
    sym = np.stack([((vals + p // 2) % p) - p // 2 for p in mods])
    lookup = {tuple(col): int(x) for col, x in zip(sym.T, vals)}
    expect = np.array([lookup[tuple(col)] for col in res.T], dtype=np.float64)
    n = 256
    m = P // n
    cres = np.zeros((N, m, n), np.int8)
    cres[:, :, :] = res.reshape(N, m, n)
    C = os2.crt(dev(cres), n, dev(np.zeros(m, np.int32)), dev(np.zeros(n, np.int32)))
    status_ok()
    assert np.array_equal(C.cpu().numpy().reshape(-1), expect)


def test_crt_random_residues_and_rounding(crt_variant):
    """Arbitrary residue vectors (X anywhere in [-P/2, P/2)) and exponents that
    push the result into the subnormal and overflow ranges."""
    rng = np.random.default_rng(2)
    for N in (1, 3, 4, 5, 8, 9, 12, 13, 16, 17, 20):
        mods = os2.moduli(N)
        m, n = 33, 65
        cres = np.zeros((N, m, 80), np.int8)
        for l, p in enumerate(mods):
            cres[l, :, :n] = rng.integers(-(p // 2), (p + 1) // 2, size=(m, n))
        e = rng.integers(-1300, 1300, size=m).astype(np.int32)
        f = rng.integers(-700, 700, size=n).astype(np.int32)
        C, X = os2.crt(dev(cres), n, dev(e), dev(f), want_X=True)
        status_ok()
        Xn = X.cpu().numpy().view(np.uint32)
        Cn = C.cpu().numpy()
        P = int(np.prod([int(p) for p in mods], dtype=object))
        for i in range(0, m, 4):
            for j in range(0, n, 3):
                res = [int(cres[l, i, j]) for l in range(N)]
                x = orc.crt_small(res, mods) if P < 2 ** 62 else None
                xv = orc.limbs_to_int(Xn[i, j])
                assert -P // 2 <= xv < P // 2 + (P % 2)
                for l, p in enumerate(mods):
                    assert (xv - res[l]) % p == 0
                if x is not None:
                    assert xv == (x - P if x >= (P + 1) // 2 else x)
                want = orc.round_scaled(xv, int(e[i]) + int(f[j]))
                assert Cn[i, j] == want or (np.isinf(Cn[i, j]) and np.isinf(want))
                assert np.signbit(Cn[i, j]) == np.signbit(want)


# ------------------------------------------------------------- end to end --
@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("m,n,k", SHAPES)
def test_gemm_end_to_end_small(mode, m, n, k, crt_variant):
    N = 14
    A, Bt = workloads.make_pair("spread", m, n, k, seed=k, phi=1.0)
    C = os2.gemm(dev(A), dev(Bt), N, mode).cpu().numpy()
    status_ok()
    ref = orc.gemm_entries(A, Bt, N, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0
    assert_bits_equal(C, ref.C, f"{mode} {m}x{n}x{k}")
    check_tolerance(C, A, Bt, np.arange(m), np.arange(n), ref.C)


def test_gemm_64cube_normal_config():
    """64^3, N(0,1) from seed 0, 14 moduli, fast mode: every entry."""
    A, Bt = workloads.make_pair("normal", 64, 64, 64, seed=0)
    C = os2.gemm(dev(A), dev(Bt), 14, "fast").cpu().numpy()
    status_ok()
    ref = orc.gemm_entries(A, Bt, 14)
    assert_bits_equal(C, ref.C, "64^3")


@pytest.mark.parametrize("variant", [os2.GEMM_SIMT, os2.GEMM_TC_1SM, os2.GEMM_TC_I8,
                                     os2.GEMM_S8_SYNC])
def test_gemm_variants_end_to_end(variant):
    A, Bt = workloads.make_pair("spread", 150, 170, 400, seed=1, phi=2.0)
    try:
        os2.set_gemm_variant(variant)
        Cs = os2.gemm(dev(A), dev(Bt), 16).cpu().numpy()
    finally:
        os2.set_gemm_variant(os2.GEMM_TC)
    Ct = os2.gemm(dev(A), dev(Bt), 16).cpu().numpy()
    status_ok()
    assert_bits_equal(Cs, Ct, "variant vs default tc")
    ref = orc.gemm_entries(A, Bt, 16, want_X=False, want_c=False, want_G=False)
    assert_bits_equal(Ct, ref.C, "tc vs oracle")


@pytest.mark.parametrize("variant", [os2.GEMM_TC_I8, os2.GEMM_S8_SYNC])
@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("m,n,k,N", [(4100, 300, 700, 16), (257, 513, 1921, 20), (3, 5, 7, 2),
                                     (300, 260, 9000, 14), (64, 48, 70000, 16)])
def test_int8_plane_variant_oracle(variant, mode, m, n, k, N):
    """The int8-plane variants (step 2 writes int8 residue planes; step 3
    widens them to FP16 on chip, or multiplies them with mma.sync s8):
    bit-exact against the oracle on a sample, with row panels (m >= 4096),
    ragged tiles, long k (several reduction chunks; k = 70000 crosses the
    65536-term reduction of the mma.sync kernel) and the host entry point's
    column panels."""
    A, Bt = workloads.make_pair("spread", m, n, k, seed=m + k, phi=2.0)
    try:
        os2.set_gemm_variant(variant)
        C = os2.gemm(dev(A), dev(Bt), N, mode).cpu().numpy()
        status_ok()
        Ch = torch.full((m, n), np.nan, dtype=torch.float64).pin_memory()
        os2.gemm_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(Bt).pin_memory(), Ch, N,
                      mode)
        torch.cuda.current_stream().synchronize()
        status_ok()
    finally:
        os2.set_gemm_variant(os2.GEMM_TC)
    rows, cols = workloads.sample_grid(m, n, 40, seed=4)
    ref = orc.gemm_entries(A, Bt, N, rows, cols, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0
    assert_bits_equal(C[np.ix_(rows, cols)], ref.C, f"int8 planes {m}x{n}x{k} N={N} {mode}")
    assert_bits_equal(Ch.numpy(), C, "int8 planes, host entry point vs device")


def test_integer_inputs_exact_on_gpu():
    A, Bt = workloads.make_pair("int", 200, 300, 500, seed=4, phi=1000)
    for mode in ("fast", "accurate"):
        C = os2.gemm(dev(A), dev(Bt), 14, mode).cpu().numpy()
        status_ok()
        assert np.array_equal(C, A @ Bt.T)


def test_edge_cases():
    # k = 0 -> zeros; m or n = 0 -> nothing
    A = torch.zeros((5, 0), dtype=torch.float64, device=DEV)
    Bt = torch.zeros((3, 0), dtype=torch.float64, device=DEV)
    C = torch.full((5, 3), 7.0, dtype=torch.float64, device=DEV)
    os2.gemm(A, Bt, 14, out=C)
    assert torch.all(C == 0)
    os2.gemm(torch.zeros((0, 4), dtype=torch.float64, device=DEV),
             torch.ones((3, 4), dtype=torch.float64, device=DEV), 14)
    # zero rows / columns, subnormals, huge magnitudes, leading dimensions > k
    rng = np.random.default_rng(8)
    Abig = rng.standard_normal((70, 100))
    Bbig = rng.standard_normal((90, 100))
    Abig[3] = 0.0
    Bbig[:, 7] = 0.0
    Bbig[5] = 0.0
    Abig[10] *= 2.0 ** -1060
    Abig[11] *= 2.0 ** 900
    Bbig[12] *= 2.0 ** 120
    At = dev(Abig)[:, :77]
    Btt = dev(Bbig)[:, :77]
    for mode, om in (("fast", orc.FAST), ("accurate", orc.ACCURATE)):
        Cg = os2.gemm(At, Btt, 16, mode).cpu().numpy()
        status_ok()
        ref = orc.gemm_entries(np.ascontiguousarray(Abig[:, :77]), np.ascontiguousarray(Bbig[:, :77]),
                               16, mode=om, want_X=False, want_c=False, want_G=False)
        assert_bits_equal(Cg, ref.C, f"edge {mode}")


@pytest.mark.parametrize("k", [1, 511, 1023, 1025, 2049, 4095, 8191, 8192, 8193])
def test_odd_leading_dimensions(k):
    """Rows that start off the 16-byte boundary (odd leading dimensions) take the
    scalar-load paths of the scaling and residue kernels; k spans the sizes at
    which the fast scaling holds a row in registers and the two-pass fallback."""
    rng = np.random.default_rng(k)
    m, n = 37, 29
    Abig = rng.standard_normal((m, k + 1)) * np.exp2(rng.integers(-20, 20, size=(m, k + 1)))
    Bbig = rng.standard_normal((n, k + 3))
    A, Bt = Abig[:, :k], Bbig[:, :k]
    for mode, om in (("fast", orc.FAST), ("accurate", orc.ACCURATE)):
        Cg = os2.gemm(dev(Abig)[:, :k], dev(Bbig)[:, :k], 14, mode).cpu().numpy()
        status_ok()
        ref = orc.gemm_entries(np.ascontiguousarray(A), np.ascontiguousarray(Bt), 14, mode=om,
                               want_X=False, want_c=False, want_G=False)
        assert ref.mismatches == 0
        assert_bits_equal(Cg, ref.C, f"odd ld, k={k}, {mode}")
    e, f = os2.scale(dev(Abig)[:, :k], dev(Bbig)[:, :k], 14, "fast")
    assert np.array_equal(e.cpu().numpy(), orc.scale_fast(np.ascontiguousarray(A), 14))
    assert np.array_equal(f.cpu().numpy(), orc.scale_fast(np.ascontiguousarray(Bt), 14))


def test_nonfinite_input_sets_status():
    A, Bt = workloads.make_pair("normal", 40, 40, 40)
    A[3, 4] = np.nan
    os2.gemm(dev(A), dev(Bt), 14)
    assert os2.get_status() == os2.binding.ERR_NONFINITE
    assert os2.get_status() == 0        # cleared
    Bt[1, 1] = -np.inf
    A[3, 4] = 1.0
    os2.gemm(dev(A), dev(Bt), 14, "accurate")
    assert os2.get_status() == os2.binding.ERR_NONFINITE


@pytest.mark.parametrize("s", [-200, -100, -50, 50, 100, 200])
def test_scale_invariance_on_gpu(s):
    """[G] Methodik 2: A * 2^s gives C * 2^s exactly, in both modes; also with
    B scaled (C * 2^2s)."""
    A, Bt = workloads.make_pair("normal", 256, 192, 512, seed=0)
    for mode in ("fast", "accurate"):
        C0 = os2.gemm(dev(A), dev(Bt), 16, mode).cpu().numpy()
        Cs = os2.gemm(dev(np.ldexp(A, s)), dev(Bt), 16, mode).cpu().numpy()
        Css = os2.gemm(dev(np.ldexp(A, s)), dev(np.ldexp(Bt, s)), 16, mode).cpu().numpy()
        status_ok()
        assert_bits_equal(Cs, np.ldexp(C0, s), f"A*2^{s}")
        assert_bits_equal(Css, np.ldexp(C0, 2 * s), f"A,B*2^{s}")


@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("m,n,k,pinned", [(100, 120, 300, True), (1001, 700, 513, True),
                                          (3, 2, 5, False), (5000, 300, 200, True),
                                          (9000, 72, 96, True), (4100, 33, 40, False),
                                          (5, 4, 0, True)])
def test_host_entry_point_matches_device(mode, m, n, k, pinned):
    """The end-to-end host entry point (B in, then A in row panels that are
    scaled, split, multiplied and reconstructed while later panels are still in
    transit, C out by panels) equals the device one.  m >= 4096 gives several
    panels, the last one ragged."""
    A, Bt = workloads.make_pair("spread", m, n, k, seed=6, phi=2.0)
    Ah = torch.from_numpy(A)
    Bh = torch.from_numpy(Bt)
    Ch = torch.full((m, n), np.nan, dtype=torch.float64)
    if pinned:
        Ah, Bh, Ch = Ah.pin_memory(), Bh.pin_memory(), Ch.pin_memory()
    os2.gemm_host(Ah, Bh, Ch, 14, mode)
    torch.cuda.current_stream().synchronize()
    status_ok()
    Cd = os2.gemm(dev(A), dev(Bt), 14, mode).cpu().numpy()
    assert_bits_equal(Ch.numpy(), Cd, "host vs device entry")


@pytest.mark.parametrize("mode", ["fast", "accurate"])
def test_host_entry_point_oracle_sample(mode, crt_variant):
    """The host entry point checked against the oracle directly (not only
    against os2_gemm): several row and column panels, ragged edges, a seeded
    48 x 48 sample with the last row and column."""
    m, n, k = 4700, 4400, 200
    A, Bt = workloads.make_pair("spread", m, n, k, seed=31, phi=2.0)
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(Bt).pin_memory()
    Ch = torch.full((m, n), np.nan, dtype=torch.float64).pin_memory()
    os2.gemm_host(Ah, Bh, Ch, 16, mode)
    torch.cuda.current_stream().synchronize()
    status_ok()
    rows, cols = workloads.sample_grid(m, n, 48, seed=7)
    ref = orc.gemm_entries(A, Bt, 16, rows, cols, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0
    assert_bits_equal(Ch.numpy()[np.ix_(rows, cols)], ref.C, f"host entry point {mode}")


def test_host_entry_point_strided_back_to_back():
    """Row strides on all three host matrices, a side stream, and two calls in
    a row on one workspace with one synchronisation at the end: the second
    call's copies in wait for the first call's kernels."""
    m, n, k = 4700, 260, 150
    A1, B1 = workloads.make_pair("spread", m, n, k, seed=11, phi=1.0)
    A2, B2 = workloads.make_pair("normal", m, n, k, seed=12)
    big = lambda r, c: torch.full((r, c), np.nan, dtype=torch.float64).pin_memory()
    Ah1, Bh1, Ah2, Bh2 = big(m, k + 9), big(n, k + 3), big(m, k + 9), big(n, k + 3)
    Ah1[:, :k] = torch.from_numpy(A1)
    Bh1[:, :k] = torch.from_numpy(B1)
    Ah2[:, :k] = torch.from_numpy(A2)
    Bh2[:, :k] = torch.from_numpy(B2)
    Ch1, Ch2 = big(m, n + 5), big(m, n + 5)
    ws = os2.alloc_workspace(os2.host_workspace_size(m, n, k, 16, "fast"))
    side = torch.cuda.Stream()
    os2.gemm_host(Ah1[:, :k], Bh1[:, :k], Ch1[:, :n], 16, "fast", workspace=ws, stream=side)
    os2.gemm_host(Ah2[:, :k], Bh2[:, :k], Ch2[:, :n], 16, "fast", workspace=ws, stream=side)
    side.synchronize()
    status_ok()
    for A, Bt, Ch in ((A1, B1, Ch1), (A2, B2, Ch2)):
        Cd = os2.gemm(dev(A), dev(Bt), 16, "fast").cpu().numpy()
        assert_bits_equal(Ch[:, :n].numpy(), Cd, "host vs device entry")
        assert torch.isnan(Ch[:, n:]).all(), "wrote past the row of C"


# ----------------------------------------------------- inner dimension >= 2^17 --
@pytest.mark.parametrize("N,m,n,k", [(16, 24, 20, 140001), (20, 8, 9, 300000), (12, 130, 5, 131073)])
def test_large_k_fast_parity(N, m, n, k):
    """[Q] 手順3: beyond 2^17 the products are split into blocks; here every
    960-term block is reduced mod p in tensor memory, so k may exceed 2^17."""
    A, Bt = workloads.make_pair("spread", m, n, k, seed=k % 97, phi=1.0)
    C = os2.gemm(dev(A), dev(Bt), N, "fast").cpu().numpy()
    status_ok()
    ref = orc.gemm_entries(A, Bt, N, want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0
    assert_bits_equal(C, ref.C, f"k={k}")


def test_large_k_accurate_parity():
    A, Bt = workloads.make_pair("spread", 10, 12, 200003, seed=3, phi=2.0)
    C = os2.gemm(dev(A), dev(Bt), 16, "accurate").cpu().numpy()
    status_ok()
    ref = orc.gemm_entries(A, Bt, 16, mode=orc.ACCURATE, want_X=False, want_c=False, want_G=False)
    assert_bits_equal(C, ref.C, "accurate, k=200003")


def test_large_k_all_ones_128bit_sums():
    """All-ones rows with k > 2^20: the fast-mode sum of squares exceeds 2^64
    (128-bit path); C = k exactly and the exponents match the oracle."""
    k = (1 << 20) + 5
    A = np.ones((4, k))
    Bt = np.ones((3, k))
    e, f = os2.scale(dev(A), dev(Bt), 16, "fast")
    assert np.array_equal(e.cpu().numpy(), orc.scale_fast(A, 16))
    C = os2.gemm(dev(A), dev(Bt), 16, "fast")
    status_ok()
    assert torch.all(C == k)


def test_modp_products_far_beyond_int32():
    """All residues -128 with k = 2^20: G = 2^14 k overflows int32, but the
    blocked mod-p accumulation gives (2^14 k) mod p exactly."""
    N, m, n, k = 5, 128, 256, 1 << 20
    RA = torch.full((N, m, k), -128.0, dtype=torch.float16, device=DEV)
    RB = torch.full((N, n, k), -128.0, dtype=torch.float16, device=DEV)
    for variant in (os2.GEMM_TC, os2.GEMM_TC_1SM, os2.GEMM_S8_SYNC):
        c = _step3(RA, RB, k, os2.OUT_MODP_INT8, variant).cpu().numpy()[:, :, :n]
        status_ok()
        for l, p in enumerate(os2.moduli(N)):
            r = (16384 * k) % p
            r = r - p if r >= (p + 1) // 2 else r
            assert np.all(c[l] == r), (variant, p)


# ------------------------------------------------------------ SGEMM emulation --
def _f32_bits_equal(got, want, what):
    got = np.ascontiguousarray(got, np.float32)
    want = np.ascontiguousarray(want, np.float32)
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, f"{what}: {bad.size} entries differ, first {bad[:5]}"


@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("N,m,n,k", [(7, 64, 64, 64), (4, 129, 257, 65), (8, 300, 200, 1000),
                                     (10, 130, 140, 1921), (14, 33, 65, 3000), (18, 70, 90, 200),
                                     (20, 64, 48, 100)])
def test_sgemm_parity(mode, N, m, n, k):
    """SGEMM emulation ([G] Ergebnisse): float operands, binary32 result,
    bit-exact against the oracle rounding the same CRT integer to binary32.
    At 18 and 20 moduli the scaled integers exceed 2^59, so step 2 takes its
    five- and six-word paths on float input."""
    A, Bt = workloads.make_pair("spread", m, n, k, seed=N + k, phi=1.0)
    A = A.astype(np.float32)
    Bt = Bt.astype(np.float32)
    C = os2.sgemm(dev(A), dev(Bt), N, mode).cpu().numpy()
    status_ok()
    ref = orc.gemm_entries(A, Bt, N, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False, out_f32=True)
    assert ref.mismatches == 0
    _f32_bits_equal(C, ref.C, f"sgemm {mode} N={N} {m}x{n}x{k}")


def test_sgemm_edge_values():
    rng = np.random.default_rng(4)
    A = rng.standard_normal((40, 96)).astype(np.float32)
    Bt = rng.standard_normal((50, 96)).astype(np.float32)
    A[0] = 0
    A[1, ::2] = np.float32(1e-45)          # float subnormals
    A[2] *= np.float32(1e37)
    Bt[3] *= np.float32(1e-30)
    Bt[4, 5] = np.float32(3e38)
    for mode, om in (("fast", orc.FAST), ("accurate", orc.ACCURATE)):
        C = os2.sgemm(dev(A), dev(Bt), 8, mode).cpu().numpy()
        status_ok()
        ref = orc.gemm_entries(A, Bt, 8, mode=om, want_X=False, want_c=False, want_G=False,
                               out_f32=True)
        _f32_bits_equal(C, ref.C, f"sgemm edges {mode}")


def test_sgemm_4096cube_sample():
    A, Bt = workloads.make_pair("spread", 4096, 4096, 4096, seed=0, phi=0.5)
    A = A.astype(np.float32)
    Bt = Bt.astype(np.float32)
    C = os2.sgemm(dev(A), dev(Bt), 7, "fast")
    status_ok()
    rows, cols = workloads.sample_grid(4096, 4096, 32, seed=1)
    ref = orc.gemm_entries(A, Bt, 7, rows, cols, want_X=False, want_c=False, want_G=False,
                           out_f32=True)
    got = C.cpu().numpy()[np.ix_(rows, cols)]
    _f32_bits_equal(got, ref.C, "sgemm 4096^3 sample")


# ------------------------------------------------------------- ZGEMM / CGEMM --
@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (64, 64, 64), (129, 65, 100), (200, 150, 700)])
def test_complex_parity(single, mode, m, n, k):
    """[G] Bedeutung: ZGEMM/CGEMM through the real block form, bit-exact
    against the oracle of the same block form."""
    A, Bt = workloads.make_pair("spread", m, n, k, seed=k, phi=1.0)        # real parts
    Ai, Bi = workloads.make_pair("spread", m, n, k, seed=k + 1, phi=1.0)  # imaginary parts
    Z = (A + 1j * Ai).astype(np.complex64 if single else np.complex128)
    W = (Bt + 1j * Bi).astype(np.complex64 if single else np.complex128)
    N = 8 if single else 16
    C = os2.zgemm(dev(Z), dev(W), N, mode).cpu().numpy()
    status_ok()
    ref, r = orc.complex_gemm_entries(Z, W, N, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                                      single=single)
    assert r.mismatches == 0
    assert np.array_equal(C.view(np.uint32 if single else np.uint64),
                          ref.view(np.uint32 if single else np.uint64))


def test_zgemm_integer_inputs_exact_on_gpu():
    rng = np.random.default_rng(9)
    Z = rng.integers(-99, 100, (70, 90)) + 1j * rng.integers(-99, 100, (70, 90))
    W = rng.integers(-99, 100, (50, 90)) + 1j * rng.integers(-99, 100, (50, 90))
    C = os2.zgemm(dev(Z.astype(np.complex128)), dev(W.astype(np.complex128)), 14).cpu().numpy()
    status_ok()
    assert np.array_equal(C, Z @ W.T)


# ------------------------------------------------------- row-panel pipeline --
def test_row_panels_equal_unpanelled_rows():
    """m >= 4096 runs A in row panels with the CRT on a side stream.  Fast-mode
    exponents depend on one row or one column only, so the panelled product
    equals, entry for entry, two calls on halves of A (each a single panel)."""
    A, Bt = workloads.make_pair("spread", 4100, 520, 300, seed=21, phi=1.5)
    C = os2.gemm(dev(A), dev(Bt), 16, "fast").cpu().numpy()
    status_ok()
    top = os2.gemm(dev(A[:2050]), dev(Bt), 16, "fast").cpu().numpy()
    bot = os2.gemm(dev(A[2050:]), dev(Bt), 16, "fast").cpu().numpy()
    status_ok()
    assert_bits_equal(C, np.vstack([top, bot]), "panelled vs halves")


@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("m", [4100, 9000])
def test_row_panels_oracle_sample(mode, m, crt_variant):
    """Ragged last panel (4100 = 2304 + 1796; 9000 = 3 x 2304 + 2088), both
    modes, a seeded 40 x 40 sample (always with the last row and column)
    bit-exact against the oracle."""
    n, k = 200, 160
    A, Bt = workloads.make_pair("spread", m, n, k, seed=m, phi=2.0)
    C = os2.gemm(dev(A), dev(Bt), 14, mode).cpu().numpy()
    status_ok()
    rows, cols = workloads.sample_grid(m, n, 40, seed=3)
    ref = orc.gemm_entries(A, Bt, 14, rows, cols, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    assert ref.mismatches == 0
    assert_bits_equal(C[np.ix_(rows, cols)], ref.C, f"panels m={m} {mode}")


def test_row_panels_sgemm_and_zgemm_sample():
    """SGEMM and ZGEMM emulation also take the row-panel path for m >= 4096."""
    m, n, k = 4100, 96, 130
    A, Bt = workloads.make_pair("spread", m, n, k, seed=5, phi=1.0)
    A32, B32 = A.astype(np.float32), Bt.astype(np.float32)
    C = os2.sgemm(dev(A32), dev(B32), 7, "fast").cpu().numpy()
    status_ok()
    rows, cols = workloads.sample_grid(m, n, 32, seed=4)
    ref = orc.gemm_entries(A32, B32, 7, rows, cols, want_X=False, want_c=False, want_G=False,
                           out_f32=True)
    _f32_bits_equal(C[np.ix_(rows, cols)], ref.C, "sgemm panels")
    Ai, Bi = workloads.make_pair("spread", m, n, k, seed=6, phi=1.0)
    Z, W = A + 1j * Ai, Bt + 1j * Bi
    Cz = os2.zgemm(dev(Z), dev(W), 16, "fast").cpu().numpy()
    status_ok()
    refz, r = orc.complex_gemm_entries(Z, W, 16, rows, cols)
    assert r.mismatches == 0
    assert np.array_equal(Cz[np.ix_(rows, cols)].view(np.uint64), refz.view(np.uint64))


@pytest.mark.parametrize("N,k", [(16, 4096), (16, 4097), (16, 9000), (2, 9000)])
def test_accurate_bound_segments(N, k):
    """Accurate mode's bound product runs in 4096-term segments on the 2-SM
    kernel (int32 partial sums between segments, ragged n); os2_scale, whose
    own workspace has no room for the partial sums, takes the single-SM kernel
    for more than one segment.  Both give the oracle's exponents, and the
    product is bit-exact.  With N = 2 the product-residue region is too small
    for the partial sums, so os2_gemm falls back to the single-SM kernel too."""
    m, n = 300, 70
    A, Bt = workloads.make_pair("spread", m, n, k, seed=k, phi=2.0)
    e_ref, f_ref = orc.scale_accu(A, Bt, N)
    e, f = os2.scale(dev(A), dev(Bt), N, "accurate")
    status_ok()
    assert np.array_equal(e.cpu().numpy(), e_ref)
    assert np.array_equal(f.cpu().numpy(), f_ref)
    C = os2.gemm(dev(A), dev(Bt), N, "accurate").cpu().numpy()
    status_ok()
    rows, cols = workloads.sample_grid(m, n, 24, seed=2)
    ref = orc.gemm_entries(A, Bt, N, rows, cols, mode=orc.ACCURATE, want_X=False, want_c=False,
                           want_G=False)
    assert_bits_equal(C[np.ix_(rows, cols)], ref.C, f"accurate k={k}")


@pytest.mark.parametrize("m,n,k", [(70000, 20, 40), (3, 70000, 40)])
def test_tall_and_wide_shapes(m, n, k, crt_variant):
    """More than 65535 rows of A or columns of B: the residue and CRT grids cap
    their y dimension and loop, and m = 70000 runs the most row panels (8)."""
    A, Bt = workloads.make_pair("spread", m, n, k, seed=m + n, phi=1.0)
    for mode, om in (("fast", orc.FAST), ("accurate", orc.ACCURATE)):
        C = os2.gemm(dev(A), dev(Bt), 14, mode).cpu().numpy()
        status_ok()
        rows, cols = workloads.sample_grid(m, n, 16, seed=5)
        ref = orc.gemm_entries(A, Bt, 14, rows, cols, mode=om, want_X=False, want_c=False,
                               want_G=False)
        assert ref.mismatches == 0
        assert_bits_equal(C[np.ix_(rows, cols)], ref.C, f"{m}x{n}x{k} {mode}")
