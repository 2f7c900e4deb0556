"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each test names the passage it follows.  Pages:
  [Q] Qiita, "8ビットの整数で53ビットの倍精度を組み立てる。中国剰余定理をGPUに載せた
      Ozaki Scheme II"
  [G] gist.science, "Improved Scaling for Fast Mode of Ozaki Scheme II"
"""
import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import bigref
from oracle import oracle as orc

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as fh:
        return json.load(fh)


# ---------------------------------------------------------------- CRT -------
def test_sunzi_example():
    """[Q] 孫子算経からガウスまで / 繰り上がりのない計算: residues 2,3,2 mod 3,5,7."""
    g = gold("sunzi.json")
    assert orc.crt_small(g["residues"], g["moduli"]) == g["answer"]
    P, M, odd, inv, W = bigref.crt_constants(g["moduli"])
    assert P == g["product"] and W == g["use_numbers"]
    s = sum(r * w for r, w in zip(g["residues"], W))
    assert s == g["weighted_sum"]
    assert s - g["turns_removed"] * P == g["answer"]
    # each use number advances exactly one clock by one tick
    for l, w in enumerate(W):
        assert [w % p for p in g["moduli"]] == [1 if i == l else 0 for i in range(3)]


def test_dayan_table_and_walk():
    """[Q] 秦九韶の大衍求一術: the table and the 2x2-grid walk that gives 70."""
    g = gold("dayan.json")
    P, M, odd, inv, W = bigref.crt_constants(g["dingmu_moduli"])
    assert P == g["yanmu_product"]
    assert M == g["yanshu_cofactors"]
    assert odd == g["jishu_cofactor_mod_p"]
    assert inv == g["chenglv_inverses"]
    assert W == g["yongshu_use_numbers"]
    for o, p, i in zip(odd, g["dingmu_moduli"], g["chenglv_inverses"]):
        assert orc.dayan_qiuyi(o, p) == i
        assert orc.inverse_bruteforce(o, p) == i
    w = g["walk_for_70"]
    assert orc.dayan_qiuyi(w["jishu"], w["dingmu"]) == w["chenglv"]
    assert 35 * w["chenglv"] == w["use_number"]


def test_dayan_is_extended_euclid_exhaustive():
    """The grid procedure computes the modular inverse for every coprime pair."""
    for p in range(2, 260):
        for a in range(1, p):
            got = orc.dayan_qiuyi(a, p)
            if math.gcd(a, p) == 1:
                assert got == pow(a, -1, p), (a, p)
                assert orc.inverse_bruteforce(a, p) == got
            else:
                assert got == 0 and orc.inverse_bruteforce(a, p) == 0


def test_crt_small_bruteforce():
    """CRT inverts residues for every integer below the product (clock picture)."""
    mods = [4, 9, 5, 7]
    P = math.prod(mods)
    for x in range(P):
        assert orc.crt_small([x % p for p in mods], mods) == x


# ------------------------------------------------------------- moduli -------
def test_moduli_sets_and_ranges():
    """[Q] 256以下の法の選び方(手順2) + footnote 6."""
    g = gold("moduli.json")
    table = orc.moduli(20)
    assert table == g["table_20"]
    assert bigref.greedy_moduli(20) == g["table_20"]          # greedy from 256 down
    for N in range(1, 21):
        assert orc.moduli(N) == table[:N]
    for a in range(20):
        for b in range(a):
            assert math.gcd(table[a], table[b]) == 1
    assert round(math.log2(math.prod(table[:16])), 1) == g["table_16_log2_range_approx"]
    assert round(math.log2(math.prod(g["paper_16"]))) == g["paper_16_log2_range_approx"]
    primes = [x for x in range(g["primes_only_16_from"], g["primes_only_16_to"] - 1, -1)
              if all(x % d for d in range(2, int(x ** 0.5) + 1))]
    assert len(primes) == 16
    assert round(math.log2(math.prod(primes))) == g["primes_only_16_log2_range_approx"]
    # composites are allowed: only coprimality matters
    for x, fac in g["composite_factorisations"].items():
        assert math.prod(fac) == int(x)
    # 256 is the only even modulus
    assert sum(1 for x in table if x % 2 == 0) == 1
    # int32 exactness bound of step 3
    assert 128 * 128 == g["max_abs_product"]
    assert (g["inner_dim_limit"] - 1) * g["max_abs_product"] < 2 ** 31
    assert g["inner_dim_limit"] * g["max_abs_product"] == 2 ** 31


@pytest.mark.parametrize("N", [1, 2, 7, 12, 14, 16, 18, 20])
def test_oracle_tables_match_definition(N):
    P, H, W, inv = orc.tables(N)
    mods = orc.moduli(N)
    assert P == math.prod(mods)
    assert H == (P - 1) // 2
    for l, p in enumerate(mods):
        M = P // p
        assert (M * inv[l]) % p == 1
        assert W[l] == M * inv[l]
        for q in mods:
            assert W[l] % q == (1 if q == p else 0)


def test_symmetric_residues_exhaustive():
    """[Q] 手順2: residues in [-128, 127]; mod 256 is the low byte."""
    mods = orc.moduli(20)
    x = np.arange(-40000, 40000, dtype=np.int64)
    low_byte = x.astype(np.int8)
    assert np.array_equal(np.array([bigref.sym(int(v), 256) for v in x]), low_byte)
    xs = x[37000:43000]
    for p in mods:
        r = np.array([bigref.sym(int(v), p) for v in xs])
        assert r.min() >= -128 and r.max() <= 127
        assert np.all((r - xs) % p == 0)
        if p % 2:
            assert r.min() == -(p - 1) // 2 and r.max() == (p - 1) // 2


def test_oracle_residues_match_python():
    A, _ = workloads.make_pair("spread", 7, 1, 33, seed=3, phi=4.0)
    e = orc.scale_fast(A, 20)
    res = orc.residues(A, e, 20)
    ints = orc.integers(A, e)
    mods = orc.moduli(20)
    for l, p in enumerate(mods):
        for i in range(7):
            for h in range(33):
                assert res[l, i, h] == bigref.sym(int(ints[i, h]), p)
    # integers are the exact truncations
    for i in range(7):
        for h in range(33):
            assert ints[i, h] == bigref.trunc_scaled(float(A[i, h]), int(e[i]))


def test_oracle_residues_of_wide_integers():
    """Residues of integers up to just below 2^89 (the widest the GPU tests
    give the residue step) against Python's exact truncation and modulo."""
    rng = np.random.default_rng(12)
    X = rng.standard_normal((5, 16))
    X[1, 3] = -X[1, 3]
    E = int(np.frexp(np.abs(X).max())[1])          # |x| < 2^E
    mods = orc.moduli(20)
    for e_val in (59 - E, 60 - E, 74 - E, 75 - E, 88 - E, 89 - E):
        e = np.full(5, e_val, np.int32)
        res = orc.residues(X, e, 20)
        for i in range(5):
            for h in range(16):
                a = bigref.trunc_scaled(float(X[i, h]), e_val)
                assert abs(a) < 2 ** 89
                for l, p in enumerate(mods):
                    assert res[l, i, h] == bigref.sym(a, p), (e_val, i, h, p)


# ------------------------------------------------------------ scaling -------
def _exact_sq(row):
    return sum(Fraction(x) ** 2 for x in row)


@pytest.mark.parametrize("N", [2, 6, 12, 14, 16, 20])
@pytest.mark.parametrize("kind,phi", [("normal", 0.0), ("spread", 4.0)])
def test_fast_scaling_meets_sufficient_condition_and_is_maximal(N, kind, phi):
    """[G] Methodik 1: 2 mu_i ||a_i|| ||b_j|| nu_j <= P - 1, and mu_i is the
    page's 2^floor(P' - 0.5 log2 sum a^2) up to the slack of the upper bound."""
    A, Bt = workloads.make_pair(kind, 9, 8, 40, seed=N, phi=phi)
    P, H, _, _ = orc.tables(N)
    e, Q = orc.scale_fast(A, N, return_Q=True)
    f = orc.scale_fast(Bt, N)
    for i in range(9):
        sa = _exact_sq(A[i])
        E = max(math.frexp(float(x))[1] for x in A[i] if x != 0)
        S_up = Fraction(int(Q[i])) * Fraction(4) ** (E - 23)
        assert S_up >= sa                                       # an upper bound
        ei = int(e[i])
        assert Fraction(4) ** ei * S_up <= H                    # the chosen mu fits
        assert Fraction(4) ** (ei + 1) * S_up > H               # and is the largest that does
        # the page's formula with an exact log2: largest e with 4^e sum a^2 <= (P-1)/2
        e_exact = 0
        while Fraction(4) ** (e_exact + 1) * sa <= Fraction(P - 1, 2):
            e_exact += 1
        while Fraction(4) ** e_exact * sa > Fraction(P - 1, 2):
            e_exact -= 1
        assert ei in (e_exact, e_exact - 1)
    for i in range(9):
        for j in range(8):
            lhs = (2 * Fraction(2) ** (int(e[i]) + int(f[j]))) ** 2 * _exact_sq(A[i]) * _exact_sq(Bt[j])
            assert lhs <= (P - 1) ** 2


def test_fast_scaling_matches_bigref():
    for seed in range(6):
        A, _ = workloads.make_pair("spread", 6, 1, 17, seed=seed, phi=3.0)
        for N in (3, 14, 20):
            _, H, _, _ = orc.tables(N)
            e = orc.scale_fast(A, N)
            assert list(e) == [bigref.scale_fast_row([float(x) for x in r], H) for r in A]


@pytest.mark.parametrize("s", [-1000, -200, -50, 0, 50, 200, 900])
def test_scale_invariance(s):
    """[G] Methodik 2: A * 2^s leaves the scaled integers unchanged and C
    scales by 2^s exactly."""
    A, Bt = workloads.make_pair("spread", 12, 10, 50, seed=5, phi=2.0)
    N = 16
    e0 = orc.scale_fast(A, N)
    As = np.ldexp(A, s)
    es = orc.scale_fast(As, N)
    assert np.array_equal(es, e0 - s)
    assert np.array_equal(orc.integers(As, es), orc.integers(A, e0))
    r0 = orc.gemm_entries(A, Bt, N)
    rs = orc.gemm_entries(As, Bt, N)
    assert r0.mismatches == 0 and rs.mismatches == 0
    assert np.array_equal(rs.C, np.ldexp(r0.C, s))
    # accurate mode too
    a0 = orc.gemm_entries(A, Bt, N, mode=orc.ACCURATE)
    as_ = orc.gemm_entries(As, Bt, N, mode=orc.ACCURATE)
    assert np.array_equal(as_.e, a0.e - s)
    assert np.array_equal(as_.C, np.ldexp(a0.C, s))


def test_accurate_scaling_bound_and_bigref():
    """Accurate mode: mu_i nu_j (|A||B|)_ij <= H for every entry (the
    condition that keeps |A'B'| below P/2), same exponents as the Python
    restatement."""
    for seed, phi in [(0, 0.5), (1, 4.0), (2, 8.0)]:
        A, Bt = workloads.make_pair("spread", 7, 6, 23, seed=seed, phi=phi)
        Bt[2, :] = 0.0
        for N in (4, 14, 20):
            P, H, _, _ = orc.tables(N)
            e, f, R, K = orc.scale_accu(A, Bt, N, return_bounds=True)
            be, bf = bigref.scale_accu([[float(x) for x in r] for r in A],
                                       [[float(x) for x in r] for r in Bt], H)
            assert list(e) == be and list(f) == bf
            for i in range(7):
                for j in range(6):
                    s = sum(abs(Fraction(float(a))) * abs(Fraction(float(b))) for a, b in zip(A[i], Bt[j]))
                    assert Fraction(2) ** (int(e[i]) + int(f[j])) * s <= H
            # maximality of the row exponent against its own bound R_i
            for i in range(7):
                if R[i]:
                    E = max(math.frexp(float(x))[1] for x in A[i] if x != 0)
                    g = int(e[i]) - 6 + E
                    assert R[i] * Fraction(4) ** g <= H < R[i] * Fraction(4) ** (g + 1)


def test_accurate_scaling_worked_example():
    """The accurate-mode reading of [Q] 手順1と5 / [G] Problemstellung 1 (one
    extra INT8 product bounds |A||B|), worked by hand on a 2 x 3 by 3 x 2
    product with 4 moduli, so that a slip in the magnitude planes' width or
    rounding, in the bound product or in the exponent search fails here
    whatever the other restatements do.

    Tight exponents (|x| < 2^E): rows of A 1, 2; columns of B 1, 0.
    Magnitude planes ceil(|x| 2^(6 - E)):
      row 0 * 32: 1, 0.5, 0.3 -> 32, 16, 10 (9.6 rounds up)
      row 1 * 16: 3, 2.5, 0   -> 48, 40, 0
      col 0 * 32: 0.25, 0.25, 1 -> 8, 8, 32
      col 1 * 64: 0.1, 0.7, 0   -> 7, 45, 0 (6.4 and 44.8 round up)
    Bound product: [[32*8 + 16*8 + 10*32, 32*7 + 16*45], [48*8 + 40*8, 48*7 + 40*45]]
                 = [[704, 944], [704, 2136]]
    R = row maxima (944, 2136), K = column maxima (704, 2136).
    N = 4: P = 256*255*253*251 = 4145475840, H = 2072737919.
    Largest g with R 4^g <= H: 944 -> 10 (944*4^10 = 989855744), 2136 -> 9
    (2136*4^9 = 559939584, 2136*4^10 > H), 704 -> 10 (704*4^10 = 738197504).
    e = g + 6 - E: row 0 10 + 5 = 15, row 1 9 + 4 = 13; f: col 0 10 + 5 = 15,
    col 1 9 + 6 = 15."""
    A = np.array([[1.0, 0.5, 0.3], [-3.0, 2.5, 0.0]])
    Bt = np.array([[0.25, 0.25, 1.0], [0.1, -0.7, 0.0]])
    P, H, _, _ = orc.tables(4)
    assert (P, H) == (4145475840, 2072737919)
    e, f, R, K = orc.scale_accu(A, Bt, 4, return_bounds=True)
    assert list(R) == [944, 2136]
    assert list(K) == [704, 2136]
    assert list(e) == [15, 13]
    assert list(f) == [15, 15]


def test_fast_scaling_worked_example():
    """The fast (revised) scaling of [G] Methodik 1, with its log2 of the sum
    of squares replaced by the exact upper bound Q = sum ceil(|x| 2^(23-E))^2,
    worked by hand on the operands of the accurate-mode example, 4 moduli
    (H = 2072737919).  E as there: rows 1, 2; columns 1, 0.
      row 0 * 2^22: 1, 0.5, 0.3 -> 4194304, 2097152, 1258292 (1258291.2 up)
        Q = 2^44 + 2^42 + 1258292^2 = 23573531312784
      row 1 * 2^21: 3, 2.5, 0 -> 6291456, 5242880, 0
        Q = 6291456^2 + 5242880^2 = 67070209294336
      col 0 * 2^22: 0.25, 0.25, 1 -> 1048576, 1048576, 4194304
        Q = 2 * 2^40 + 2^44 = 19791209299968
      col 1 * 2^23: 0.1, 0.7, 0 -> 838861, 5872026, 0 (838860.8, 5872025.6 up)
        Q = 838861^2 + 5872026^2 = 35184377121997
    Largest g with Q 4^g <= H: -7 (Q / 4^7 = 1438814167.04; / 4^6 > H),
    -8 (Q / 4^8 = 1023410176; / 4^7 > H), -7 (1207959552; / 4^6 > H),
    -8 (536870988.8; / 4^7 = 2147483955.2 > H).  e = g + 23 - E: 15, 13;
    f: 15, 15."""
    A = np.array([[1.0, 0.5, 0.3], [-3.0, 2.5, 0.0]])
    Bt = np.array([[0.25, 0.25, 1.0], [0.1, -0.7, 0.0]])
    e, Qa = orc.scale_fast(A, 4, return_Q=True)
    f, Qb = orc.scale_fast(Bt, 4, return_Q=True)
    assert [int(x) for x in Qa] == [23573531312784, 67070209294336]
    assert [int(x) for x in Qb] == [19791209299968, 35184377121997]
    assert list(e) == [15, 13]
    assert list(f) == [15, 15]


# ------------------------------------------------------- full pipeline ------
def _rand_special(rng, m, k):
    A = rng.standard_normal((m, k)) * np.exp2(rng.integers(-30, 30, size=(m, k)))
    A[rng.random((m, k)) < 0.15] = 0.0
    return A


@pytest.mark.parametrize("mode", ["fast", "accurate"])
@pytest.mark.parametrize("N", [2, 5, 12, 16, 20])
def test_bruteforce_tiny_matches_bigref(mode, N):
    """Brute force on tiny inputs: the C oracle and the Python restatement
    agree on exponents, residue products, CRT values and C, and the CRT value
    equals the direct exact integer product."""
    rng = np.random.default_rng(N)
    A = _rand_special(rng, 5, 11)
    Bt = _rand_special(rng, 4, 11)
    A[1, :] = 0.0
    Bt[0, 3] = 5e-324            # a subnormal
    A[2, 0] = -2.0 ** 900
    ref = bigref.gemm([[float(x) for x in r] for r in A], [[float(x) for x in r] for r in Bt], N, mode)
    got = orc.gemm_entries(A, Bt, N, mode=orc.FAST if mode == "fast" else orc.ACCURATE)
    assert got.mismatches == 0
    assert list(got.e) == ref["e"] and list(got.f) == ref["f"]
    for i in range(5):
        for j in range(4):
            assert ref["X"][i][j] == ref["Xd"][i][j]
            assert abs(ref["X"][i][j]) <= ref["H"]
            assert orc.X_int(got, i, j) == ref["X"][i][j]
            assert list(got.G[i, j]) == ref["G"][i][j]
            assert list(got.c[i, j]) == ref["c"][i][j]
            assert got.C[i, j] == ref["C"][i][j] or (math.isnan(got.C[i, j]) and math.isnan(ref["C"][i][j]))
            assert math.copysign(1, got.C[i, j]) == math.copysign(1, ref["C"][i][j])


def test_integer_inputs_are_exact():
    """[Q] 2の累乗による整数化(手順1と5): only the truncation loses bits, so
    integer-valued inputs give exactly A B."""
    A, Bt = workloads.make_pair("int", 20, 17, 64, seed=2, phi=1000)
    r = orc.gemm_entries(A, Bt, 14)
    assert r.mismatches == 0
    exact = A @ Bt.T            # integers far below 2^53: exact in float64
    assert np.array_equal(r.C, exact)


@pytest.mark.parametrize("N", [12, 16, 20])
def test_all_ones_closed_form(N):
    """All-ones matrices: every entry of A B equals k."""
    for k in (1, 7, 64, 300):
        A, Bt = workloads.make_pair("ones", 3, 4, k)
        r = orc.gemm_entries(A, Bt, N)
        assert np.all(r.C == k)
        ra = orc.gemm_entries(A, Bt, N, mode=orc.ACCURATE)
        assert np.all(ra.C == k)


def test_truncation_error_bound():
    """|C - AB| <= 2^-(e+f) sum_h (mu|a| + nu|b| + 1) + half an ulp: the only
    losses are the truncations of step 2 and the final rounding."""
    A, Bt = workloads.make_pair("spread", 6, 5, 30, seed=9, phi=3.0)
    for N in (6, 10, 14):
        r = orc.gemm_entries(A, Bt, N)
        for i in range(6):
            for j in range(5):
                ex = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[i], Bt[j]))
                mu = Fraction(2) ** int(r.e[i])
                nu = Fraction(2) ** int(r.f[j])
                bound = sum(mu * abs(Fraction(float(a))) + nu * abs(Fraction(float(b))) + 1
                            for a, b in zip(A[i], Bt[j])) / (mu * nu)
                c = Fraction(float(r.C[i, j]))
                half_ulp = Fraction(math.ulp(float(r.C[i, j]))) / 2
                assert abs(c - ex) <= bound + half_ulp


def test_more_moduli_means_more_accuracy():
    """[Q] 行列積の回数と性能: about 4 more bits per element per modulus."""
    A, Bt = workloads.make_pair("normal", 8, 8, 64, seed=0)
    exact = [[sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[i], Bt[j]))
              for j in range(8)] for i in range(8)]
    errs = []
    for N in (8, 10, 12, 14, 16):
        r = orc.gemm_entries(A, Bt, N)
        errs.append(max(abs(Fraction(float(r.C[i, j])) - exact[i][j]) for i in range(8) for j in range(8)))
    for a, b in zip(errs, errs[1:]):
        assert b <= a
    assert errs[0] > 0 and errs[0] / max(errs[2], Fraction(1, 2 ** 1100)) > 2 ** 10


# ------------------------------------------------------------ rounding ------
def test_round_scaled_against_fraction():
    """Step 5 is one correctly rounded conversion (RN-even, subnormals)."""
    rnd = random.Random(7)
    cases = [(1, 0), (-1, 0), (3, 1), (5, 2), (2 ** 53 + 1, 0), (2 ** 54 + 2, 1), (-(2 ** 53 + 3), 0),
             (1, 1074), (1, 1075), (3, 1076), (2, 1076), (1, 1076), (-1, 1075), (2 ** 60 - 1, 1074 + 60),
             (2 ** 52 + 1, 1074 + 52), ((1 << 150) - 1, -800), (1 << 120, -950), (-(1 << 155) + 12345, -900)]
    for _ in range(3000):
        b = rnd.randint(1, 200)
        X = rnd.getrandbits(b) * rnd.choice((1, -1))
        s = rnd.randint(-1100, 1300)
        cases.append((X, s))
        # exact ties at the 53-bit boundary
        base = rnd.getrandbits(53) | (1 << 52)
        sh = rnd.randint(1, 100)
        cases.append(((2 * base + 1) << (sh - 1), sh + rnd.randint(-900, 900)))
    for X, s in cases:
        try:
            want = float(Fraction(X, 1) / Fraction(2) ** s) if X else 0.0
        except OverflowError:
            want = math.copysign(math.inf, X)
        got = orc.round_scaled(X, s)
        assert got == want or (math.isinf(got) and math.isinf(want)), (X, s, got, want)
        assert math.copysign(1, got) == math.copysign(1, want), (X, s)


def test_nonfinite_rejected():
    A, Bt = workloads.make_pair("normal", 4, 4, 8)
    A[1, 2] = np.nan
    with pytest.raises(orc.OracleError) as ei:
        orc.gemm_entries(A, Bt, 14)
    assert ei.value.status == orc.ERR_NONFINITE
    A[1, 2] = np.inf
    with pytest.raises(orc.OracleError):
        orc.scale_fast(A, 14)


# ------------------------------------------------------- SGEMM emulation ----
def _round_fraction(fr, prec, emin, emax):
    """Correct RN-even rounding of a rational to a binary format (reference)."""
    if fr == 0:
        return 0.0
    sign = -1.0 if fr < 0 else 1.0
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e, emin) - (prec - 1)
    scaled = a / Fraction(2) ** q
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = Fraction(n) * Fraction(2) ** q
    if val >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * float(val)


def test_round_scaled_f32_against_fraction():
    """Binary32 unscale (SGEMM emulation, [G] Ergebnisse): one RN-even rounding
    to 24 bits, subnormals down to 2^-149, overflow at 2^128."""
    rnd = random.Random(11)
    cases = [(1, 149), (1, 150), (3, 151), (2 ** 24 + 1, 0), (-(2 ** 25 + 3), 1), (1, -127), (3, -127),
             ((1 << 24) - 1, -104), ((1 << 25) - 1, -104)]
    for _ in range(3000):
        X = rnd.getrandbits(rnd.randint(1, 160)) * rnd.choice((1, -1))
        cases.append((X, rnd.randint(-300, 400)))
        base = rnd.getrandbits(24) | (1 << 23)
        sh = rnd.randint(1, 60)
        cases.append(((2 * base + 1) << (sh - 1), sh + rnd.randint(-150, 150)))
    for X, s in cases:
        want = _round_fraction(Fraction(X) / Fraction(2) ** s, 24, -126, 127) if X else 0.0
        got = orc.round_scaled_f32(X, s)
        assert got == want or (math.isinf(got) and math.isinf(want)), (X, s, got, want)
        assert math.copysign(1, got) == math.copysign(1, want), (X, s)
        if not math.isinf(got):
            assert float(np.float32(got)) == got      # representable in binary32


def test_sgemm_oracle_integer_inputs_exact():
    A, Bt = workloads.make_pair("int", 12, 10, 50, seed=1, phi=100)
    r = orc.gemm_entries(A.astype(np.float32), Bt.astype(np.float32), 7, out_f32=True)
    assert r.C.dtype == np.float32
    assert np.array_equal(r.C, (A @ Bt.T).astype(np.float32))


# ------------------------------------------------------------ complex --------
def test_complex_oracle_integer_inputs_exact():
    """[G] Bedeutung (ZGEMM/CGEMM): the block form reproduces the complex
    product; small-integer complex inputs give it exactly."""
    rng = np.random.default_rng(3)
    A = rng.integers(-50, 51, (9, 23)) + 1j * rng.integers(-50, 51, (9, 23))
    Bt = rng.integers(-50, 51, (7, 23)) + 1j * rng.integers(-50, 51, (7, 23))
    C, r = orc.complex_gemm_entries(A, Bt, 14)
    assert r.mismatches == 0
    assert np.array_equal(C, A @ Bt.T)
    Cs, _ = orc.complex_gemm_entries(A.astype(np.complex64), Bt.astype(np.complex64), 8, single=True)
    assert np.array_equal(Cs, (A @ Bt.T).astype(np.complex64))


def test_complex_scaling_uses_complex_norms():
    """The stacked row norm is the complex row norm: mu_i^2 sum_h |a_ih|^2 <= H."""
    rng = np.random.default_rng(5)
    A = rng.standard_normal((6, 30)) + 1j * rng.standard_normal((6, 30)) * 4.0
    A2, _ = orc.stack_complex(A, np.zeros((1, 30), complex))
    for N in (8, 16):
        _, H, _, _ = orc.tables(N)
        e = orc.scale_fast(A2, N)
        for i in range(6):
            norm2 = sum(Fraction(float(z.real)) ** 2 + Fraction(float(z.imag)) ** 2 for z in A[i])
            assert Fraction(4) ** int(e[i]) * norm2 <= H


def test_complex_emulation_error_small():
    A, Bt = workloads.make_pair("normal", 5, 4, 40, seed=2)
    Ai, Bi = workloads.make_pair("normal", 5, 4, 40, seed=3)
    Z, W = A + 1j * Ai, Bt + 1j * Bi
    C, _ = orc.complex_gemm_entries(Z, W, 16)
    for i in range(5):
        for j in range(4):
            re = sum(Fraction(float(a.real)) * Fraction(float(b.real)) - Fraction(float(a.imag)) * Fraction(float(b.imag)) for a, b in zip(Z[i], W[j]))
            im = sum(Fraction(float(a.real)) * Fraction(float(b.imag)) + Fraction(float(a.imag)) * Fraction(float(b.real)) for a, b in zip(Z[i], W[j]))
            scale = float(sum(abs(a) * abs(b) for a, b in zip(Z[i], W[j])))
            assert abs(float(Fraction(C[i, j].real) - re)) <= 2.0 ** -48 * scale
            assert abs(float(Fraction(C[i, j].imag) - im)) <= 2.0 ** -48 * scale
