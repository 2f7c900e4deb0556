"""Pure-Python big-integer restatement of Ozaki Scheme II, for tiny inputs.

TEST INFRASTRUCTURE ONLY.  A second, independent statement of the oracle's
arithmetic (Python ints and fractions.Fraction, no C), used to cross-check
``os2_oracle.c`` on inputs small enough for pure-Python loops.

Sources:
  [Q] Qiita, "8ビットの整数で53ビットの倍精度を組み立てる。中国剰余定理をGPUに載せた
      Ozaki Scheme II".
  [G] gist.science, "Improved Scaling for Fast Mode of Ozaki Scheme II".
"""
from __future__ import annotations

import math
from fractions import Fraction


def greedy_moduli(N: int, top: int = 256) -> list[int]:
    """[Q] "256以下の法の選び方(手順2)": pairwise coprime, as large as possible.
    Taken greedily from 256 downwards."""
    out: list[int] = []
    x = top
    while len(out) < N and x > 1:
        if all(math.gcd(x, y) == 1 for y in out):
            out.append(x)
        x -= 1
    return out


def crt_constants(mods):
    """[Q] "秦九韶の大衍求一術": 衍母 P, 衍数 M_l, 奇数 M_l mod p_l, 乗率 inv_l,
    用数 W_l = M_l * inv_l."""
    P = math.prod(mods)
    M = [P // p for p in mods]
    odd = [Ml % p for Ml, p in zip(M, mods)]
    inv = [pow(o, -1, p) if p > 1 else 0 for o, p in zip(odd, mods)]
    W = [Ml * i for Ml, i in zip(M, inv)]
    return P, M, odd, inv, W


def sym(x: int, p: int) -> int:
    """Residue held around zero: [-floor(p/2), ceil(p/2) - 1]."""
    r = x % p
    return r - p if r >= (p + 1) // 2 else r


def crt(residues, mods) -> int:
    """Textbook CRT lifted to [-P/2, P/2)."""
    P, _, _, _, W = crt_constants(mods)
    r = sum(c * w for c, w in zip(residues, W)) % P
    return r - P if r >= (P + 1) // 2 else r


def _max_exp(row) -> int | None:
    """E with |x| < 2^E for every entry, tight (1 + floor(log2 max|x|))."""
    nz = [x for x in row if x != 0.0]
    if not nz:
        return None
    return max(math.frexp(x)[1] for x in nz)


def _fits(Q: int, g: int, H: int) -> bool:
    return Fraction(Q) * Fraction(4) ** g <= H


def _largest_g(Q: int, H: int) -> int:
    """Largest integer g with Q * 4^g <= H (as rationals)."""
    g = 0
    if _fits(Q, 0, H):
        while _fits(Q, g + 1, H):
            g += 1
    else:
        while not _fits(Q, g, H):
            g -= 1
    return g


def scale_fast_row(row, H: int) -> int:
    """[G] "Methodik" 1, exact-integer form: e = g + 23 - E with g the largest
    integer such that Q 4^g <= H, Q = sum ceil(|x| 2^(23-E))^2."""
    E = _max_exp(row)
    if E is None:
        return 0
    Q = sum(math.ceil(Fraction(abs(x)) * Fraction(2) ** (23 - E)) ** 2 for x in row)
    return _largest_g(Q, H) + 23 - E


def bars(row):
    E = _max_exp(row)
    if E is None:
        return 0, [0] * len(row)
    return E, [math.ceil(Fraction(abs(x)) * Fraction(2) ** (6 - E)) for x in row]


def scale_accu(A, Bt, H: int):
    """Accurate mode: Abar Bbar bounds, row/col maxima -> exponents."""
    EA, Ab = zip(*[bars(r) for r in A]) if A else ((), ())
    EB, Bb = zip(*[bars(r) for r in Bt]) if Bt else ((), ())
    Cb = [[sum(a * b for a, b in zip(Ab[i], Bb[j])) for j in range(len(Bt))] for i in range(len(A))]
    e, f = [], []
    for i in range(len(A)):
        R = max(Cb[i]) if Cb[i] else 0
        e.append(-EA[i] if R == 0 else _largest_g(R, H) + 6 - EA[i])
    for j in range(len(Bt)):
        K = max(Cb[i][j] for i in range(len(A))) if A else 0
        f.append(-EB[j] if K == 0 else _largest_g(K, H) + 6 - EB[j])
    return e, f


def trunc_scaled(x: float, e: int) -> int:
    """trunc(x * 2^e) toward zero ([Q] "2の累乗による整数化(手順1と5)")."""
    return int(Fraction(x) * Fraction(2) ** e)


def gemm(A, Bt, N: int, mode: str = "fast"):
    """Full pipeline on lists of Python floats.  Returns dict with e, f,
    integer matrices, residues, per-modulus products, X, C."""
    mods = greedy_moduli(N)
    P = math.prod(mods)
    H = (P - 1) // 2
    if mode == "fast":
        e = [scale_fast_row(r, H) for r in A]
        f = [scale_fast_row(r, H) for r in Bt]
    else:
        e, f = scale_accu(A, Bt, H)
    Ai = [[trunc_scaled(x, e[i]) for x in r] for i, r in enumerate(A)]
    Bi = [[trunc_scaled(x, f[j]) for x in r] for j, r in enumerate(Bt)]
    m, n = len(A), len(Bt)
    Xd = [[sum(a * b for a, b in zip(Ai[i], Bi[j])) for j in range(n)] for i in range(m)]
    G = [[[sum(sym(a, p) * sym(b, p) for a, b in zip(Ai[i], Bi[j])) for p in mods]
          for j in range(n)] for i in range(m)]
    c = [[[sym(g, p) for g, p in zip(G[i][j], mods)] for j in range(n)] for i in range(m)]
    X = [[crt(c[i][j], mods) for j in range(n)] for i in range(m)]
    C = [[float(Fraction(X[i][j]) / Fraction(2) ** (e[i] + f[j])) for j in range(n)] for i in range(m)]
    return dict(mods=mods, P=P, H=H, e=e, f=f, Ai=Ai, Bi=Bi, Xd=Xd, G=G, c=c, X=X, C=C)
