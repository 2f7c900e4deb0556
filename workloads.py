"""Seeded synthetic inputs for the Ozaki Scheme II GEMM.

Shared by the tests, the benchmark and the oracle checks.  This module holds
no arithmetic of the method: it only draws matrices.

All generators use numpy's PCG64 (``numpy.random.default_rng(seed)``); A is
drawn first, then B, from one stream.  B is drawn directly in its
K-contiguous form Bt (n x k row-major, B = Bt.T); its entries are i.i.d., so
that is the same distribution as drawing B and transposing.

Value recipes (the pages test random matrices whose exponent spread is set by
phi, see "Improved Scaling for Fast Mode of Ozaki Scheme II", "Ergebnisse"):
  normal      N(0, 1)
  spread      (U(0,1) - 0.5) * exp(phi * N(0, 1))
  ones        all ones
  int         integers uniform in [-lo, lo]
"""
from __future__ import annotations

import numpy as np


def _draw(rng, kind, shape, phi):
    if kind == "normal":
        return rng.standard_normal(shape)
    if kind == "spread":
        u = rng.random(shape)
        g = rng.standard_normal(shape)
        return (u - 0.5) * np.exp(phi * g)
    if kind == "ones":
        return np.ones(shape)
    if kind == "int":
        return rng.integers(-int(phi), int(phi) + 1, size=shape).astype(np.float64)
    raise ValueError(f"unknown input kind {kind!r}")


def make_pair(kind: str, m: int, n: int, k: int, seed: int = 0, phi: float = 0.5):
    """Return (A, Bt): A m x k and Bt n x k, float64, C-contiguous."""
    rng = np.random.default_rng(seed)
    A = np.ascontiguousarray(_draw(rng, kind, (m, k), phi), dtype=np.float64)
    Bt = np.ascontiguousarray(_draw(rng, kind, (n, k), phi), dtype=np.float64)
    return A, Bt


def sample_grid(m: int, n: int, count: int = 64, seed: int = 1):
    """Seeded sample of output entries: `count` distinct rows x `count`
    distinct columns (count*count entries), sorted, always including the
    last row and column (the ragged tail)."""
    rng = np.random.default_rng(seed)
    def pick(size):
        c = min(count, size)
        s = set(rng.choice(size, size=c, replace=False).tolist())
        if size - 1 not in s:
            s.pop()
            s.add(size - 1)
        return np.array(sorted(s), dtype=np.int32)
    return pick(m), pick(n)


# The five workloads, by name: (shape, value recipe, moduli counts, modes).
CONFIGS = {
    "64cube_normal": dict(m=64, n=64, k=64, kind="normal", phi=0.0, N=[14], modes=["fast"]),
    "1024cube_spread": dict(m=1024, n=1024, k=1024, kind="spread", phi=[0.5, 2.0, 4.0],
                            N=[12, 14, 16, 18, 20], modes=["fast", "accurate"]),
    "4096cube_scale_sweep": dict(m=4096, n=4096, k=4096, kind=["ones", "normal"],
                                 s=[-200, -100, -50, 0, 50, 100, 200], N=[16],
                                 modes=["fast", "accurate"]),
    "8192cube_spread": dict(m=8192, n=8192, k=8192, kind="spread", phi=0.5, N=[14, 16, 18],
                            modes=["fast", "accurate"]),
    "16384sq_k32768_spread": dict(m=16384, n=16384, k=32768, kind="spread", phi=1.0, N=[18],
                                  modes=["fast"]),
}
