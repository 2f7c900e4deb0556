"""CPU oracle for Ozaki Scheme II -- Python side.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
CPU-baseline leg of the benchmark, never by the library.  It shares no code
with the CUDA path.

Wraps ``os2_oracle.c`` (plain C, exact integer arithmetic, OpenMP over output
entries) through ctypes.  ``build()`` compiles it with gcc into
``oracle/_build/liboracle.so`` (git-ignored); ``load()`` builds on first use.

Layouts follow the library boundary: A is m x k row-major (lda >= k), Bt is
n x k row-major (so B = Bt.T, its columns contiguous).
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "os2_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liboracle.so")

FAST, ACCURATE = 0, 1
OK, ERR_ARG, ERR_NONFINITE = 0, 1, 4
NL = 8  # 32-bit limbs per big integer

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP). Returns the .so path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, SRC])
        os.replace(tmp, LIB)
    return LIB


def load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ct.CDLL(build())
            P = ct.c_void_p
            i32, i64, l = ct.c_int, ct.c_int64, ct.c_long
            lib.orc_moduli.argtypes = [i32, P]
            lib.orc_tables.argtypes = [i32, P, P, P, P]
            lib.orc_inverse_bruteforce.argtypes = [i64, i64]
            lib.orc_inverse_bruteforce.restype = i64
            lib.orc_dayan_qiuyi.argtypes = [i64, i64]
            lib.orc_dayan_qiuyi.restype = i64
            lib.orc_crt_small.argtypes = [i32, P, P, P]
            lib.orc_scale_fast.argtypes = [i32, i32, P, l, i32, P, P]
            lib.orc_scale_accu.argtypes = [i32, i32, i32, P, l, P, l, i32, i32, P, P, i32, P, P, P, P]
            lib.orc_row_exponents.argtypes = [i32, i32, P, l, P]
            lib.orc_exps_from_bounds.argtypes = [i32, P, P, i32, P]
            lib.orc_integers.argtypes = [i32, i32, P, l, P, P]
            lib.orc_residues.argtypes = [i32, i32, P, l, P, i32, P]
            lib.orc_round_scaled.argtypes = [P, i32]
            lib.orc_round_scaled.restype = ct.c_double
            lib.orc_round_scaled_f32.argtypes = [P, i32]
            lib.orc_round_scaled_f32.restype = ct.c_double
            lib.orc_set_output_f32.argtypes = [i32]
            lib.orc_gemm_entries.argtypes = [i32, i32, i32, P, l, P, l, i32, i32, P, i32, P,
                                             i32, P, P, P, P, P, P, P]
            lib.orc_num_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ct.c_void_p)


def _check(st, what):
    if st != OK:
        raise OracleError(st, f"{what} failed with status {st}")


class OracleError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(msg)
        self.status = status


def num_threads() -> int:
    return int(load().orc_num_threads())


# --------------------------------------------------------------------------
# big integers <-> Python int
# --------------------------------------------------------------------------
def limbs_to_int(w) -> int:
    """8 little-endian u32 limbs, two's complement 256-bit -> Python int."""
    v = 0
    for i, x in enumerate(np.asarray(w, dtype=np.uint64)):
        v |= int(x) << (32 * i)
    if v >> 255:
        v -= 1 << 256
    return v


def int_to_limbs(v: int) -> np.ndarray:
    v &= (1 << 256) - 1
    return np.array([(v >> (32 * i)) & 0xFFFFFFFF for i in range(NL)], dtype=np.uint32)


# --------------------------------------------------------------------------
# tables
# --------------------------------------------------------------------------
def moduli(N: int) -> list[int]:
    out = np.zeros(20, np.int32)
    if load().orc_moduli(N, _ptr(out)) != N:
        raise OracleError(ERR_ARG, f"no moduli set for N={N}")
    return [int(x) for x in out[:N]]


def tables(N: int):
    """Return (P, H, W list, inv list) as Python ints."""
    P = np.zeros(NL, np.uint32)
    H = np.zeros(NL, np.uint32)
    W = np.zeros(NL * 20, np.uint32)
    inv = np.zeros(20, np.int32)
    _check(load().orc_tables(N, _ptr(P), _ptr(H), _ptr(W), _ptr(inv)), "orc_tables")
    return (limbs_to_int(P), limbs_to_int(H),
            [limbs_to_int(W[NL * l:NL * (l + 1)]) for l in range(N)], [int(x) for x in inv[:N]])


def inverse_bruteforce(a: int, p: int) -> int:
    return int(load().orc_inverse_bruteforce(a, p))


def dayan_qiuyi(a: int, p: int) -> int:
    return int(load().orc_dayan_qiuyi(a, p))


def crt_small(residues, mods) -> int:
    r = np.asarray(residues, np.int64)
    m = np.asarray(mods, np.int64)
    out = np.zeros(1, np.int64)
    _check(load().orc_crt_small(len(r), _ptr(r), _ptr(m), _ptr(out)), "orc_crt_small")
    return int(out[0])


def round_scaled(X: int, s: int) -> float:
    """RN-even of X * 2^-s as binary64 (the oracle's unscale step)."""
    return float(load().orc_round_scaled(_ptr(int_to_limbs(X)), s))


def round_scaled_f32(X: int, s: int) -> float:
    """RN-even of X * 2^-s to binary32 (value returned as a Python float)."""
    return float(load().orc_round_scaled_f32(_ptr(int_to_limbs(X)), s))


# --------------------------------------------------------------------------
# steps
# --------------------------------------------------------------------------
def _rows(X):
    X = np.asarray(X)
    assert X.dtype == np.float64 and X.ndim == 2 and X.strides[1] == 8
    return X, X.strides[0] // 8


def scale_fast(X, N: int, return_Q: bool = False):
    """Fast-mode (revised) exponents e_i of every row of X (rows x k)."""
    X, ld = _rows(X)
    e = np.zeros(X.shape[0], np.int32)
    Q = np.zeros(X.shape[0], np.uint64)
    _check(load().orc_scale_fast(X.shape[0], X.shape[1], _ptr(X), ld, N, _ptr(e), _ptr(Q)),
           "orc_scale_fast")
    return (e, Q) if return_Q else e


def scale_accu(A, Bt, N: int, rows=None, cols=None, return_bounds: bool = False):
    """Accurate-mode exponents for the selected rows of A and columns of B."""
    A, lda = _rows(A)
    Bt, ldb = _rows(Bt)
    m, k = A.shape
    n = Bt.shape[0]
    rows = np.arange(m, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    cols = np.arange(n, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    e = np.zeros(len(rows), np.int32)
    f = np.zeros(len(cols), np.int32)
    R = np.zeros(len(rows), np.int64)
    K = np.zeros(len(cols), np.int64)
    _check(load().orc_scale_accu(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, N, len(rows), _ptr(rows),
                                 _ptr(e), len(cols), _ptr(cols), _ptr(f), _ptr(R), _ptr(K)),
           "orc_scale_accu")
    return (e, f, R, K) if return_bounds else (e, f)


def row_exponents(X):
    """Exponent bases E_i of the rows of X (|x_ih| < 2^E_i, 0 for a zero row),
    as the accurate mode uses them."""
    X, ld = _rows(X)
    E = np.zeros(X.shape[0], np.int32)
    _check(load().orc_row_exponents(X.shape[0], X.shape[1], _ptr(X), ld, _ptr(E)),
           "orc_row_exponents")
    return E


def exps_from_bounds(R, E, N: int):
    """Accurate-mode exponents from bounds R and exponent bases E (the last
    step of ``scale_accu``, for bounds reduced across the blocks of a split
    product)."""
    R = np.ascontiguousarray(R, np.int64)
    E = np.ascontiguousarray(E, np.int32)
    e = np.zeros(len(R), np.int32)
    _check(load().orc_exps_from_bounds(len(R), _ptr(R), _ptr(E), N, _ptr(e)),
           "orc_exps_from_bounds")
    return e


def integers(X, e):
    """Scaled integers trunc(x_ih * 2^e_i) as a Python-int object array."""
    X, ld = _rows(X)
    e = np.ascontiguousarray(e, np.int32)
    out = np.zeros((X.shape[0], X.shape[1], 2), np.int64)
    _check(load().orc_integers(X.shape[0], X.shape[1], _ptr(X), ld, _ptr(e), _ptr(out)),
           "orc_integers")
    lo = out[..., 0].astype(np.uint64).astype(object)
    hi = out[..., 1].astype(object)
    return hi * (1 << 64) + lo


def residues(X, e, N: int):
    """Symmetric residue planes, int8 [N][rows][k]."""
    X, ld = _rows(X)
    e = np.ascontiguousarray(e, np.int32)
    out = np.zeros((N, X.shape[0], X.shape[1]), np.int8)
    _check(load().orc_residues(X.shape[0], X.shape[1], _ptr(X), ld, _ptr(e), N, _ptr(out)),
           "orc_residues")
    return out


class Entries:
    """Oracle results for a grid of output entries (rows x cols)."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def gemm_entries(A, Bt, N: int, rows=None, cols=None, mode: int = FAST, e=None, f=None,
                 want_X=True, want_c=True, want_G=True, out_f32=False) -> Entries:
    """Steps 1-5 for the output entries rows x cols.

    In FAST mode the exponents are computed from the selected rows/columns
    alone.  In ACCURATE mode they come from ``scale_accu`` (or are passed in
    as e, f for the selected rows/columns).  float32 inputs are taken as the
    doubles they equal; out_f32 rounds C to binary32 (SGEMM emulation).
    """
    A = np.ascontiguousarray(A, dtype=np.float64) if np.asarray(A).dtype == np.float32 else A
    Bt = np.ascontiguousarray(Bt, dtype=np.float64) if np.asarray(Bt).dtype == np.float32 else Bt
    A, lda = _rows(A)
    Bt, ldb = _rows(Bt)
    m, k = A.shape
    n = Bt.shape[0]
    rows = np.arange(m, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    cols = np.arange(n, dtype=np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    nr, nc = len(rows), len(cols)
    compute = 1
    if e is not None or f is not None or mode == ACCURATE:
        if e is None or f is None:
            e, f = scale_accu(A, Bt, N, rows, cols)
        e = np.ascontiguousarray(e, np.int32).copy()
        f = np.ascontiguousarray(f, np.int32).copy()
        compute = 0
    else:
        e = np.zeros(nr, np.int32)
        f = np.zeros(nc, np.int32)
    C = np.zeros((nr, nc), np.float64)
    X = np.zeros((nr, nc, NL), np.uint32) if want_X else None
    c = np.zeros((nr, nc, N), np.int8) if want_c else None
    G = np.zeros((nr, nc, N), np.int64) if want_G else None
    bad = np.zeros(1, np.int64)
    lib = load()
    with _lock:
        lib.orc_set_output_f32(1 if out_f32 else 0)
        try:
            _check(lib.orc_gemm_entries(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, N, nr, _ptr(rows),
                                        nc, _ptr(cols), compute, _ptr(e), _ptr(f), _ptr(C), _ptr(X),
                                        _ptr(c), _ptr(G), _ptr(bad)), "orc_gemm_entries")
        finally:
            lib.orc_set_output_f32(0)
    if out_f32:
        C = C.astype(np.float32)
    return Entries(rows=rows, cols=cols, e=e, f=f, C=C, X=X, c=c, G=G, mismatches=int(bad[0]))


def X_int(ent: Entries, a: int, b: int) -> int:
    return limbs_to_int(ent.X[a, b])


# --------------------------------------------------------------------------
# complex products
# --------------------------------------------------------------------------
def stack_complex(A, Bt):
    """The real block form of a complex product: C_r = [A_r|A_i].[B_r;-B_i],
    C_i = [A_r|A_i].[B_i;B_r].  Returns (A2 m x 2k, Bt2 2n x 2k) as float64
    (complex64 parts are exact in float64)."""
    A = np.asarray(A)
    Bt = np.asarray(Bt)
    A2 = np.ascontiguousarray(np.concatenate([A.real, A.imag], axis=1), dtype=np.float64)
    Br = np.concatenate([Bt.real, -Bt.imag], axis=1)
    Bi = np.concatenate([Bt.imag, Bt.real], axis=1)
    Bt2 = np.ascontiguousarray(np.concatenate([Br, Bi], axis=0), dtype=np.float64)
    return A2, Bt2


def complex_gemm_entries(A, Bt, N: int, rows=None, cols=None, mode: int = FAST,
                         single: bool = False):
    """Oracle of the emulated complex product for the entries rows x cols:
    the real oracle on the block form (rows of A2, columns j and n + j)."""
    A2, Bt2 = stack_complex(A, Bt)
    n = np.asarray(Bt).shape[0]
    m = np.asarray(A).shape[0]
    rows = np.arange(m, dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    cols = np.arange(n, dtype=np.int32) if cols is None else np.asarray(cols, np.int32)
    cols2 = np.concatenate([cols, cols + n]).astype(np.int32)
    if mode == ACCURATE:
        e, f = scale_accu(A2, Bt2, N, rows, cols2)
        r = gemm_entries(A2, Bt2, N, rows, cols2, mode=ACCURATE, e=e, f=f, want_X=False,
                         want_c=False, want_G=False, out_f32=single)
    else:
        r = gemm_entries(A2, Bt2, N, rows, cols2, want_X=False, want_c=False, want_G=False,
                         out_f32=single)
    nc = len(cols)
    C = r.C[:, :nc] + 1j * r.C[:, nc:]
    return C.astype(np.complex64 if single else np.complex128), r
