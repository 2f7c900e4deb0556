"""Thin Python binding of libos2 (include/os2.h).

Argument marshalling only: every step of the emulated GEMM runs in the CUDA
kernels of libos2.  PyTorch provides device memory and streams.  There is no
CPU fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes as ct
import os
import threading

import torch

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE = 0, 1, 2, 3
ERR_NONFINITE, ERR_RANGE, ERR_TIMEOUT, ERR_CUDA, ERR_BOUNDS = 4, 5, 6, 7, 8
MODE_FAST, MODE_ACCURATE = 0, 1
GEMM_TC, GEMM_SIMT, GEMM_TC_1SM, GEMM_TC_I8, GEMM_S8_SYNC = 0, 1, 2, 3, 4
CRT_TC, CRT_SIMT, CRT_AUTO = 0, 1, 2
OUT_MODP_INT8, OUT_RAW_INT32 = 0, 1
KP_ALIGN, CRES_ALIGN = 64, 16

# every function declared in include/os2.h
EXPORTS = ("os2_workspace_size", "os2_gemm", "os2_host_workspace_size", "os2_gemm_host",
           "os2_scale", "os2_residues", "os2_gemm_residues", "os2_crt", "os2_moduli",
           "os2_get_status", "os2_set_gemm_variant", "os2_status_string",
           "os2_gemm_launch_count", "os2_profile_start", "os2_profile_stop",
           "os2_gemm_noalloc", "os2_sgemm", "os2_complex_workspace_size", "os2_zgemm",
           "os2_cgemm", "os2_wait_selftest", "os2_peak_probe", "os2_set_crt_variant",
           "os2_scale_bounds", "os2_exponents_from_bounds", "os2_gemm_exponents")

_lib = None
_lock = threading.Lock()


class Os2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib_path() -> str:
    """The library this process loads: the in-tree build, or the path in the
    environment variable OS2_LIB (for example the debug build)."""
    return os.environ.get("OS2_LIB") or _build.LIB


def load(build_if_missing: bool = True):
    """Load libos2.so (building it first if it is missing and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            if not build_if_missing or path != _build.LIB:
                raise RuntimeError(f"libos2 not built: {path} is missing")
            _build.build()
        L = ct.CDLL(path)
        i, sz, vp, d = ct.c_int, ct.c_size_t, ct.c_void_p, ct.c_void_p
        L.os2_workspace_size.argtypes = [i, i, i, i, i]
        L.os2_workspace_size.restype = sz
        L.os2_host_workspace_size.argtypes = [i, i, i, i, i]
        L.os2_host_workspace_size.restype = sz
        L.os2_gemm.argtypes = [i, i, i, d, i, d, i, d, i, i, i, vp, sz, vp]
        L.os2_gemm.restype = i
        L.os2_gemm_host.argtypes = [i, i, i, d, i, d, i, d, i, i, i, vp, sz, vp]
        L.os2_gemm_host.restype = i
        L.os2_scale.argtypes = [i, i, i, d, i, d, i, i, i, vp, vp, vp, sz, vp]
        L.os2_scale.restype = i
        L.os2_residues.argtypes = [i, i, d, i, vp, i, vp, i, vp]
        L.os2_residues.restype = i
        L.os2_gemm_residues.argtypes = [i, i, i, vp, vp, i, i, i, vp, i, i, vp]
        L.os2_gemm_residues.restype = i
        L.os2_crt.argtypes = [i, i, vp, i, i, vp, vp, d, i, vp, vp]
        L.os2_crt.restype = i
        L.os2_moduli.argtypes = [i, vp]
        L.os2_moduli.restype = i
        L.os2_get_status.argtypes = [vp]
        L.os2_get_status.restype = i
        L.os2_set_gemm_variant.argtypes = [i]
        L.os2_set_gemm_variant.restype = i
        L.os2_status_string.argtypes = [i]
        L.os2_status_string.restype = ct.c_char_p
        L.os2_gemm_launch_count.argtypes = [i, i, i, i, i]
        L.os2_gemm_launch_count.restype = i
        L.os2_profile_start.argtypes = []
        L.os2_profile_start.restype = i
        L.os2_profile_stop.argtypes = [i, vp, vp, vp]
        L.os2_profile_stop.restype = i
        L.os2_gemm_noalloc.argtypes = [i, i, i, d, i, d, i, d, i, i, i, vp]
        L.os2_gemm_noalloc.restype = i
        L.os2_sgemm.argtypes = [i, i, i, d, i, d, i, d, i, i, i, vp, sz, vp]
        L.os2_sgemm.restype = i
        L.os2_complex_workspace_size.argtypes = [i, i, i, i, i, i]
        L.os2_complex_workspace_size.restype = sz
        L.os2_zgemm.argtypes = [i, i, i, d, i, d, i, d, i, i, i, vp, sz, vp]
        L.os2_zgemm.restype = i
        L.os2_cgemm.argtypes = [i, i, i, d, i, d, i, d, i, i, i, vp, sz, vp]
        L.os2_wait_selftest.argtypes = [ct.c_longlong, vp, vp]
        L.os2_wait_selftest.restype = i
        L.os2_cgemm.restype = i
        L.os2_peak_probe.argtypes = [i, i, i, vp, ct.POINTER(ct.c_double), vp]
        L.os2_peak_probe.restype = i
        L.os2_set_crt_variant.argtypes = [i]
        L.os2_set_crt_variant.restype = i
        L.os2_scale_bounds.argtypes = [i, i, i, d, i, d, i, vp, vp, vp, vp, vp, sz, vp]
        L.os2_scale_bounds.restype = i
        L.os2_exponents_from_bounds.argtypes = [i, vp, vp, i, vp, vp]
        L.os2_exponents_from_bounds.restype = i
        L.os2_gemm_exponents.argtypes = [i, i, i, d, i, d, i, d, i, i, vp, vp, vp, sz, vp]
        L.os2_gemm_exponents.restype = i
        _lib = L
        return L


def status_string(st: int) -> str:
    return load().os2_status_string(int(st)).decode()


def _check(st: int, where: str):
    if st != OK:
        raise Os2Error(st, where)


def _mode(mode) -> int:
    if isinstance(mode, str):
        return {"fast": MODE_FAST, "accurate": MODE_ACCURATE}[mode]
    return int(mode)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _kmat(X, name):
    """float64 CUDA matrix whose rows are contiguous; returns (X, ld)."""
    if not (X.is_cuda and X.dtype == torch.float64 and X.dim() == 2 and
            (X.stride(1) == 1 or X.shape[1] <= 1)):
        raise ValueError(f"{name} must be a 2-D float64 CUDA tensor with contiguous rows")
    return X, max(X.stride(0), max(X.shape[1], 1))


def moduli(num_moduli: int) -> list[int]:
    out = (ct.c_int32 * 20)()
    n = load().os2_moduli(num_moduli, out)
    if n != num_moduli:
        raise Os2Error(ERR_INVALID_ARG, "os2_moduli")
    return list(out[:n])


def workspace_size(m, n, k, num_moduli, mode="fast") -> int:
    return int(load().os2_workspace_size(m, n, k, num_moduli, _mode(mode)))


def host_workspace_size(m, n, k, num_moduli, mode="fast") -> int:
    return int(load().os2_host_workspace_size(m, n, k, num_moduli, _mode(mode)))


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Caller-owned device workspace (torch allocation, 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device or "cuda")


def launch_count(m, n, k, num_moduli, mode="fast") -> int:
    return int(load().os2_gemm_launch_count(m, n, k, num_moduli, _mode(mode)))


def set_gemm_variant(variant: int):
    _check(load().os2_set_gemm_variant(int(variant)), "os2_set_gemm_variant")


def set_crt_variant(variant: int):
    """Kernel of steps 4 + 5: CRT_TC (tensor-core limb sums), CRT_SIMT
    (CUDA-core multiply-adds) or CRT_AUTO (the default: CUDA cores beside a
    product, tensor cores alone); results are bit-identical."""
    _check(load().os2_set_crt_variant(int(variant)), "os2_set_crt_variant")


def get_status(stream=None) -> int:
    return int(load().os2_get_status(_stream(stream)))


PROBE_F16_1SM, PROBE_F16_2SM, PROBE_S8_SYNC = 0, 1, 2


def peak_probe(kind: int, iters: int, check: bool = False, stream=None):
    """Enqueue one pipe-peak probe launch (see os2_peak_probe).  Returns the
    flop it performs; with check=True it synchronises and returns
    (flop, mismatches, ctas_checked) instead."""
    fl = ct.c_double(0.0)
    res = torch.zeros(4, dtype=torch.int32, device="cuda") if check else None
    _check(load().os2_peak_probe(int(kind), int(iters), 1 if check else 0,
                                 _ptr(res) if check else None, ct.byref(fl), _stream(stream)),
           "os2_peak_probe")
    if not check:
        return fl.value
    torch.cuda.synchronize()
    r = res.cpu().tolist()
    return fl.value, int(r[0]), int(r[1])


def wait_selftest(limit_cycles: int = 2_000_000, stream=None) -> list[int]:
    """Failure-detection self-test: one CTA whose bounded mbarrier waits run out
    after `limit_cycles` clock cycles.  Returns the kernel's eight result words
    (see os2_wait_selftest); the device status word is left at ERR_TIMEOUT."""
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    _check(load().os2_wait_selftest(int(limit_cycles), _ptr(out), _stream(stream)),
           "os2_wait_selftest")
    torch.cuda.synchronize()
    return [int(v) for v in out.cpu()]

def gemm(A: torch.Tensor, Bt: torch.Tensor, num_moduli: int = 14, mode="fast", out=None,
         workspace=None, stream=None) -> torch.Tensor:
    """C = A @ Bt.T emulated with Ozaki Scheme II.

    A: m x k, Bt: n x k (B = Bt.T in column-major form), float64 CUDA tensors
    with contiguous rows.  Returns C (m x n, float64)."""
    A, lda = _kmat(A, "A")
    Bt, ldb = _kmat(Bt, "Bt")
    m, k = A.shape
    n = Bt.shape[0]
    if Bt.shape[1] != k:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((m, n), dtype=torch.float64, device=A.device)
    ldc = max(out.stride(0), max(n, 1))
    need = workspace_size(m, n, k, num_moduli, mode)
    if workspace is None:
        workspace = alloc_workspace(need, A.device)
    st = load().os2_gemm(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, _ptr(out), ldc, num_moduli,
                         _mode(mode), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "os2_gemm")
    return out


def sgemm(A: torch.Tensor, Bt: torch.Tensor, num_moduli: int = 7, mode="fast", out=None,
          workspace=None, stream=None) -> torch.Tensor:
    """C = A @ Bt.T for float32 operands (SGEMM emulation); layouts as in gemm."""
    for X, nm in ((A, "A"), (Bt, "Bt")):
        if not (X.is_cuda and X.dtype == torch.float32 and X.dim() == 2 and X.stride(1) == 1):
            raise ValueError(f"{nm} must be a 2-D float32 CUDA tensor with contiguous rows")
    m, k = A.shape
    n = Bt.shape[0]
    if Bt.shape[1] != k:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=A.device)
    need = workspace_size(m, n, k, num_moduli, mode)
    if workspace is None:
        workspace = alloc_workspace(need, A.device)
    st = load().os2_sgemm(m, n, k, _ptr(A), max(A.stride(0), max(k, 1)), _ptr(Bt),
                          max(Bt.stride(0), max(k, 1)), _ptr(out), max(out.stride(0), max(n, 1)),
                          num_moduli, _mode(mode), _ptr(workspace), workspace.numel(),
                          _stream(stream))
    _check(st, "os2_sgemm")
    return out


def complex_workspace_size(m, n, k, num_moduli, mode="fast", single=False) -> int:
    return int(load().os2_complex_workspace_size(m, n, k, num_moduli, _mode(mode), int(single)))


def zgemm(A: torch.Tensor, Bt: torch.Tensor, num_moduli: int = 16, mode="fast", out=None,
          workspace=None, stream=None) -> torch.Tensor:
    """C = A @ Bt.T for complex operands (complex128 -> ZGEMM, complex64 -> CGEMM).

    A: m x k, Bt: n x k (B = Bt.T column-major), complex CUDA tensors with
    contiguous rows (interleaved re/im).  Returns C (m x n) of the same dtype."""
    if A.dtype not in (torch.complex128, torch.complex64) or Bt.dtype != A.dtype:
        raise ValueError("A and Bt must both be complex128 or both complex64")
    for X, nm in ((A, "A"), (Bt, "Bt")):
        if not (X.is_cuda and X.dim() == 2 and X.stride(1) == 1):
            raise ValueError(f"{nm} must be a 2-D CUDA tensor with contiguous rows")
    single = A.dtype == torch.complex64
    m, k = A.shape
    n = Bt.shape[0]
    if Bt.shape[1] != k:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((m, n), dtype=A.dtype, device=A.device)
    if workspace is None:
        workspace = alloc_workspace(complex_workspace_size(m, n, k, num_moduli, mode, single),
                                    A.device)
    fn = load().os2_cgemm if single else load().os2_zgemm
    st = fn(m, n, k, _ptr(A), max(A.stride(0), max(k, 1)), _ptr(Bt), max(Bt.stride(0), max(k, 1)),
            _ptr(out), max(out.stride(0), max(n, 1)), num_moduli, _mode(mode), _ptr(workspace),
            workspace.numel(), _stream(stream))
    _check(st, "os2_cgemm" if single else "os2_zgemm")
    return out


def matmul(A: torch.Tensor, B: torch.Tensor, num_moduli: int = 14, mode="fast") -> torch.Tensor:
    """Convenience: C = A @ B for a row-major k x n B (copied to column-major)."""
    return gemm(A.contiguous(), B.t().contiguous(), num_moduli, mode)


def gemm_host(A, Bt, C, num_moduli=14, mode="fast", workspace=None, stream=None):
    """End-to-end call on HOST tensors (pinned for asynchronous copies): copies
    in, five steps, copy out, all enqueued on `stream`; synchronise before use."""
    for X, nm in ((A, "A"), (Bt, "Bt"), (C, "C")):
        if X.is_cuda or X.dtype != torch.float64 or X.dim() != 2 or (
                X.stride(1) != 1 and X.shape[1] > 1):
            raise ValueError(f"{nm} must be a 2-D float64 host tensor with contiguous rows")
    m, k = A.shape
    n = Bt.shape[0]
    need = host_workspace_size(m, n, k, num_moduli, mode)
    if workspace is None:
        workspace = alloc_workspace(need)
    st = load().os2_gemm_host(m, n, k, _ptr(A), max(A.stride(0), max(k, 1)), _ptr(Bt),
                              max(Bt.stride(0), max(k, 1)), _ptr(C), max(C.stride(0), max(n, 1)),
                              num_moduli, _mode(mode), _ptr(workspace), workspace.numel(),
                              _stream(stream))
    _check(st, "os2_gemm_host")
    return C


def scale(A, Bt, num_moduli=14, mode="fast", stream=None):
    """Step 1: exponents (e for rows of A, f for columns of B), int32 tensors."""
    A, lda = _kmat(A, "A")
    Bt, ldb = _kmat(Bt, "Bt")
    m, k = A.shape
    n = Bt.shape[0]
    e = torch.empty(m, dtype=torch.int32, device=A.device)
    f = torch.empty(n, dtype=torch.int32, device=A.device)
    ws = None
    nbytes = 0
    if _mode(mode) == MODE_ACCURATE:
        nbytes = workspace_size(m, n, k, 1, mode)
        ws = alloc_workspace(nbytes, A.device)
    st = load().os2_scale(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, num_moduli, _mode(mode),
                          _ptr(e), _ptr(f), _ptr(ws), nbytes, _stream(stream))
    _check(st, "os2_scale")
    return e, f


def residues(X, exps, num_moduli, ldp=None, stream=None) -> torch.Tensor:
    """Step 2: FP16 residue planes [N, rows, ldp] of trunc(X * 2^exps)."""
    X, ldx = _kmat(X, "X")
    rows, k = X.shape
    if ldp is None:
        ldp = (max(k, 1) + KP_ALIGN - 1) // KP_ALIGN * KP_ALIGN
    planes = torch.empty((num_moduli, rows, ldp), dtype=torch.float16, device=X.device)
    exps = exps.to(torch.int32).contiguous()
    st = load().os2_residues(rows, k, _ptr(X), ldx, _ptr(exps), num_moduli, _ptr(planes), ldp,
                             _stream(stream))
    _check(st, "os2_residues")
    return planes


def gemm_residues(RA, RB, k, out_kind=OUT_MODP_INT8, variant=GEMM_TC, stream=None):
    """Step 3: N residue products of FP16 planes RA [N,m,ldp], RB [N,n,ldp]
    (int8 planes for GEMM_S8_SYNC).
    Returns int8 [N, m, ldo] (mod p, symmetric) or int32 [N, m, ldo] (raw)."""
    N, m, ldp = RA.shape
    n = RB.shape[1]
    want = torch.int8 if variant == GEMM_S8_SYNC else torch.float16
    if RA.dtype != want or RB.dtype != want:
        raise TypeError(f"gemm_residues: variant {variant} takes {want} planes, got "
                        f"{RA.dtype} and {RB.dtype}")
    if out_kind == OUT_MODP_INT8:
        ldo = (max(n, 1) + CRES_ALIGN - 1) // CRES_ALIGN * CRES_ALIGN
        out = torch.empty((N, m, ldo), dtype=torch.int8, device=RA.device)
    else:
        ldo = (max(n, 1) + 3) // 4 * 4
        out = torch.empty((N, m, ldo), dtype=torch.int32, device=RA.device)
    st = load().os2_gemm_residues(m, n, k, _ptr(RA), _ptr(RB), ldp, N, out_kind, _ptr(out), ldo,
                                  variant, _stream(stream))
    _check(st, "os2_gemm_residues")
    return out


def crt(cres, n, e, f, want_X=False, stream=None):
    """Steps 4-5 from int8 residues [N, m, ldcres]; returns C (and X limbs)."""
    N, m, ldcres = cres.shape
    C = torch.empty((m, n), dtype=torch.float64, device=cres.device)
    X = torch.empty((m, n, 8), dtype=torch.int32, device=cres.device) if want_X else None
    st = load().os2_crt(m, n, _ptr(cres), ldcres, N, _ptr(e.to(torch.int32).contiguous()),
                        _ptr(f.to(torch.int32).contiguous()), _ptr(C), max(n, 1), _ptr(X),
                        _stream(stream))
    _check(st, "os2_crt")
    return (C, X) if want_X else C


def profile_start():
    """Start per-kernel CUDA-event timing of os2_gemm launches."""
    _check(load().os2_profile_start(), "os2_profile_start")


def profile_stop() -> dict:
    """Stop timing; returns {kernel role: (total_ms, launches)}."""
    names = ct.create_string_buffer(32 * 16)
    tot = (ct.c_double * 16)()
    cnt = (ct.c_int * 16)()
    n = load().os2_profile_stop(16, names, tot, cnt)
    if n < 0:
        raise Os2Error(ERR_CUDA, "os2_profile_stop")
    raw = names.raw
    return {raw[32 * i:32 * i + 32].split(b"\0")[0].decode(): (tot[i], cnt[i]) for i in range(n)}


def scale_bounds(A: torch.Tensor, Bt: torch.Tensor, workspace=None, stream=None):
    """Accurate-mode bound maxima of a block: (R, K, EA, EB), int32 CUDA
    tensors (see os2_scale_bounds)."""
    A, lda = _kmat(A, "A")
    Bt, ldb = _kmat(Bt, "Bt")
    m, k = A.shape
    n = Bt.shape[0]
    dev = A.device
    R = torch.empty(m, dtype=torch.int32, device=dev)
    K = torch.empty(n, dtype=torch.int32, device=dev)
    EA = torch.empty(m, dtype=torch.int32, device=dev)
    EB = torch.empty(n, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(m, n, k, 1, "accurate"), dev)
    _check(load().os2_scale_bounds(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, _ptr(R), _ptr(K),
                                   _ptr(EA), _ptr(EB), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "os2_scale_bounds")
    return R, K, EA, EB


def exponents_from_bounds(bound: torch.Tensor, E: torch.Tensor, num_moduli: int, stream=None):
    """Accurate-mode exponents from bounds and exponent bases (int32 CUDA)."""
    bound = bound.to(torch.int32).contiguous()
    E = E.to(torch.int32).contiguous()
    e = torch.empty_like(E)
    _check(load().os2_exponents_from_bounds(bound.numel(), _ptr(bound), _ptr(E), int(num_moduli),
                                            _ptr(e), _stream(stream)), "os2_exponents_from_bounds")
    return e


def gemm_exponents(A: torch.Tensor, Bt: torch.Tensor, num_moduli: int, e: torch.Tensor,
                   f: torch.Tensor, out=None, workspace=None, stream=None) -> torch.Tensor:
    """Steps 2-5 with given exponents e (rows of A) and f (columns = rows of Bt)."""
    A, lda = _kmat(A, "A")
    Bt, ldb = _kmat(Bt, "Bt")
    m, k = A.shape
    n = Bt.shape[0]
    C = out if out is not None else torch.empty((m, n), dtype=torch.float64, device=A.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(m, n, k, num_moduli, "fast"), A.device)
    e = e.to(torch.int32).contiguous()
    f = f.to(torch.int32).contiguous()
    _check(load().os2_gemm_exponents(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, _ptr(C), C.stride(0),
                                     int(num_moduli), _ptr(e), _ptr(f), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "os2_gemm_exponents")
    return C


NOALLOC_SCRATCH_BYTES = 128 << 20


def gemm_noalloc(A: torch.Tensor, Bt: torch.Tensor, num_moduli: int = 14, mode="fast", out=None,
                 stream=None) -> torch.Tensor:
    """C = A @ Bt.T like ``gemm``, for callers that cannot allocate device
    memory at the call: the scratch is a fixed 128 MiB array inside libos2
    (shared by every call; serialise calls that could overlap on the GPU).
    ``out`` must be given by such callers; the default allocates it here."""
    A, lda = _kmat(A, "A")
    Bt, ldb = _kmat(Bt, "Bt")
    m, k = A.shape
    n = Bt.shape[0]
    if Bt.shape[1] != k:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty((m, n), dtype=torch.float64, device=A.device)
    ldc = max(out.stride(0), max(n, 1))
    st = load().os2_gemm_noalloc(m, n, k, _ptr(A), lda, _ptr(Bt), ldb, _ptr(out), ldc,
                                 num_moduli, _mode(mode), _stream(stream))
    _check(st, "os2_gemm_noalloc")
    return out
