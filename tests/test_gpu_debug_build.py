"""The debug build (OS2_DEBUG): every kernel checks its hand-computed global
indices against the extent of the array they address, records
OS2_ERR_BOUNDS on a failure and skips the access.  Built here, loaded in a
fresh process (OS2_LIB), and run over small parity shapes -- both modes, both
CRT kernels, row panels, the host entry point, the int8-plane variants, SGEMM
and the CRT alone: every status must stay clean and every result must equal
the oracle's bits."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import numpy as np, torch
import rns_emulated_fp64_gb300 as os2
import workloads
from oracle import oracle as orc
assert os2.binding.lib_path().endswith("_build_debug/libos2.so"), os2.binding.lib_path()

def same(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint64), np.ascontiguousarray(b).view(np.uint64))

def check(C, A, Bt, N, mode, rows=None, cols=None):
    st = os2.get_status()
    assert st == 0, os2.status_string(st)
    ref = orc.gemm_entries(A, Bt, N, rows, cols, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    got = C if rows is None else C[np.ix_(rows, cols)]
    assert same(got, ref.C)

dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
for (m, n, k) in [(64, 64, 64), (3, 5, 7), (129, 257, 65), (300, 520, 1000), (130, 140, 1921)]:
    A, Bt = workloads.make_pair("spread", m, n, k, seed=k, phi=1.0)
    for mode in ("fast", "accurate"):
        for crt in (os2.CRT_TC, os2.CRT_SIMT):
            os2.set_crt_variant(crt)
            check(os2.gemm(dev(A), dev(Bt), 14, mode).cpu().numpy(), A, Bt, 14, mode)
os2.set_crt_variant(os2.CRT_AUTO)
m, n, k = 4100, 200, 300
A, Bt = workloads.make_pair("spread", m, n, k, seed=3, phi=2.0)
rows, cols = workloads.sample_grid(m, n, 24, seed=1)
for mode in ("fast", "accurate"):
    check(os2.gemm(dev(A), dev(Bt), 16, mode).cpu().numpy(), A, Bt, 16, mode, rows, cols)
    Ch = torch.empty((m, n), dtype=torch.float64).pin_memory()
    os2.gemm_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(Bt).pin_memory(), Ch, 16, mode)
    torch.cuda.synchronize()
    check(Ch.numpy(), A, Bt, 16, mode, rows, cols)
os2.set_gemm_variant(os2.GEMM_TC_I8)
check(os2.gemm(dev(A), dev(Bt), 16, "fast").cpu().numpy(), A, Bt, 16, "fast", rows, cols)
os2.set_gemm_variant(os2.GEMM_S8_SYNC)
check(os2.gemm(dev(A), dev(Bt), 16, "fast").cpu().numpy(), A, Bt, 16, "fast", rows, cols)
Ch = torch.empty((m, n), dtype=torch.float64).pin_memory()
os2.gemm_host(torch.from_numpy(A).pin_memory(), torch.from_numpy(Bt).pin_memory(), Ch, 16, "accurate")
torch.cuda.synchronize()
check(Ch.numpy(), A, Bt, 16, "accurate", rows, cols)
os2.set_gemm_variant(os2.GEMM_TC_1SM)
check(os2.gemm(dev(A), dev(Bt), 16, "accurate").cpu().numpy(), A, Bt, 16, "accurate", rows, cols)
os2.set_gemm_variant(os2.GEMM_TC)
A32, B32 = A.astype(np.float32), Bt.astype(np.float32)
C = os2.sgemm(dev(A32), dev(B32), 7, "fast").cpu().numpy()
assert os2.get_status() == 0
ref = orc.gemm_entries(A32, B32, 7, rows, cols, want_X=False, want_c=False, want_G=False, out_f32=True)
assert np.array_equal(C[np.ix_(rows, cols)].view(np.uint32), ref.C.view(np.uint32))
# the CRT alone, rows not a multiple of 16 bytes (CUDA-core kernel) and aligned (tensor cores)
A, Bt = workloads.make_pair("spread", 37, 45, 90, seed=2, phi=2.0)
ref = orc.gemm_entries(A, Bt, 16)
for ld in (48, 52):
    cres = np.zeros((16, 37, ld), np.int8)
    cres[:, :, :45] = np.transpose(ref.c, (2, 0, 1))
    C = os2.crt(dev(cres), 45, dev(ref.e), dev(ref.f)).cpu().numpy()
    assert os2.get_status() == 0
    assert same(C, ref.C)
print("debug build clean")
'''


def test_debug_build_index_checks_stay_clean():
    from rns_emulated_fp64_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, OS2_LIB=lib)
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build clean" in r.stdout
