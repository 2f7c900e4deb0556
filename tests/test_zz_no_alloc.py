"""os2_gemm_noalloc: the emulated DGEMM for callers that cannot allocate
device memory where they call it (a plugin or host library whose device
memory is owned by another allocator and has no workspace to pass, or a
latency-critical loop that must not call cudaMalloc/cudaFree because those
can synchronise the whole device).  Its scratch is a fixed array inside
libos2.  Checked against os2_gemm (caller-supplied workspace) through the C
ABI, bit for bit, on two calls in a row.

Named so that pytest collects it last."""
import ctypes as ct

import numpy as np
import pytest
import torch

import rns_emulated_fp64_gb300 as os2
import workloads
from rns_emulated_fp64_gb300 import binding

pytestmark = pytest.mark.gpu


def _noalloc(A, Bt, C, N, mode):
    lib = os2.load()
    m, k = A.shape
    n = Bt.shape[0]
    return lib.os2_gemm_noalloc(m, n, k, A.data_ptr(), k, Bt.data_ptr(), k, C.data_ptr(), n, N,
                                mode, ct.c_void_p(torch.cuda.current_stream().cuda_stream))


def _with_workspace(A, Bt, N, mode):
    lib = os2.load()
    m, k = A.shape
    n = Bt.shape[0]
    C = torch.empty((m, n), dtype=torch.float64, device="cuda")
    ws = os2.alloc_workspace(os2.workspace_size(m, n, k, N, mode))
    st = lib.os2_gemm(m, n, k, A.data_ptr(), k, Bt.data_ptr(), k, C.data_ptr(), n, N, mode,
                      ws.data_ptr(), ws.numel(), ct.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, os2.status_string(st)
    return C


@pytest.mark.parametrize("mode", [binding.MODE_FAST, binding.MODE_ACCURATE])
def test_noalloc_matches_workspace_entry_point_twice(mode):
    cases = [("spread", 300, 260, 700, 16, 2.0, 3), ("normal", 129, 517, 1000, 20, 0.0, 4)]
    for kind, m, n, k, N, phi, seed in cases:          # two calls in a row, different shapes
        A, Bt = workloads.make_pair(kind, m, n, k, seed=seed, phi=phi)
        Ad = torch.from_numpy(A).cuda()
        Bd = torch.from_numpy(Bt).cuda()
        C = torch.full((m, n), np.nan, dtype=torch.float64, device="cuda")
        st = _noalloc(Ad, Bd, C, N, mode)
        assert st == 0, os2.status_string(st)
        assert os2.get_status() == 0
        want = _with_workspace(Ad, Bd, N, mode)
        assert os2.get_status() == 0
        got = C.cpu().numpy()
        ref = want.cpu().numpy()
        assert np.array_equal(got.view(np.uint64), ref.view(np.uint64)), \
            f"{np.count_nonzero(got != ref)} entries differ"


def test_noalloc_larger_then_smaller_calls():
    """The shared array keeps the previous call's contents.  A large call (many
    rows, the largest planes) followed by smaller ones, among them an accurate
    product with k > 4096 whose bound product keeps int32 partial sums between
    its 4096-term segments in the array, must still equal os2_gemm bit for bit:
    every call clears what it needs.  9000 x 72 x 96 is a shape os2_gemm would
    cut into row panels; the no-alloc entry point runs it in one pass."""
    cases = [("spread", 9000, 72, 96, 20, binding.MODE_FAST, 1.0, 7),
             ("spread", 200, 200, 5000, 16, binding.MODE_ACCURATE, 2.0, 8),
             ("normal", 65, 33, 17, 14, binding.MODE_ACCURATE, 0.0, 9),
             ("spread", 200, 200, 5000, 16, binding.MODE_ACCURATE, 4.0, 10)]
    for kind, m, n, k, N, mode, phi, seed in cases:
        assert os2.workspace_size(m, n, k, N, mode) <= binding.NOALLOC_SCRATCH_BYTES
        A, Bt = workloads.make_pair(kind, m, n, k, seed=seed, phi=phi)
        Ad = torch.from_numpy(A).cuda()
        Bd = torch.from_numpy(Bt).cuda()
        C = torch.full((m, n), np.nan, dtype=torch.float64, device="cuda")
        st = _noalloc(Ad, Bd, C, N, mode)
        assert st == 0, os2.status_string(st)
        assert os2.get_status() == 0
        want = _with_workspace(Ad, Bd, N, mode)
        assert os2.get_status() == 0
        got = C.cpu().numpy()
        ref = want.cpu().numpy()
        assert np.array_equal(got.view(np.uint64), ref.view(np.uint64)), \
            f"{m}x{n}x{k}: {np.count_nonzero(got != ref)} entries differ"


def test_noalloc_k_zero_beyond_scratch_zeroes_c():
    """k = 0 touches no scratch, so sizes whose workspace would exceed the
    array are accepted, as os2_gemm accepts them: C becomes 0."""
    m = n = 4096
    assert os2.workspace_size(m, n, 0, 20) > binding.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((m, 1), dtype=torch.float64, device="cuda")
    C = torch.full((m, n), np.nan, dtype=torch.float64, device="cuda")
    lib = os2.load()
    st = lib.os2_gemm_noalloc(m, n, 0, A.data_ptr(), 1, A.data_ptr(), 1, C.data_ptr(), n, 20,
                              binding.MODE_FAST,
                              ct.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, os2.status_string(st)
    assert os2.get_status() == 0
    assert bool((C == 0).all())


def test_noalloc_rejects_problems_beyond_its_scratch():
    m = n = k = 2048
    N = 7
    assert os2.workspace_size(m, n, k, N) > binding.NOALLOC_SCRATCH_BYTES
    A = torch.zeros((m, k), dtype=torch.float64, device="cuda")
    C = torch.zeros((m, n), dtype=torch.float64, device="cuda")
    assert _noalloc(A, A, C, N, binding.MODE_FAST) == binding.ERR_WORKSPACE
    assert os2.workspace_size(m, n, k, 6) <= binding.NOALLOC_SCRATCH_BYTES
