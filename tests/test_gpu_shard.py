"""The entry points of the output-block split (os2_scale_bounds,
os2_exponents_from_bounds, os2_gemm_exponents) on one GPU: the blocks of a
2 x 3 grid are computed one after another, their bound maxima reduced with a
MAX across the blocks of each grid row and column (torch on the device, no
collective kernel), and the assembled C must equal os2_gemm on the whole
product bit for bit, and the oracle on a sample."""
import numpy as np
import pytest
import torch

import rns_emulated_fp64_gb300 as os2
import workloads
from oracle import oracle as orc
from rns_emulated_fp64_gb300 import shard

pytestmark = pytest.mark.gpu


def test_scale_bounds_match_oracle():
    m, n, k, N = 133, 75, 300, 16
    A, Bt = workloads.make_pair("spread", m, n, k, seed=3, phi=2.5)
    A[7] = 0.0
    R, K, EA, EB = os2.scale_bounds(torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda())
    assert os2.get_status() == 0
    e, f, Rr, Kr = orc.scale_accu(A, Bt, N, return_bounds=True)
    assert np.array_equal(R.cpu().numpy(), Rr) and np.array_equal(K.cpu().numpy(), Kr)
    assert np.array_equal(EA.cpu().numpy(), orc.row_exponents(A))
    assert np.array_equal(EB.cpu().numpy(), orc.row_exponents(Bt))
    ed = os2.exponents_from_bounds(R, EA, N)
    fd = os2.exponents_from_bounds(K, EB, N)
    assert np.array_equal(ed.cpu().numpy(), e) and np.array_equal(fd.cpu().numpy(), f)


@pytest.mark.parametrize("mode", ["fast", "accurate"])
def test_block_grid_equals_whole_product(mode):
    m, n, k, N = 611, 533, 257, 16
    A, Bt = workloads.make_pair("spread", m, n, k, seed=9, phi=3.0)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
    whole = os2.gemm(Ad, Bd, N, mode)
    world = 6
    grids = [shard.Grid(m, n, r, world) for r in range(world)]
    pr, pc = grids[0].pr, grids[0].pc
    C = torch.full((m, n), float("nan"), dtype=torch.float64, device="cuda")
    if mode == "fast":
        for g in grids:
            (r0, r1), (c0, c1) = g.rows, g.cols
            C[r0:r1, c0:c1] = os2.gemm(Ad[r0:r1], Bd[c0:c1], N, "fast")
    else:
        parts = {}
        for g in grids:
            (r0, r1), (c0, c1) = g.rows, g.cols
            parts[(g.a, g.b)] = os2.scale_bounds(Ad[r0:r1], Bd[c0:c1])
        for g in grids:
            (r0, r1), (c0, c1) = g.rows, g.cols
            R = torch.stack([parts[(g.a, b)][0] for b in range(pc)]).amax(0)  # over the grid row
            K = torch.stack([parts[(a, g.b)][1] for a in range(pr)]).amax(0)  # over the grid column
            e = os2.exponents_from_bounds(R, parts[(g.a, g.b)][2], N)
            f = os2.exponents_from_bounds(K, parts[(g.a, g.b)][3], N)
            C[r0:r1, c0:c1] = os2.gemm_exponents(Ad[r0:r1].contiguous(), Bd[c0:c1].contiguous(),
                                                 N, e, f)
    assert os2.get_status() == 0
    assert torch.equal(C.view(torch.int64), whole.view(torch.int64))
    rows, cols = workloads.sample_grid(m, n, 24, seed=2)
    ref = orc.gemm_entries(A, Bt, N, rows, cols, mode=orc.FAST if mode == "fast" else orc.ACCURATE,
                           want_X=False, want_c=False, want_G=False)
    got = C.cpu().numpy()[np.ix_(rows, cols)]
    assert np.array_equal(got.view(np.uint64), ref.C.view(np.uint64))
