"""Output-block sharding of one product (rns_emulated_fp64_gb300.shard) on CPU
with gloo ranks, checked against the oracle of the unsplit product.

Each rank owns a row block of A and a column block of B.  Fast mode needs no
collective: the oracle on a block gives the unsplit product's entries.
Accurate mode: each rank takes the bound maxima over its own block; after the
MAX-allreduce over its grid row (R) and grid column (K) they must equal the
unsplit oracle's bounds, and so must the exponents and the entries."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads
from oracle import oracle as orc
from rns_emulated_fp64_gb300 import shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [1, 2, 3, 4, 6, 8])
def test_grid_blocks_partition_the_output(world):
    m, n = 37, 29
    cover = np.zeros((m, n), np.int32)
    for rank in range(world):
        g = shard.Grid(m, n, rank, world)
        assert g.pr * g.pc == world and g.pr <= g.pc
        cover[g.rows[0]:g.rows[1], g.cols[0]:g.cols[1]] += 1
    assert np.all(cover == 1)


def _worker(rank, world, port, N, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m, n, k = 37, 29, 70
        A, Bt = workloads.make_pair("spread", m, n, k, seed=5, phi=3.0)
        g = shard.Grid.current(m, n, backend="gloo")
        r0, r1 = g.rows
        c0, c1 = g.cols
        Ab, Bb = np.ascontiguousarray(A[r0:r1]), np.ascontiguousarray(Bt[c0:c1])
        # accurate mode: block bounds, reduced over the grid row / column
        _, _, Rb, Kb = orc.scale_accu(Ab, Bb, N, return_bounds=True)
        R = torch.from_numpy(Rb.copy())
        K = torch.from_numpy(Kb.copy())
        shard.reduce_bounds(R, K, g)
        e = orc.exps_from_bounds(R.numpy(), orc.row_exponents(Ab), N)
        f = orc.exps_from_bounds(K.numpy(), orc.row_exponents(Bb), N)
        e_local = orc.exps_from_bounds(Rb, orc.row_exponents(Ab), N)
        f_local = orc.exps_from_bounds(Kb, orc.row_exponents(Bb), N)
        acc = orc.gemm_entries(Ab, Bb, N, mode=orc.ACCURATE, e=e, f=f, want_X=False,
                               want_c=False, want_G=False)
        fast = orc.gemm_entries(Ab, Bb, N, want_X=False, want_c=False, want_G=False)
        out[rank] = dict(rows=(r0, r1), cols=(c0, c1), R=R.numpy(), K=K.numpy(), e=e, f=f,
                         changed=bool(np.any(e != e_local) or np.any(f != f_local)),
                         C_acc=acc.C, C_fast=fast.C, bad=acc.mismatches + fast.mismatches)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_product_equals_unsplit_oracle(world):
    N = 14
    orc.load()  # built before the ranks start
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), N, out), nprocs=world, join=True)
    m, n, k = 37, 29, 70
    A, Bt = workloads.make_pair("spread", m, n, k, seed=5, phi=3.0)
    e, f, R, K = orc.scale_accu(A, Bt, N, return_bounds=True)
    acc = orc.gemm_entries(A, Bt, N, mode=orc.ACCURATE, want_X=False, want_c=False, want_G=False)
    fast = orc.gemm_entries(A, Bt, N, want_X=False, want_c=False, want_G=False)
    changed = False
    for rank in range(world):
        d = out[rank]
        (r0, r1), (c0, c1) = d["rows"], d["cols"]
        assert d["bad"] == 0
        assert np.array_equal(d["R"], R[r0:r1]) and np.array_equal(d["K"], K[c0:c1])
        assert np.array_equal(d["e"], e[r0:r1]) and np.array_equal(d["f"], f[c0:c1])
        assert np.array_equal(d["C_acc"].view(np.uint64), acc.C[r0:r1, c0:c1].view(np.uint64))
        assert np.array_equal(d["C_fast"].view(np.uint64), fast.C[r0:r1, c0:c1].view(np.uint64))
        changed |= d["changed"]
    # the reduction matters for these inputs: block-local bounds alone would
    # have given other exponents somewhere
    assert changed
