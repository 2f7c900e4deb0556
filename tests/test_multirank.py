"""Host-side logic of the multi-rank benchmark path, on CPU with gloo
(world size 2): each rank runs its own problem (weak scaling, no data
collective); the timing is the max over ranks and the reported value is the
whole-job throughput.  The reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 * (rank + 1)          # rank 1 is the slow one
        flop = 2.0 * 8192 ** 3
        ms_max, value = bench.aggregate(world, ms_local, flop, steps=5, device="cpu")
        out[rank] = (ms_max, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_weak_scaling_aggregate_two_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    flop = 2.0 * 8192 ** 3
    for rank in range(world):
        ms_max, value = out[rank]
        assert ms_max == 20.0
        assert value == pytest.approx(world * flop * 5 / 0.020 / 1e12)


def test_single_rank_aggregate_is_local():
    ms, v = bench.aggregate(1, 12.5, 2.0 * 1024 ** 3, 4, device="cpu")
    assert ms == 12.5 and v == pytest.approx(2.0 * 1024 ** 3 * 4 / 0.0125 / 1e12)


def test_reference_arm_only_on_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    import argparse
    ns = argparse.Namespace(m=64, n=64, k=64, num_moduli=14, mode="fast", phi=0.5, steps=1,
                            warmup=0)
    bench.run_reference(ns)
    assert capsys.readouterr().out == ""
