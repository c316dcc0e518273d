"""The benchmark's N > 1 host logic on CPU: two gloo ranks agree on the slowest rank's time, and the
whole-job throughput counts every rank's videos.  (Each rank decodes an independent latent; there is
no collective on the data path, so this is all the multi-rank code there is.)"""
import os
import socket
import zlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _port(name):
    base = 20000 + zlib.crc32(name.encode()) % 10000
    for p in range(base, base + 50):
        with socket.socket() as s:
            try:
                s.bind(("127.0.0.1", p))
                return p
            except OSError:
                continue
    raise RuntimeError("no free port")


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [2.5, 4.0][rank]
        t = bench.max_over_ranks(local, dist, "cpu")
        out[rank] = (t, bench.latent_seed(rank), bench.throughput(72990720, 5, world, t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, _port("multirank"), out), nprocs=2, start_method="spawn", join=True)
        r0, r1 = out[0], out[1]
    assert r0[0] == r1[0] == 4.0
    assert r0[1] != r1[1]                                   # independent videos
    assert r0[2] == pytest.approx(72990720 * 5 * 2 / 4.0 / 1e6)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.throughput(100, 2, 1, 1.0) == pytest.approx(2e-4)
