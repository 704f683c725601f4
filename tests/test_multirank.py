"""The benchmark's multi-rank host logic on CPU with gloo, world size 2:
ranks own disjoint sequences whose inputs equal the single-process draw, and
the reported time is the maximum over ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from ssm_recurrence_verify_b300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = synth.custom_workload(3, 4, 16, 16, 2, 3, synth.BF16, seed=21)
    batch, offset = bench.shard(wl.batch, rank)
    d = synth.draw_layer_round(wl, batch=batch, batch_offset=offset)
    out[rank] = {"offset": offset, "x": d["x"], "state0": d["state0"], "accept_len": d["accept_len"],
                 "max": bench.max_over_ranks(10.0 + rank, world)}
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_rank_sharding_and_max():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    wl = synth.custom_workload(6, 4, 16, 16, 2, 3, synth.BF16, seed=21)
    full = synth.draw_layer_round(wl)
    assert res[0]["offset"] == 0 and res[1]["offset"] == 3
    for r in (0, 1):
        sl = slice(3 * r, 3 * r + 3)
        assert torch.equal(res[r]["x"], full["x"][sl])
        assert torch.equal(res[r]["state0"], full["state0"][sl])
        assert torch.equal(res[r]["accept_len"], full["accept_len"][sl])
        assert res[r]["max"] == 11.0
