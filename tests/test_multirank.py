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


def _stubbed_rank(argv):
    """One rank of `bench.py --gpus 2` on CPU: everything as in a GPU run
    except the device leg, which reports that rank r's timed region took
    10 + r ms."""
    import bench as b

    def leg(args, wl, rank, world, local_rank):
        batch, _ = b.shard(wl.batch, rank)
        return {"elapsed_ms": 10.0 + rank, "steps": args.steps, "per_step": 1, "batch": batch, "nsets": 3,
                "launch_bytes": 1.0e6, "wall_s": 0.01, "graphs": 1, "e2e": None,
                "clocks": {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}}

    b.device_leg = leg
    return b.main(argv)


def test_bench_gpus_2_launches_its_own_ranks(monkeypatch, capfd):
    """`bench.py --gpus 2` with no outside launcher spawns two ranks (gloo
    here, no GPU); rank 0 alone prints one JSON line, with n_gpus 2, the
    slower rank's time and both ranks' sequences in the value."""
    real = bench.launch_ranks
    monkeypatch.setattr(bench, "launch_ranks", lambda argv, world: real(argv, world, entry=_stubbed_rank))
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    steps = 4
    assert bench.main(["--gpus", "2", "--workload", "0", "--steps", str(steps), "--warmup", "3",
                       "--no-cpu-baseline", "--e2e-steps", "0"]) == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    import json
    line = json.loads(lines[0])
    wl = synth.WORKLOADS[0]
    assert line["n_gpus"] == 2 and line["scaling"] == "weak" and line["steps"] == steps
    assert line["config"]["parallelism"] == "dp2"
    assert abs(line["ms_per_step"] - 11.0 / steps) < 1e-12  # the maximum over the ranks
    want = wl.batch * wl.ntok * 2 * wl.nlayers * steps / 11.0e-3
    assert abs(line["value"] - want) < 1e-9 * want
