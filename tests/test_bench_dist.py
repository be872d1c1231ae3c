"""The N > 1 logic of bench.py on CPU: two gloo ranks combine their timings
(max of step times, sum of bytes and elements), work on disjoint data, and
only rank 0 runs the reference arm."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, nbytes, elems = bench.combine_over_ranks(dist, torch.device("cpu"), 1.5 + rank, 100.0 * (rank + 1),
                                                  10.0 * (rank + 1))
    out[rank] = (ms, nbytes, elems)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_combine_timings():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        ps = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in ps:
            p.start()
        for p in ps:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1] == (2.5, 300.0, 30.0)


def test_single_process_passthrough():
    assert bench.combine_over_ranks(None, None, 3.0, 7.0, 1.0) == (3.0, 7.0, 1.0)


def test_ranks_take_disjoint_shards():
    seen = set()
    for rank in range(8):
        seeds = bench.rank_data_seeds(rank)
        assert len(seeds) == 8 and not (seen & set(seeds))
        seen |= set(seeds)


def test_reference_arm_runs_on_rank0_only(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 3, "gpus": 2})()
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
