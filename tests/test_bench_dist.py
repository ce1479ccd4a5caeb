"""Multi-rank host logic of bench.py (barrier, max-over-ranks time, summed
units) on CPU with the gloo backend, world size 2."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    ms, units = bench.reduce_max_sum(w, 10.0 + rank, 100.0 * (rank + 1))
    out[rank] = (r, w, lr, ms, units)
    torch.distributed.destroy_process_group()


def test_two_rank_reduction_on_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        r, w, lr, ms, units = out[rank]
        assert (r, w, lr) == (rank, world, rank)
        assert ms == 11.0 and units == 300.0


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_sum(1, 3.5, 7.0) == (3.5, 7.0)


def test_reference_arm_line_shape(capsys, monkeypatch):
    """--impl reference prints one JSON line with the oracle as the reference arm."""
    import json

    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
