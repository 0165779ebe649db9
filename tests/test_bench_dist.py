"""Host logic of bench.py at N > 1: two gloo ranks on the CPU.

Each rank times its own batch shard; the reported time is the slowest rank's and the
throughput counts every rank's tokens. No GPU and no collective on the data path.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import path_inputs as pi


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_setup(world, backend="gloo")
    assert (r, w, local) == (rank, world, rank)
    local_ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
    t_max, ms_step, value = bench.aggregate(local_ms, w, 32, 4096, 4)
    wl = bench.shard_workload(pi.TINY_FP32, rank)
    x = pi.workload_inputs(wl)
    digest = float(x["q"].double().sum())
    bench.barrier(w)
    out[rank] = torch.tensor([t_max, ms_step, value, digest, wl.seed], dtype=torch.float64)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_aggregate_and_shards():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    r0, r1 = out[0].tolist(), out[1].tolist()
    # both ranks agree on the slowest rank's time
    assert r0[0] == r1[0] == 15.0
    assert r0[1] == r1[1] == 15.0 / 4
    # every rank's tokens over that time
    assert r0[2] == pytest.approx(2 * 32 * 4096 * 4 / 15e-3)
    # rank 0's shard is the single-GPU workload; rank 1 draws its own rows
    assert r0[4] == pi.TINY_FP32.seed and r1[4] != r0[4]
    assert r0[3] != r1[3]


def test_single_rank_is_local():
    t_max, ms_step, value = bench.aggregate(8.0, 1, 32, 4096, 2)
    assert (t_max, ms_step) == (8.0, 4.0)
    assert value == pytest.approx(32 * 4096 * 2 / 8e-3)
    assert bench.shard_workload(pi.BF16_L4096, 0) is pi.BF16_L4096


def test_line_order_ends_with_the_headline_legs():
    # the legs a reader of the line's last 3 KB needs come last, in LINE_END order; the
    # contract keys keep their place at the front
    line = {"metric": "m", "value": 1.0, "sweep_L": {}, "bwd": {}, "producer": {},
            "fox": {}, "decode": {}, "fwd_f32": {}, "bwd_d128": {}, "fwd_d128": {}}
    keys = list(bench.order_line(line))
    assert keys[:2] == ["metric", "value"]
    assert keys[-6:] == list(bench.LINE_END)
    assert set(keys) == set(line)
    # absent legs are skipped, not invented
    assert list(bench.order_line({"metric": "m", "fox": {}})) == ["metric", "fox"]

