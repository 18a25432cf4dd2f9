"""Host-side logic of the multi-GPU (replica) bench path, run as two gloo
ranks on CPU: ranks agree on the slowest rank's time and report the
whole-job aggregate."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = 1.0 + rank * 0.5          # rank 1 is slower
    worst = bench._max_over_ranks(my_ms, True, "cpu")
    bench._barrier(True)
    q.put((rank, worst))
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 1.5), (1, 1.5)]


def test_replica_aggregate_is_weak_scaling():
    # value = units all ranks processed / slowest rank's time
    lay = bench.workloads.config_layout(1, 0)
    kvb = bench.kv_bytes(lay.seq_lens, lay.num_kv_heads, lay.head_dim)
    one = 1 * kvb / (2.0e-3) / 1e9
    two = 2 * kvb / (2.0e-3) / 1e9
    assert two == pytest.approx(2 * one)


def test_kv_bytes_matches_the_pages_formula():
    # one layer of Llama-2-7B: 2 (K, V) x 32 heads x 128 dims x 2 bytes per token
    from oracle import metadata
    per_token = metadata.kv_bytes_per_token(1, 32, 128, 2)
    assert bench.kv_bytes([4096], 32, 128) == per_token * 4096
