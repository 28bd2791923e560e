"""Multi-rank host logic of the benchmark, on CPU ranks with the gloo backend: the path
runs as independent replicas (no data-path collective), timing is the max over ranks,
and the whole-job value counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from sink_kv_attention_gb300 import synth
    try:
        # each replica draws different inputs
        pos, head, _ = synth.window_state(13 + bench.replica_seed_base(rank), 32, 4092, 4096, 32768)
        gathered = [torch.zeros_like(pos) for _ in range(world)]
        dist.all_gather(gathered, pos)
        distinct = not torch.equal(gathered[0], gathered[1])
        # the slowest rank sets the time
        t = bench._max_over_ranks(1.0 + rank, world, device="cpu")
        results[rank] = (distinct, t, bench.weak_scaling_value(537_000_000, t, world))
    finally:
        dist.destroy_process_group()


def test_replicas_and_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        distinct, t, value = results[r]
        assert distinct
        assert t == 2.0                     # max over ranks of 1.0 and 2.0 ms
        assert value == pytest.approx(2 * 537_000_000 / 2e-3 / 1e9)
