"""Replica bookkeeping for N > 1 GPUs, exercised with world_size-2 gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from prefill_only_decision_gb300 import replicas


def test_shard_round_robin():
    units = list(range(11))
    parts = [replicas.shard(units, r, 3) for r in range(3)]
    assert sorted(sum(parts, [])) == units
    assert parts[0] == [0, 3, 6, 9] and parts[2] == [2, 5, 8]
    with pytest.raises(ValueError):
        replicas.shard(units, 3, 3)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # per-rank timed region
        mine = replicas.shard(list(range(74)), rank, world)
        total = replicas.sum_over_ranks(len(mine))
        q.put((rank, replicas.max_over_ranks(ms), total, replicas.world()[:2]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [15.0, 15.0]          # max over ranks
    assert [o[2] for o in out] == [74.0, 74.0]          # every unit processed once
    assert [o[3] for o in out] == [(2, 0), (2, 1)]
