"""The multi-rank benchmark logic on CPU with gloo, world size 2: every rank
gets its own shard (weak scaling), no collective touches the data, and the
job time is the max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from bit_kv_cache_ott_gb300 import synth
    w = synth.WORKLOADS["tiny"]
    ws = bench.shard(w, rank, world)
    k, _, _ = synth.step_kvq(ws, 0)
    local_ms = 10.0 + 5.0 * rank              # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms)
    q.put((rank, ws.seed, float(k.float().sum()), ms,
           bench.job_tokens_per_s(w.B, 100, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_and_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seed0, sum0, ms0, tps0), (r1, seed1, sum1, ms1, tps1) = res
    assert seed0 != seed1 and sum0 != sum1           # different shards
    assert ms0 == ms1 == 15.0                         # max over ranks
    assert tps0 == tps1 == pytest.approx(1 * 100 * 2 / 15e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
