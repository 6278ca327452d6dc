"""Weak-scaling shards on two gloo ranks (CPU): each rank runs its own
sequences with no data-path collective, and the union of the shards equals
the unsharded run of the same recipe. The timing reduction is a max."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _steps(wl, batch_offset, full_batch, nsteps=3):
    import oracle
    from decode_kv_cache_step_gb300.workloads import initial_state, step_inputs
    st = initial_state(wl, batch_offset=batch_offset, threads=1)
    ws = np.full((wl.B, wl.Hkv), -1, dtype=np.int32)
    outs, nexts = [], []
    for t in range(nsteps):
        inp = step_inputs(wl, t, batch_offset=batch_offset, full_batch=full_batch)
        r = oracle.decode_step(inp["q"], st["k_cache"], st["v_cache"], st["mask"], inp["new_k"],
                               inp["new_v"], ws, wl.W, wl.scale, nthreads=1)
        outs.append(r["out"])
        nexts.append(r["next_slot"])
        ws = r["next_slot"].copy()
    return np.stack(outs), np.stack(nexts), st["mask"]


def _rank_main(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    from decode_kv_cache_step_gb300.sharding import max_over_ranks, weak_shard
    from decode_kv_cache_step_gb300.workloads import WORKLOADS
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sh = weak_shard(WORKLOADS["tiny_b2_s256"], rank, world)
    out, nxt, mask = _steps(sh.workload, sh.batch_offset, sh.full_batch)
    gathered = [None] * world
    dist.all_gather_object(gathered, (out, nxt, mask))
    tmax = max_over_ranks(1.5 + rank)
    if rank == 0:
        q.put((gathered, tmax))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_equal_the_unsharded_run():
    from decode_kv_cache_step_gb300.workloads import WORKLOADS
    oracle_build = __import__("oracle").build
    oracle_build()
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert tmax == 2.5
    wl = WORKLOADS["tiny_b2_s256"]
    full = wl.with_batch(wl.B * world)
    out, nxt, mask = _steps(full, 0, full.B)
    B = wl.B
    for r, (o, n, m) in enumerate(gathered):
        np.testing.assert_array_equal(o, out[:, r * B:(r + 1) * B])
        np.testing.assert_array_equal(n, nxt[:, r * B:(r + 1) * B])
        np.testing.assert_array_equal(m, mask[r * B:(r + 1) * B])


def test_weak_shard_rejects_bad_ranks():
    from decode_kv_cache_step_gb300.sharding import weak_shard
    from decode_kv_cache_step_gb300.workloads import WORKLOADS
    with pytest.raises(ValueError):
        weak_shard(WORKLOADS["tiny_b2_s256"], 2, 2)
    sh = weak_shard(WORKLOADS["tiny_b2_s256"], 1, 4)
    assert (sh.batch_offset, sh.full_batch) == (2, 8)
