"""The N > 1 host path on CPU: world-size-2 gloo ranks.

Requests are independent under the MIS mask, so ranks split them with no
exchange on the data path. Each rank plans its own share with the host
planner; together the shares must cover every request exactly once and add
up to the whole batch's visible pairs and tiles. The bench's timing
reduction must return the slowest rank's time on every rank.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from ranking_prefill_gb300 import lib, synth
        w = synth.WORKLOADS["varlen-16"]
        s = synth.draw_shapes(w)
        mine = synth.shard_requests(len(s.prefix_tokens), rank, world)
        ptr = np.concatenate([[0], np.cumsum(s.n_items)])
        lens = np.concatenate([s.item_lens[ptr[b]:ptr[b + 1]] for b in mine]) if len(mine) else []
        lay = lib.mis_build_layout(s.prefix_tokens[mine], s.n_items[mine], lens)
        st = lib.Plan.host_only(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets,
                                w.hq, w.hkv, w.head_dim).stats()
        t = torch.tensor([st["visible_pairs"], st["n_tiles"], lay.M, len(mine)], dtype=torch.int64)
        dist.all_reduce(t)
        got = [None] * world
        dist.all_gather_object(got, mine.tolist())
        slowest = bench.max_over_ranks(1.5 + rank, dist)
        q.put((rank, t.tolist(), got, slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_request_split_and_timing():
    sys.path.insert(0, ROOT)
    from ranking_prefill_gb300 import lib, synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.WORKLOADS["varlen-16"]
    s = synth.draw_shapes(w)
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    full = lib.Plan.host_only(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets,
                              w.hq, w.hkv, w.head_dim).stats()
    for rank, tot, shards, slowest in res:
        assert tot == [full["visible_pairs"], full["n_tiles"], lay.M, len(s.prefix_tokens)]
        flat = sorted(sum(shards, []))
        assert flat == list(range(len(s.prefix_tokens)))
        assert slowest == 2.5


@pytest.mark.parametrize("n,world", [(16, 2), (5, 3), (1, 4), (256, 8)])
def test_shard_requests_partition(n, world):
    sys.path.insert(0, ROOT)
    from ranking_prefill_gb300 import synth
    parts = [synth.shard_requests(n, r, world) for r in range(world)]
    assert sorted(np.concatenate(parts).tolist()) == list(range(n))
    sizes = [len(p) for p in parts]
    assert max(sizes) - min(sizes) <= 1
