"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2): each
rank draws an independent problem, and the timed result is the maximum over
ranks.  No GPU and no data-path collective are involved."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank, 7.0 * (rank + 1)]
        got = bench.reduce_max_over_ranks(mine, world, torch.device("cpu"))
        q.put((rank, got, bench.rank_seed(1003, rank)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_and_draw_distinct_problems():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, seed in results:
        assert got == [11.0, 5.0, 14.0]
    seeds = {seed for _, _, seed in results}
    assert len(seeds) == world


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_over_ranks([1.0, 2.0], 1, None) == [1.0, 2.0]


def _gather_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import transformer_attention_07_b300 as da
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # a rank's partial states: [B*H, splits, 2, dv + 4], tagged with the rank
        part = torch.full((3, 2, 2, 8), float(rank)) + torch.arange(3 * 2 * 2 * 8, dtype=torch.float32).view(3, 2, 2, 8)
        got = da.gather_partials(part)
        q.put((rank, got.shape, got[:, 0, 0, 0, 0].tolist(), torch.equal(got[rank], part)))
    finally:
        dist.destroy_process_group()


def test_gather_partials_stacks_ranks_in_order():
    """The exchange step of sequence-sharded decode: every rank receives all
    ranks' partial states, stacked in rank order (the [parts, ...] layout the
    merge kernel reads)."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, shape, firsts, own in results:
        assert tuple(shape) == (2, 3, 2, 2, 8)
        assert firsts == [0.0, 1.0]
        assert own


def test_head_range_partitions_every_head_once():
    """The head-partitioned prefill's split of B*H heads over the ranks:
    contiguous, in rank order, sizes within one of each other."""
    import sys
    sys.path.insert(0, ROOT)
    import transformer_attention_07_b300 as da
    for heads in (0, 1, 5, 16, 17, 1024):
        for world in (1, 2, 3, 8):
            ranges = [da.head_range(heads, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == heads
            assert all(ranges[r][1] == ranges[r + 1][0] for r in range(world - 1))
            sizes = [hi - lo for lo, hi in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        da.head_range(4, 2, 2)


def _heads_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import transformer_attention_07_b300 as da
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H = 3, 5   # 15 heads over the ranks: unequal shares
        lo, hi = da.head_range(B * H, world, rank)
        # this rank's output slice: head i holds the value i everywhere
        mine = torch.arange(lo, hi, dtype=torch.float32).view(-1, 1, 1).expand(hi - lo, 4, 6).contiguous()
        full = da.gather_heads(mine, B, H)
        q.put((rank, tuple(full.shape), full[:, 0, 0].tolist()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gather_heads_reassembles_the_output_in_head_order(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_heads_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, shape, firsts in results:
        assert shape == (15, 4, 6)
        assert firsts == [float(i) for i in range(15)]
