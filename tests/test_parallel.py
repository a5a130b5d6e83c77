"""Multi-rank host logic on CPU (gloo, world size 2): head sharding and the max-over-ranks
timing reduction the benchmark uses. No GPU and no data-path collective are involved."""
import os
import socket

import pytest

from exact_attention_02_gb300.parallel import head_shard, max_over_ranks


@pytest.mark.parametrize("total,world", [(32, 2), (33, 2), (512, 8), (3, 4), (1, 1), (0, 3)])
def test_head_shards_cover_every_head_once(total, world):
    seen = []
    for r in range(world):
        a, b = head_shard(total, r, world)
        assert 0 <= a <= b <= total
        seen += list(range(a, b))
    assert seen == list(range(total))
    sizes = [head_shard(total, r, world)[1] - head_shard(total, r, world)[0] for r in range(world)]
    assert max(sizes) - min(sizes) <= 1


def test_head_shard_rejects_bad_requests():
    for args in ((4, 2, 2), (4, -1, 2), (4, 0, 0), (-1, 0, 1)):
        with pytest.raises(ValueError):
            head_shard(*args)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "measured" (10 + r) ms for the step and (1 - r) ms elsewhere
        got = max_over_ranks([10.0 + rank, 1.0 - rank])
        a, b = head_shard(32, rank, world)
        out.put((rank, got, (a, b)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [[11.0, 1.0], [11.0, 1.0]]
    assert [r[2] for r in res] == [(0, 16), (16, 32)]


def test_max_over_ranks_without_a_group_is_identity():
    assert max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
