"""The benchmark's multi-rank host logic (replicas, barrier, max over ranks)
with world_size 2 on CPU over gloo: the aggregation the GPU runs do over
NCCL, checked without a GPU."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    sys.argv = ["bench.py"]
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # Every rank's elapsed time differs; all must see the slowest.
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        dist.barrier()
        value = bench.job_us_per_step(slowest / 4, world)   # 4 timed steps
        out.put((rank, slowest, value, bench.max_over_ranks(3.5, None, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    res = sorted(out.get(timeout=5) for _ in range(world))
    for rank, slowest, value, local in res:
        assert slowest == 15.0                       # max of 10 and 15
        assert value == pytest.approx(15.0 / 4 * 1e3 / world)   # us per step, whole job
        assert local == 3.5                          # no process group: the rank's own value


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    # Ranks other than 0 return at once (before reading any argument) and
    # print nothing.
    assert bench.run_reference(None, 1, 2) == 0
    assert capsys.readouterr().out == ""


def _shard_rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    sys.argv = ["bench.py"]
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Each rank takes its KV heads and their query heads (GQA 32/8 and
        # MHA 32/32); the shards of all ranks, gathered, tile the heads.
        got = {}
        for hq, hkv in ((32, 8), (32, 32), (8, 2)):
            mine = torch.tensor(bench.head_shard(hq, hkv, rank, world), dtype=torch.int64)
            every = [torch.zeros(4, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(every, mine)
            got[(hq, hkv)] = [tuple(int(x) for x in t) for t in every]
        # A step split by KV head is done when the slowest shard is: the
        # value is that rank's time per step, not divided by the ranks.
        slowest = bench.max_over_ranks(20.0 + 2.0 * rank, dist, "cpu")
        out.put((rank, got, slowest))
    finally:
        dist.destroy_process_group()


def test_kv_head_shards_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    res = sorted(out.get(timeout=5) for _ in range(world))
    for rank, got, slowest in res:
        assert slowest == 22.0
        for (hq, hkv), shards in got.items():
            G = hq // hkv
            qs = [h for q0, q1, _, _ in shards for h in range(q0, q1)]
            ks = [h for _, _, k0, k1 in shards for h in range(k0, k1)]
            assert qs == list(range(hq)) and ks == list(range(hkv))   # a partition, in rank order
            for q0, q1, k0, k1 in shards:
                assert (q0, q1) == (k0 * G, k1 * G)                    # whole GQA groups
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(ValueError):
        bench.head_shard(32, 8, 0, 3)                                  # 8 KV heads over 3 ranks
