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
