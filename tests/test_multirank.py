"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2), as torchrun would start
them.  bench.py runs one replica of the workload per rank with no collective on the data path; the
host logic is the slowest-rank timing, the aggregate throughput over all ranks and the replicas'
identical seeded inputs."""
import hashlib
import multiprocessing
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results, fail_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import datetime

    import torch.distributed as dist
    from gated_delta_rule_23_gb300.inputs import make_workload

    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    try:
        if rank == fail_rank:
            raise RuntimeError("rank left before the timing exchange")
        ms = [10.0, 12.5, 11.0, 9.0][rank]
        slowest = bench.max_over_ranks(ms, world, "cpu")
        value = bench.aggregate_throughput(1000, world, slowest)
        p = make_workload(0)
        digest = hashlib.sha256(p.q.tobytes() + p.k.tobytes() + p.v.tobytes() + p.g.tobytes()).hexdigest()
        digests = [None] * world
        dist.all_gather_object(digests, digest)
        results.put((rank, slowest, value, digests))
    except Exception as e:  # reported to the parent, which checks who failed and how
        results.put((rank, "error", type(e).__name__, str(e)[:200]))
    finally:
        try:
            dist.destroy_process_group()
        except Exception:
            pass


def _run(world, fail_rank=-1, timeout=120):
    ctx = multiprocessing.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results, fail_rank)) for r in range(world)]
    for pr in procs:
        pr.start()
    out = {}
    try:
        for _ in range(world):
            item = results.get(timeout=timeout)
            out[item[0]] = item[1:]
    finally:
        for pr in procs:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.kill()
    return out


def test_two_ranks_report_the_slowest_time_and_the_whole_job_throughput():
    out = _run(2)
    for rank in range(2):
        slowest, value, digests = out[rank]
        assert slowest == 12.5
        assert value == pytest.approx(2 * 1000 / 12.5e-3)
        assert digests[0] == digests[1]      # every replica processes the same seeded workload


def test_a_rank_that_leaves_is_an_error_not_a_hang():
    """Rank 1 leaves before the timing exchange: rank 0's barrier ends with an error within the
    process-group timeout instead of waiting for ever."""
    out = _run(2, fail_rank=1)
    assert out[1][0] == "error"
    assert out[0][0] == "error"
