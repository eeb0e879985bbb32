"""The benchmark's multi-GPU logic (independent replicas, barrier, maximum of the
per-rank times, whole-job rate) on two gloo ranks on the CPU (no GPU)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    seconds = 1.0 + rank          # rank 1 is the slower replica
    slowest = bench.reduce_max(seconds, w)
    rate = bench.whole_job_rate(100.0, w, slowest)
    q.put((r, w, local, slowest, rate))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, slowest, rate) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert slowest == 2.0               # the maximum over ranks
        assert rate == 100.0 * 2 / 2.0      # units of every rank / slowest time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_prints_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = bench.argparse.Namespace(workload="tiny", tokens=None, cpu_tokens=64, steps=1,
                                    warmup=0)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
    bench.run_reference(args, rank=0, world=2)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1 and '"impl": "reference"' in out[0]
