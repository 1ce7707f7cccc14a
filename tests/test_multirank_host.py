"""The N > 1 host path of bench.py on CPU: two gloo ranks rendezvous on
127.0.0.1, pass the timing barrier, agree on the slowest rank's time, and
report the whole-job throughput; the reference arm's other ranks do no
work.  No GPU is used (the ranks hide every CUDA device)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank), "CUDA_VISIBLE_DEVICES": ""})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank r "took" 1 + r seconds: every rank must see the slowest
    t = bench.max_over_ranks(1.0 + r, w)
    value = bench.job_gbs(1e9, 10, w, t)
    with open(os.path.join(out_dir, f"rank{r}.txt"), "w") as f:
        f.write(f"{t} {value}\n")
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        t, value = map(float, (tmp_path / f"rank{r}.txt").read_text().split())
        assert t == 2.0                      # max over ranks of 1 + rank
        assert value == pytest.approx(10.0)  # 2 ranks x 10 steps x 1 GB / 2 s


def test_reference_arm_other_ranks_do_no_work():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 3, 3
    assert bench.reference_arm(Args(), 1, 2) is None


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_gbs(85_082_112, 100, 1, 2e-3)
    four = bench.job_gbs(85_082_112, 100, 4, 2e-3)
    assert four == pytest.approx(4 * one)
