"""The multi-GPU path is replicas (each rank runs its own step, no data-path
collective); what bench.py adds for N > 1 is host logic: ranks from the
launcher's environment, the slowest rank's step time as the job's time, and
the whole-job throughput.  Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, times, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r, w, local = bench.rank_info()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        ms = bench.max_over_ranks(torch, times[r], w, device="cpu")
        with open(os.path.join(out_dir, "rank%d.txt" % r), "w") as f:
            f.write("%d %d %d %r %r\n" % (r, w, local, ms, bench.job_gbs(w, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_bytes(tmp_path):
    world, times = 2, [0.95, 1.25]  # ms per step on each rank
    mp.spawn(rank_main, args=(world, free_port(), times, str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(world)]
    for r, row in enumerate(rows):
        rr, w, local, ms, gbs = int(row[0]), int(row[1]), int(row[2]), float(row[3]), float(row[4])
        assert (rr, w, local) == (r, world, r)
        assert ms == max(times)  # every rank sees the slowest rank's time
        assert gbs == pytest.approx(world * bench.BYTES_PER_STEP / (max(times) * 1e-3) / 1e9, rel=1e-12)


def test_one_rank_is_the_identity():
    assert bench.max_over_ranks(torch, 0.5, 1) == 0.5
    assert bench.job_gbs(1, 1.0) == pytest.approx(bench.BYTES_PER_STEP / 1e-3 / 1e9)
