"""The bench's replica path over two ranks, on CPU (gloo).

With N > 1 every rank runs its own verify cycles; the job is done when the
slowest rank is, so the timed region is the maximum over ranks and the
whole-job value is all ranks' cycles over that time.  These run the same
helpers the GPU bench calls, on two `gloo` processes on 127.0.0.1.
"""
import contextlib
import io
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        # rank r took (r + 1) * 0.25 s for its 10 cycles
        slowest = bench.max_over_ranks(torch, (rank + 1) * 0.25, w, torch.device("cpu"))
        rate = bench.job_rate(10, w, slowest)
        printed = ""
        rc = None
        if rank != 0:
            # the reference arm: every rank but 0 leaves at once, printing nothing
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                rc = bench.main(["--impl", "reference", "--gpus", str(w), "--steps", "1",
                                 "--warmup", "3"])
            printed = buf.getvalue()
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"env": [w, r, local], "slowest": slowest, "rate": rate,
                       "rc": rc, "printed": printed}, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_max_time_and_job_rate(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["env"] == [world, r, r]
        # both ranks see the slowest rank's time ...
        assert d["slowest"] == pytest.approx(0.5, rel=0, abs=0)
        # ... and the value counts every rank's cycles: 2 x 10 cycles in 0.5 s
        assert d["rate"] == pytest.approx(40.0)
    assert res[1]["rc"] == 0 and res[1]["printed"] == ""


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(torch, 0.125, 1, torch.device("cpu")) == 0.125
    assert bench.job_rate(20, 1, 0.1) == pytest.approx(200.0)
