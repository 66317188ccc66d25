"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one process
each, rendezvous on 127.0.0.1) take the maximum of their step times, and the
whole-job value counts every rank's bytes over that slowest time.  The
reference arm exits at once on ranks other than 0."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    ms = bench.max_over_ranks(1.0 + rank, dist, torch.device("cpu"))
    dist.barrier()
    out[rank] = (r, w, ms, bench.whole_job_gbs(1e9, w, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, ms, gbs) in res.items():
        assert (r, w) == (rank, 2)
        assert ms == 2.0  # the slower rank's time, on both ranks
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_reference_arm_is_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0  # no work, no output on rank 1
