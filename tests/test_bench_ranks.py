"""The N > 1 replica path of bench.py on the host: two gloo ranks on CPU
reduce their timed-loop and end-to-end times to the slowest rank's, and the
whole-job rate counts every rank's tokens over that time (on a GPU node the
same functions run over NCCL, one process per GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r: a timed loop of 10 + r ms, an end-to-end loop of 20 - 3 r ms
        ms, e2e = bench.ranks_max(dist, [10.0 + rank, 20.0 - 3 * rank], device="cpu")
        dist.barrier()
        out.put((rank, ms, e2e, bench.job_rates(64, ms, e2e, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r[0] for r in res) == [0, 1]
    for _, ms, e2e, (value, e2e_value) in res:
        assert ms == 11.0 and e2e == 20.0          # each the slowest rank's
        assert value == pytest.approx(64 * 2 / 11e-3)
        assert e2e_value == pytest.approx(64 * 2 / 20e-3)


def test_one_rank_is_unchanged():
    import bench
    assert bench.ranks_max(None, [3.5, 7]) == [3.5, 7.0]
    assert bench.job_rates(10, 2.0, 4.0, 1) == pytest.approx((5000.0, 2500.0))
