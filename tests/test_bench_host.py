"""Host logic of the benchmark: max-over-ranks timing and whole-job
aggregation, exercised with two gloo ranks on CPU; JSON contract fields."""
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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(dist, 1.5 + rank)   # rank 1 is the slow one
        out[rank] = (t, bench.aggregate(100.0, world, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world, port = 2, _free_port()
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
    assert res[0] == res[1] == (2.5, 100.0 * 2 / 2.5)


def test_single_process_identity():
    import bench
    assert bench.reduce_max(None, 3.25) == 3.25
    assert bench.aggregate(10.0, 1, 2.0) == 5.0


def test_peaks_file_or_fallback():
    import bench
    p = bench.load_peaks()
    assert p["source"] in ("measured", "fallback")
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 500


def test_clock_summary_parsing():
    import bench
    c = bench.ClockSampler()
    c.lines = ["0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active",
               "0, 1980, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1972.5 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
