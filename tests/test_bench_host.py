"""Host logic of the benchmark: the shard plan that deals one problem's
(batch entry, kv head) pairs out over the ranks, max-over-ranks timing and
whole-job aggregation, exercised with two gloo ranks on CPU; JSON contract
fields."""
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


def _plan_rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        segs = bench.shard_plan(4, 4, world, rank)      # the causal GQA workload's pairs
        pairs = [(b, hk) for b0, b1, k0, k1 in segs for b in range(b0, b1) for hk in range(k0, k1)]
        gathered = [None] * world
        dist.all_gather_object(gathered, pairs)
        # this rank's (simulated) time for its pairs; the job time is the slowest rank's
        t = bench.reduce_max(dist, 0.001 * len(pairs))
        out[rank] = (gathered, t)
    finally:
        dist.destroy_process_group()


def test_shard_plan_with_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_plan_rank_main, args=(r, world, port, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    g0, t0 = res[0]
    g1, t1 = res[1]
    assert g0 == g1
    allp = [p for ranks in g0 for p in ranks]
    assert sorted(allp) == [(b, hk) for b in range(4) for hk in range(4)]
    assert len(set(map(tuple, allp))) == 16
    assert t0 == t1 == 0.008


@pytest.mark.parametrize("B,Hkv", [(1, 16), (2, 16), (4, 4), (64, 8), (1, 1), (3, 5)])
def test_shard_plan_covers_every_pair_once(B, Hkv):
    import bench
    for world in range(1, 9):
        seen = []
        sizes = []
        for rank in range(world):
            segs = bench.shard_plan(B, Hkv, world, rank)
            n = 0
            for b0, b1, k0, k1 in segs:
                assert 0 <= b0 < b1 <= B and 0 <= k0 < k1 <= Hkv
                # one contiguous slice of [B, H, ...]: whole batch entries, or
                # a head range of a single batch entry
                assert (k0, k1) == (0, Hkv) or b1 == b0 + 1
                seen += [(b, hk) for b in range(b0, b1) for hk in range(k0, k1)]
                n += (b1 - b0) * (k1 - k0)
            sizes.append(n)
        assert sorted(seen) == [(b, hk) for b in range(B) for hk in range(Hkv)]
        assert max(sizes) - min(sizes) <= 1            # balanced within one pair
    assert bench.shard_plan(B, Hkv, 1, 0) == [(0, B, 0, Hkv)]   # one launch on one GPU


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
