"""Multi-rank host logic of bench.py (barrier, max/sum over ranks, whole-job
throughput) on world-size-2 gloo process groups on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, _ = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    # rank r moves (r + 1) GB in (10 + 5 r) ms
    gbs, ms_max, total = bench.whole_job_gbs(dist, (r + 1) * 1e9, 10.0 + 5.0 * r)
    mx = bench.reduce_max(dist, float(r))
    sm = bench.reduce_sum(dist, float(r + 1))
    out[r] = (r, w, gbs, ms_max, total, mx, sm)
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        rr, w, gbs, ms_max, total, mx, sm = out[r]
        assert (rr, w) == (r, world)
        assert ms_max == 15.0 and total == 3e9 and mx == 1.0 and sm == 3.0
        assert gbs == pytest.approx(3e9 / 15e-3 / 1e9)


def test_single_process_is_identity():
    import bench

    assert bench.dist_init(1, "gloo") is None
    gbs, ms, total = bench.whole_job_gbs(None, 2e9, 4.0)
    assert (ms, total) == (4.0, 2e9) and gbs == pytest.approx(500.0)


def test_config_percentiles_and_call_counts():
    import bench

    med, p10, p90 = bench.percentiles([5.0, 1.0, 4.0, 2.0, 3.0])
    assert (med, p10, p90) == (3.0, 1.4, 4.6)
    # every config times at least CONFIG_MIN_CALLS calls, in whole graph launches
    for reps in (1, 6, 12, 21, 977):
        launches = max(5, -(-bench.CONFIG_MIN_CALLS // reps))
        assert launches * reps >= bench.CONFIG_MIN_CALLS and launches >= 5


def test_headline_mode_is_the_faster_chain_mode():
    import bench

    assert bench.choose_head({"fused": 5.17, "sequential": 4.96}) == "sequential"
    assert bench.choose_head({"fused": 4.0, "sequential": 4.96}) == "fused"
    assert bench.choose_head({"fused": 5.0, "sequential": 5.0}) == "fused"
    assert bench.choose_head({"fused": 5.1, "phased": 4.2, "sequential": 4.9}) == "phased"
    # launches per step with one launch per dependency phase: q, k, v share one
    descs = [{"after": a} for a in bench.layer_dependencies(12)]
    assert bench.count_phases(descs) == 8
    cfg = bench._config(16, 64, 1, "sequential", 384)
    assert cfg["launches_per_step"] == 384 and "sequential" in cfg["headline"]
    assert bench._config(16, 64, 1)["launches_per_step"] == 1


def test_e2e_chunks_cover_the_layers():
    import bench
    assert bench.e2e_chunks(64, "8") == [8] * 8
    assert bench.e2e_chunks(64, "2,6,8,8,8,8,8,8,6,2") == [2, 6] + [8] * 6 + [6, 2]
    assert bench.e2e_chunks(6, "4") == [4, 2]
    assert bench.e2e_chunks(64, "taper") == [2, 6] + [8] * 6 + [6, 2]
    assert bench.e2e_chunks(2, "taper") == [2]
    with pytest.raises(ValueError):
        bench.e2e_chunks(64, "8,8")
