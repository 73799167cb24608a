"""Host logic of the benchmark: byte model, the pages' bandwidth convention, and
the multi-rank aggregation (gloo, world size 2, CPU)."""
import json
import os
import statistics

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from combine_ep_dispatch_gb300.inputs import CONFIGS, make_routing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_pages_bandwidth_convention():
    with open(os.path.join(GOLDEN, "mori_bandwidth.json")) as f:
        g = json.load(f)
    dev = []
    for row in g["rows"]:
        R = bench.expected_rows(row["tokens"], g["E"], g["k"], g["W"])
        v = bench.pages_convention_gbs(R, g["H"], g["elem_bytes"], row["us"] * 1e-6)
        dev.append(abs(v / row["gbs"] - 1))
    assert max(dev) < 0.03
    assert statistics.median(dev) < 0.01


def test_expected_rows_matches_sampled_routing():
    cfg = CONFIGS["dsv3"]
    idx = make_routing(np.random.default_rng(0), cfg.T, cfg.E, cfg.k)
    R = int(oracle.layout(idx, cfg.E, cfg.W)["rank_offset"][-1])
    ER = bench.expected_rows(cfg.T, cfg.E, cfg.k, cfg.W)
    assert abs(R - ER) < 4 * np.sqrt(cfg.T * cfg.W * 0.25)      # a few standard deviations
    assert abs(ER / cfg.T - 5.2947) < 1e-3


def test_alg_bytes_dsv3():
    b = bench.alg_bytes(4096, 7168, 256, 8, 8, 21706)
    assert b["dispatch"] == 4096 * 7168 * 2 + 4096 * 64 + 4096 * 32 + 21706 * 7168 * 2 + 21706 * 68
    assert b["combine"] == 21706 * 7168 * 2 + 4096 * 32 + 4096 * 7168 * 2
    assert 370e6 < b["dispatch"] < 373e6 and 369e6 < b["combine"] < 372e6


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    stats, total = bench.aggregate([1.0 + rank, 5.0 - rank], 100.0 * (rank + 1), world,
                                   torch.device("cpu"))
    q.put((rank, stats, total))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, stats, total in res:
        assert stats == [2.0, 5.0]          # max over ranks, per entry
        assert total == 300.0               # bytes summed over ranks


def test_aggregate_single_rank_is_identity():
    s, t = bench.aggregate([1.5, 2.5], 7.0, 1, torch.device("cpu"))
    assert s == [1.5, 2.5] and t == 7.0


def test_alg_bytes_fp8_payload():
    """FP8 rows: one byte per value plus one fp32 scale per 128 values, the
    rest of the dispatch's bytes as for bf16; combine unchanged."""
    T, H, E, k, W, R = 4096, 7168, 256, 8, 8, 11815
    b16, b8 = bench.alg_bytes(T, H, E, k, W, R), bench.alg_bytes(T, H, E, k, W, R, fp8=True)
    assert b16["dispatch"] - b8["dispatch"] == R * H * 2 - (R * H + R * (H // 128) * 4)
    assert b8["combine"] == b16["combine"] and b8["layout"] == b16["layout"]
    assert b8["step"] == b8["layout"] + b8["dispatch"] + b8["combine"]


def test_trimmed_mean_drops_the_tails():
    v = [10.0] * 90 + [1000.0] * 5 + [0.0] * 5
    assert bench.trimmed_mean(v) == 10.0
    assert bench.trimmed_mean([3.0, 5.0]) == 4.0
    # on a 1 us tick grid, the mean of the middle resolves finer than the median
    ticks = [1.024 * (50 + (i % 4 == 0)) for i in range(100)]
    assert abs(bench.trimmed_mean(ticks) - 1.024 * 50.25) < 0.03


def test_profile_traffic_needs_matching_sources(tmp_path, monkeypatch):
    """DRAM bytes come from a profile summary only while its source hash is the
    current one (a summary of other sources would describe another kernel)."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = bench.kernel_source_hash("combine")
    (prof / "combine_dsv3.txt").write_text(f"source_sha256_16: {good}\ndram_bytes_per_launch: 123\n")
    (prof / "dispatch_dsv3.txt").write_text("source_sha256_16: 0000\ndram_bytes_per_launch: 456\n")
    real_join = os.path.join

    def join(*a):
        if len(a) >= 2 and a[1] == "profiles":
            return real_join(str(tmp_path), *a[1:])
        return real_join(*a)

    monkeypatch.setattr(bench.os.path, "join", join)
    assert bench._traffic_from_profile("combine", "dsv3") == 123.0
    assert bench._traffic_from_profile("dispatch", "dsv3") is None
    assert bench._traffic_from_profile("combine", "qwen") is None
