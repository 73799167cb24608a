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
