"""Seeded random shapes through every entry point, against the oracle, bit
for bit: rank-major layout, dispatch (bf16 and FP8) and combine (plain and
weighted); the single layout + dispatch call (rank-major, both payloads);
expert-major layout, dispatch and weighted combine; the one-launch dispatch
where the batch allows it; local ids; FP8 cast and transposed cast.
Each case draws T, H, E, k, W, the routing (uniform or Zipf, with invalid ids
and repeated experts) and the capacity from its own seed."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_bf16, make_routing
from gpu_util import (assert_rows_equal, run_combine, run_dispatch, run_layout, run_with_layout,
                      to_dev_bf16, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    W = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
    Er = int(rng.integers(1, 33))
    E = W * Er
    k = int(rng.integers(1, min(E, 16) + 1))
    T = int(rng.choice([0, 1, 7, 100, 513, 1024, 1025, 3000, 6000]))
    H = int(rng.choice([128, 256, 384, 1024, 2048, 4096, 7168]))
    idx = make_routing(rng, T, E, k, "zipf" if rng.random() < 0.5 else "uniform") if T else \
        np.zeros((0, k), np.int32)
    if T and rng.random() < 0.5:
        idx[rng.random(idx.shape) < 0.03] = int(rng.choice([-1, E, E + 5]))
    if T and k > 1 and rng.random() < 0.3:
        rep = rng.random(T) < 0.2
        idx[rep, 1] = idx[rep, 0]
    x = make_bf16(rng, (T, H), scale=float(rng.choice([0.01, 1.0, 100.0])))
    w = rng.standard_normal((T, k)).astype(np.float32)
    return rng, T, H, E, k, W, idx, x, w


@pytest.mark.parametrize("seed", range(30))
def test_fuzz_rank_major(seed):
    rng, T, H, E, k, W, idx, x, w = _case(seed)
    lay = oracle.layout(idx, E, W)
    got = run_layout(idx, E, W)
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
        assert_rows_equal(got[key], lay[key], key)
    R = int(lay["rank_offset"][-1])
    cap = max(1, R - int(rng.integers(0, 3)) * (R // 10))      # sometimes short of R
    for quant in (ep.EP_QUANT_BF16, ep.EP_QUANT_FP8_E4M3_B128):
        want = oracle.dispatch(x, idx, w, lay["slot"], cap, quant)
        g = run_dispatch(x, idx, w, lay["slot"], cap, quant)
        n = min(R, cap)
        assert g["status"] == want["status"]
        assert_rows_equal(g["recv_x"][:n], want["recv_x"][:n], "recv_x")
        if quant == ep.EP_QUANT_FP8_E4M3_B128:
            assert_rows_equal(g["recv_scale"][:n].view(np.uint32), want["recv_scale"][:n].view(np.uint32),
                              "recv_scale")
        for key in ("recv_topk_idx", "recv_src"):
            assert_rows_equal(g[key][:n], want[key][:n], key)
        # the same through the single layout + dispatch call (whichever of its
        # paths this size takes)
        if quant == ep.EP_QUANT_BF16 or H % 128 == 0:
            gw = run_with_layout(x, idx, w, E, W, cap, quant)
            for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
                assert_rows_equal(gw[key], lay[key], "with_layout " + key)
            assert gw["status"] == lay["status"] | want["status"]
            assert_rows_equal(gw["recv_x"][:n], want["recv_x"][:n], "with_layout recv_x")
            if quant == ep.EP_QUANT_FP8_E4M3_B128:
                assert_rows_equal(gw["recv_scale"][:n].view(np.uint32),
                                  want["recv_scale"][:n].view(np.uint32), "with_layout recv_scale")
            for key in ("recv_topk_idx", "recv_src"):
                assert_rows_equal(gw[key][:n], want[key][:n], "with_layout " + key)
        if quant == ep.EP_QUANT_BF16 and cap >= R and T:
            local = oracle.localize_ids(want["recv_topk_idx"], E, W, lay["rank_offset"])
            ri = torch.from_numpy(np.ascontiguousarray(g["recv_topk_idx"])).cuda()
            ep.ep_localize_expert_ids(ri, torch.from_numpy(lay["rank_offset"]).cuda(), E, W)
            torch.cuda.synchronize()
            assert_rows_equal(ri.cpu().numpy()[:R], local[:R], "local ids")
    y = make_bf16(rng, (cap, H))
    assert_rows_equal(run_combine(y, lay["slot"], H, cap)["out"],
                      oracle.combine(y, lay["slot"], cap)["out"], "combine")
    wr = rng.standard_normal(lay["slot"].shape).astype(np.float32)
    yd = to_dev_bf16(y)
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_combine_weighted(yd, torch.from_numpy(lay["slot"]).cuda(), torch.from_numpy(wr).cuda(), out, st)
    torch.cuda.synchronize()
    assert_rows_equal(u16(out), oracle.combine_weighted(y, lay["slot"], wr, cap)["out"], "combine_weighted")
    if 0 < T <= ep.EP_FUSED_MAX_TOKENS and k <= 16 and E <= 8192:
        dc = ep.DispatchCombine(T, H, E, k, W, capacity_rows=max(R, 1))
        dc.dispatch_fused(to_dev_bf16(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda())
        torch.cuda.synchronize()
        assert_rows_equal(dc.slot.cpu().numpy(), lay["slot"], "fused slot")
        assert_rows_equal(u16(dc.recv_x)[:R], oracle.dispatch(x, idx, w, lay["slot"], R)["recv_x"][:R],
                          "fused recv_x")


@pytest.mark.parametrize("seed", range(30, 45))
def test_fuzz_expert_major(seed):
    rng, T, H, E, k, W, idx, x, w = _case(seed)
    if T == 0 or k > 32:
        pytest.skip("empty batch")
    E = min(E, 4096)
    idx = np.where(idx >= E, E + 1, idx).astype(np.int32)
    lay = oracle.layout_experts(idx, E)
    dc = ep.DispatchCombine(T, H, E, k, W if E % W == 0 else 1, order="expert")
    xd, idd, wd = to_dev_bf16(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    dc.layout(idd)
    dc.dispatch(xd, idd, wd)
    torch.cuda.synchronize()
    assert_rows_equal(dc.slot.cpu().numpy(), lay["slot"], "slot")
    assert_rows_equal(dc.expert_offset.cpu().numpy(), lay["expert_offset"], "expert_offset")
    R = int(lay["expert_offset"][-1])
    dis = oracle.dispatch(x, idx, w, lay["slot"], max(R, 1))
    assert_rows_equal(u16(dc.recv_x)[:R], dis["recv_x"][:R], "recv_x")
    out = dc.combine(None, wd)
    torch.cuda.synchronize()
    assert_rows_equal(u16(out), oracle.combine_weighted(dis["recv_x"], lay["slot"], w)["out"], "out")
    if H % 256 == 0 and R:
        scale = (2.0 ** rng.uniform(-4, 6, size=E)).astype(np.float32)
        c, t, amax = dc.cast_transpose(torch.from_numpy(scale).cuda())
        torch.cuda.synchronize()
        want = oracle.cast_transpose(dis["recv_x"][:R], lay["expert_offset"], scale)
        assert_rows_equal(c.cpu().numpy()[:R], want["out_c"], "cast")
        assert np.array_equal(t.cpu().numpy()[:want["out_t"].size], want["out_t"])
        np.testing.assert_array_equal(amax.cpu().numpy().view(np.uint32), want["amax"].view(np.uint32))
