"""ep_dispatch_fused (layout + bf16 dispatch in one launch, small batches)
against the CPU oracle, bit for bit: every layout output and every dispatch
output, with sentinel-filled buffers to catch stray writes."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_bf16, make_inputs, make_routing
from gpu_util import SENT_BF16, SENT_I32, assert_rows_equal, to_dev_bf16, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _run_fused(x, idx_dev, w, E, W, cap):
    T, H = x.shape
    k = idx_dev.shape[1]
    i32 = dict(dtype=torch.int32, device="cuda")
    out = {"num_tokens_per_expert": torch.full((E,), SENT_I32, **i32),
           "num_tokens_per_rank": torch.full((W,), SENT_I32, **i32),
           "rank_offset": torch.full((W + 1,), SENT_I32, **i32),
           "slot": torch.full((T, W), SENT_I32, **i32),
           "recv_x": torch.full((cap, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16),
           "recv_topk_idx": torch.full((cap, k), SENT_I32, **i32),
           "recv_topk_w": torch.full((cap, k), -3.0, dtype=torch.float32, device="cuda"),
           "recv_src": torch.full((cap,), SENT_I32, **i32),
           "status": torch.zeros(1, **i32)}
    ep.ep_dispatch_fused(to_dev_bf16(x), idx_dev, torch.from_numpy(w).cuda(), E, W,
                         out["num_tokens_per_expert"], out["num_tokens_per_rank"],
                         out["rank_offset"], out["slot"], out["recv_x"], out["recv_topk_idx"],
                         out["recv_topk_w"], out["recv_src"], out["status"])
    torch.cuda.synchronize()
    res = {kk: v.cpu().numpy() for kk, v in out.items() if kk not in ("recv_x", "status")}
    res["recv_x"] = u16(out["recv_x"])
    res["status"] = int(out["status"].item())
    return res


def _check(x, idx, w, E, W, cap=None, idx_dev=None):
    lay = oracle.layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    cap = max(R, 1) if cap is None else cap
    dis = oracle.dispatch(x, idx, w, lay["slot"], cap)
    if idx_dev is None:
        idx_dev = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    got = _run_fused(x, idx_dev, w, E, W, cap)
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
        assert_rows_equal(got[key], lay[key], key)
    n = min(R, cap)
    assert_rows_equal(got["recv_x"][:n], dis["recv_x"][:n], "recv_x")
    assert_rows_equal(got["recv_topk_idx"][:n], dis["recv_topk_idx"][:n], "recv_topk_idx")
    assert_rows_equal(got["recv_topk_w"][:n].view(np.uint32), dis["recv_topk_w"][:n].view(np.uint32),
                      "recv_topk_w")
    assert_rows_equal(got["recv_src"][:n], dis["recv_src"][:n], "recv_src")
    assert np.all(got["recv_x"][n:] == SENT_BF16) and np.all(got["recv_src"][n:] == SENT_I32)
    assert got["status"] == (lay["status"] | dis["status"])
    return got


@pytest.mark.parametrize("T,H,E,k,W", [
    (0, 256, 16, 4, 4),          # empty batch: counts and offsets still written
    (1, 8, 4, 2, 2),             # one token, register copies
    (128, 256, 16, 4, 4),        # the tiny workload's shape
    (256, 7168, 256, 8, 8),      # the decode workload's shape (bulk copies)
    (777, 512, 64, 6, 8),        # 1 KB rows, ragged token count
    (1024, 4096, 128, 8, 8),     # the largest batch taken
    (1000, 136, 7, 3, 1),        # W = 1, odd E, register copies
    (600, 1024, 64, 16, 32),     # W = 32, up to 16 destinations, scalar id loads
    (300, 10000, 96, 5, 3),      # rows above 16 KB: register copies
])
def test_fused_matches_oracle(T, H, E, k, W):
    rng = np.random.default_rng(T * 31 + H)
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k) if T else np.zeros((0, k), np.int32)
    w = rng.random((T, k), dtype=np.float32)
    _check(x, idx, w, E, W)


def test_fused_decode_workload_and_zipf():
    inp = make_inputs("decode", seed=5)
    cfg = inp["cfg"]
    _check(inp["x"], inp["topk_idx"], inp["topk_w"], cfg.E, cfg.W)
    rng = np.random.default_rng(6)
    idx = make_routing(rng, 512, 256, 8, "zipf")
    _check(make_bf16(rng, (512, 2048)), idx, rng.random((512, 8), dtype=np.float32), 256, 8)


def test_fused_bad_ids_capacity_and_unaligned_ids():
    rng = np.random.default_rng(7)
    T, H, E, k, W = 700, 2048, 64, 8, 8
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k)
    idx[rng.random(idx.shape) < 0.05] = -1
    idx[5, :] = E + 7
    w = rng.random((T, k), dtype=np.float32)
    got = _check(x, idx, w, E, W)
    assert got["status"] & ep.EP_STATUS_BAD_EXPERT
    R = int(oracle.layout(idx, E, W)["rank_offset"][-1])
    got = _check(x, idx, w, E, W, cap=R - 100)
    assert got["status"] & ep.EP_STATUS_CAPACITY
    flat = torch.zeros(T * k + 1, dtype=torch.int32, device="cuda")
    flat[1:] = torch.from_numpy(idx.ravel()).cuda()
    _check(x, idx, w, E, W, idx_dev=flat[1:].view(T, k))      # 4-byte aligned rows


def test_fused_rejects_large_batches():
    T, H, E, k, W = ep.EP_FUSED_MAX_TOKENS + 1, 256, 16, 4, 4
    dc = ep.DispatchCombine(T, H, E, k, W)
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T, k, dtype=torch.float32, device="cuda")
    with pytest.raises(ep.EPError) as e:
        dc.dispatch_fused(x, idx, w)
    assert e.value.code == ep.EP_ERR_UNSUPPORTED
