"""GPU parity of ep_dispatch_with_layout (layout and dispatch in one call,
the dispatch loading x while the layout kernels run): every output against the
oracle's layout and dispatch, bit for bit, on both layout paths (one CTA up to
1024 tokens, count + scan above), both payloads, both dispatch kernels (bulk
copies for rows of 1 KB and more, registers below)."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_bf16, make_inputs, make_routing
from gpu_util import SENT_BF16, SENT_I32, SENT_U8, assert_rows_equal, run_with_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _check(x, idx, w, E, W, cap, quant):
    lay = oracle.layout(idx, E, W)
    want = oracle.dispatch(x, idx, w, lay["slot"], cap, quant)
    got = run_with_layout(x, idx, w, E, W, cap, quant)
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
        assert_rows_equal(got[key], lay[key], key)
    assert got["status"] == (lay["status"] | want["status"])
    R = min(int(lay["rank_offset"][-1]), cap)
    assert_rows_equal(got["recv_x"][:R], want["recv_x"][:R], "recv_x")
    if quant == ep.EP_QUANT_FP8_E4M3_B128:
        assert_rows_equal(got["recv_scale"][:R].view(np.uint32),
                          want["recv_scale"][:R].view(np.uint32), "recv_scale")
    assert_rows_equal(got["recv_topk_idx"][:R], want["recv_topk_idx"][:R], "recv_topk_idx")
    assert_rows_equal(got["recv_topk_w"][:R].view(np.uint32),
                      want["recv_topk_w"][:R].view(np.uint32), "recv_topk_w")
    assert_rows_equal(got["recv_src"][:R], want["recv_src"][:R], "recv_src")
    sent = SENT_BF16 if quant == ep.EP_QUANT_BF16 else SENT_U8
    assert np.all(got["recv_x"][R:] == sent)
    assert np.all(got["recv_src"][R:] == SENT_I32)
    return got


@pytest.mark.parametrize("name", ["tiny", "decode", "dsv3", "dsv3_zipf_fp8", "qwen"])
def test_workloads(name):
    inp = make_inputs(name, seed=3)
    cfg = inp["cfg"]
    quant = ep.EP_QUANT_FP8_E4M3_B128 if cfg.quant == "fp8" else ep.EP_QUANT_BF16
    _check(inp["x"], inp["topk_idx"], inp["topk_w"], cfg.E, cfg.W,
           ep.ep_max_recv_rows(cfg.T, cfg.k, cfg.W), quant)


@pytest.mark.parametrize("quant", [0, 1])
@pytest.mark.parametrize("T,H,E,k,W", [
    (1, 7168, 256, 8, 8),       # one token
    (1024, 7168, 256, 8, 8),    # largest one-CTA layout
    (1025, 7168, 256, 8, 8),    # smallest count + scan layout
    (3001, 2048, 64, 6, 8),     # ragged chunks
    (700, 256, 32, 4, 4),       # rows under 1 KB: the register dispatch kernel
    (513, 1536, 96, 3, 6),
    (10000, 7168, 256, 8, 8),   # FP8: one segment per token, longer than the units quantised early
    (2500, 1152, 72, 5, 8),     # FP8: 9 blocks, a partial quadruple in every unit
])
def test_shapes(T, H, E, k, W, quant):
    if quant == ep.EP_QUANT_FP8_E4M3_B128 and H % 128:
        pytest.skip("FP8 needs H % 128 == 0")
    rng = np.random.default_rng(T * 7 + H + quant)
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "uniform")
    w = rng.random((T, k), dtype=np.float32)
    _check(x, idx, w, E, W, ep.ep_max_recv_rows(T, k, W), quant)


@pytest.mark.parametrize("T,H,E,k,W,launches", [
    (16384, 512, 64, 4, 32, 2),    # chunk table exactly 16 KB (128 chunks x 32 ranks)
    (16385, 512, 64, 4, 32, 3),    # one chunk more: count + scan + dispatch
    (65536, 512, 64, 2, 8, 2),     # 512 chunks x 8 ranks, exactly 16 KB
    (5000, 1024, 48, 5, 6, 2),     # W not a multiple of 4
])
def test_finalize_limits(T, H, E, k, W, launches):
    assert ep.ep_dispatch_with_layout_launches(T, H, k, W) == launches
    rng = np.random.default_rng(T + W)
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "uniform")
    w = rng.random((T, k), dtype=np.float32)
    _check(x, idx, w, E, W, ep.ep_max_recv_rows(T, k, W), ep.EP_QUANT_BF16)


@pytest.mark.parametrize("T", [700, 3000])
@pytest.mark.parametrize("quant", [0, 1])
def test_max_experts_and_ranks(T, quant):
    """E = 8192 experts (the rank layout's limit: an 8192-entry histogram in
    shared memory) over W = 32 ranks, one-CTA and chunked layouts, both
    payloads, through both the separate calls and the single call."""
    from gpu_util import run_dispatch, run_layout
    rng = np.random.default_rng(T + quant)
    E, W, k, H = 8192, 32, 8, 1024
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "zipf" if quant else "uniform")
    w = rng.random((T, k), dtype=np.float32)
    lay = oracle.layout(idx, E, W)
    got = run_layout(idx, E, W)
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
        assert_rows_equal(got[key], lay[key], key)
    cap = ep.ep_max_recv_rows(T, k, W)
    want = oracle.dispatch(x, idx, w, lay["slot"], cap, quant)
    R = int(lay["rank_offset"][-1])
    g = run_dispatch(x, idx, w, lay["slot"], cap, quant)
    assert_rows_equal(g["recv_x"][:R], want["recv_x"][:R], "recv_x")
    _check(x, idx, w, E, W, cap, quant)


def test_empty_batch():
    x = np.zeros((0, 7168), np.uint16)
    idx = np.zeros((0, 8), np.int32)
    w = np.zeros((0, 8), np.float32)
    got = run_with_layout(x, idx, w, 256, 8, 16, ep.EP_QUANT_BF16)
    assert np.all(got["num_tokens_per_rank"] == 0) and np.all(got["rank_offset"] == 0)
    assert np.all(got["num_tokens_per_expert"] == 0) and got["status"] == 0


def test_capacity_and_bad_ids_flagged():
    rng = np.random.default_rng(5)
    T, H, E, k, W = 2000, 1024, 64, 4, 8
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "zipf")
    idx[::17, 1] = E + 3   # invalid ids: ignored and flagged
    idx[::29, 2] = -1
    w = rng.random((T, k), dtype=np.float32)
    got = _check(x, idx, w, E, W, 1500, ep.EP_QUANT_BF16)
    assert got["status"] == ep.EP_STATUS_BAD_EXPERT | ep.EP_STATUS_CAPACITY


def test_back_to_back_calls_match_separate_calls():
    """Several steps in a row on one stream (each call's dispatch overlapping
    its own layout, and the next call's layout following the dispatch): the
    receive buffers after the last call equal the layout + dispatch calls'."""
    dev = "cuda"
    inps = [make_inputs("dsv3", seed=s) for s in (11, 12, 13)]
    cfg = inps[0]["cfg"]
    a = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W, device=dev)
    b = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W, device=dev)
    for inp in inps:
        x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
        idx = torch.from_numpy(inp["topk_idx"]).to(dev)
        w = torch.from_numpy(inp["topk_w"]).to(dev)
        for _ in range(3):
            a.layout_dispatch(x, idx, w)
        b.layout(idx)
        b.dispatch(x, idx, w)
        torch.cuda.synchronize()
        R = int(b.rank_offset[cfg.W].item())
        assert torch.equal(a.slot, b.slot) and torch.equal(a.rank_offset, b.rank_offset)
        assert torch.equal(a.recv_x[:R].view(torch.int16), b.recv_x[:R].view(torch.int16))
        assert torch.equal(a.recv_src[:R], b.recv_src[:R])
        assert int(a.status.item()) == 0


# ------------------------------------------------------------ expert-major

def _run_experts_with_layout(x, idx, w, E, cap, quant):
    T, H = x.shape
    k = idx.shape[1]
    i32 = dict(dtype=torch.int32, device="cuda")
    from gpu_util import to_dev_bf16, u16
    ne = torch.full((E,), SENT_I32, **i32)
    off = torch.full((E + 1,), SENT_I32, **i32)
    slot = torch.full((T, k), SENT_I32, **i32)
    ws = torch.full((max(ep.ep_layout_experts_workspace_bytes(T, k, E), 16),), 0x5A,
                    dtype=torch.uint8, device="cuda")
    if quant == ep.EP_QUANT_BF16:
        rx = torch.full((cap, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        rs = None
    else:
        rx = torch.full((cap, H), SENT_U8, dtype=torch.uint8, device="cuda")
        rs = torch.full((cap, H // 128), -7.0, dtype=torch.float32, device="cuda")
    ri = torch.full((cap, k), SENT_I32, **i32)
    rw = torch.full((cap, k), -3.0, dtype=torch.float32, device="cuda")
    rsrc = torch.full((cap,), SENT_I32, **i32)
    st = torch.zeros(1, **i32)
    ep.ep_dispatch_experts_with_layout(
        to_dev_bf16(x), torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda(),
        torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda(), E, ne, off, slot, ws, rx,
        ri, rw, rsrc, rs, quant, st)
    torch.cuda.synchronize()
    out = {"num_tokens_per_expert": ne.cpu().numpy(), "expert_offset": off.cpu().numpy(),
           "slot": slot.cpu().numpy(),
           "recv_x": u16(rx) if quant == ep.EP_QUANT_BF16 else rx.cpu().numpy(),
           "recv_topk_idx": ri.cpu().numpy(), "recv_topk_w": rw.cpu().numpy(),
           "recv_src": rsrc.cpu().numpy(), "status": int(st.item())}
    if rs is not None:
        out["recv_scale"] = rs.cpu().numpy()
    return out


@pytest.mark.parametrize("quant", [0, 1])
@pytest.mark.parametrize("T,H,E,k", [
    (600, 1024, 4096, 8),     # the expert layout's limit: 4096 experts, chunked kernels
    (200, 1024, 64, 8),       # one-CTA expert layout (<= 2048 pairs)
    (4096, 7168, 256, 8),     # dsv3 shape: count + assign kernels
    (3001, 512, 48, 6),       # ragged; rows under 1 KB take the register kernel (bf16)
])
def test_experts_with_layout(T, H, E, k, quant):
    rng = np.random.default_rng(T + H + quant)
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "zipf")
    w = rng.random((T, k), dtype=np.float32)
    lay = oracle.layout_experts(idx, E)
    R = int(lay["expert_offset"][-1])
    want = oracle.dispatch(x, idx, w, lay["slot"], R, quant)
    got = _run_experts_with_layout(x, idx, w, E, R, quant)
    for key in ("num_tokens_per_expert", "expert_offset", "slot"):
        assert_rows_equal(got[key], lay[key], key)
    assert got["status"] == (lay["status"] | want["status"]) == 0
    assert_rows_equal(got["recv_x"], want["recv_x"], "recv_x")
    if quant == ep.EP_QUANT_FP8_E4M3_B128:
        assert_rows_equal(got["recv_scale"].view(np.uint32), want["recv_scale"].view(np.uint32),
                          "recv_scale")
    assert_rows_equal(got["recv_topk_idx"], want["recv_topk_idx"], "recv_topk_idx")
    assert_rows_equal(got["recv_topk_w"].view(np.uint32), want["recv_topk_w"].view(np.uint32),
                      "recv_topk_w")
    assert_rows_equal(got["recv_src"], want["recv_src"], "recv_src")


@pytest.mark.parametrize("T", [300, 2000])
def test_zero_capacity(T):
    """capacity_rows = 0 with recv buffers of zero rows: the layout is still
    complete, nothing is written, and EP_STATUS_CAPACITY is set (the one-launch
    kernel at T = 300, the finishing dispatch at T = 2000)."""
    rng = np.random.default_rng(T)
    H, E, k, W = 1024, 64, 4, 8
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "uniform")
    w = rng.random((T, k), dtype=np.float32)
    got = run_with_layout(x, idx, w, E, W, 0, ep.EP_QUANT_BF16)
    lay = oracle.layout(idx, E, W)
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
        assert_rows_equal(got[key], lay[key], key)
    assert got["status"] == ep.EP_STATUS_CAPACITY


def test_two_streams_do_not_interfere():
    """The library keeps no state between calls: two pipelines with their own
    buffers, interleaved on two streams (one taking the one-launch kernel, one
    the count kernel + finishing dispatch), give the results each gives alone."""
    dev = "cuda"
    setups = []
    for name, T_, seed in (("decode", None, 31), ("dsv3", 2048, 32)):
        inp = make_inputs(name, seed=seed, T=T_)
        cfg = inp["cfg"]
        dc = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W, device=dev)
        x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
        idx = torch.from_numpy(inp["topk_idx"]).to(dev)
        w = torch.from_numpy(inp["topk_w"]).to(dev)
        dc.step(x, idx, w)  # alone, on the current stream
        torch.cuda.synchronize()
        ref = (dc.slot.clone(), dc.out.clone())
        setups.append((dc, x, idx, w, ref, torch.cuda.Stream(device=dev)))
    for _ in range(5):
        for dc, x, idx, w, _ref, s in setups:
            with torch.cuda.stream(s):
                dc.step(x, idx, w, stream=s)
    torch.cuda.synchronize()
    for dc, _x, _idx, _w, (slot, out), _s in setups:
        assert torch.equal(dc.slot, slot)
        assert torch.equal(dc.out.view(torch.int16), out.view(torch.int16))
        assert int(dc.status.item()) == 0


@pytest.mark.parametrize("T", [1825, 4096, 12000])
def test_token_claims_give_the_same_bits_every_call(T):
    """Past the first three tokens per warp the single call's dispatch hands
    out tokens from a counter, so which warp sends which token changes from
    call to call; every output must not.  Twelve calls in a row on one
    workspace (the count kernel zeroes the counter each time) against the
    oracle, T just past the static tokens (3 x 608 warps), at dsv3 and larger."""
    rng = np.random.default_rng(T)
    H, E, k, W = 7168, 256, 8, 8
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "uniform")
    w = rng.random((T, k), dtype=np.float32)
    lay = oracle.layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    want = oracle.dispatch(x, idx, w, lay["slot"], R)
    dc = ep.DispatchCombine(T, H, E, k, W, capacity_rows=R)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    idd, wd = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    first = None
    for i in range(12):
        dc.recv_x.view(torch.int16).fill_(0x7FAB)
        dc.layout_dispatch(xd, idd, wd)
        torch.cuda.synchronize()
        got = (dc.recv_x.view(torch.int16).clone(), dc.slot.clone(), dc.recv_src.clone(),
               dc.recv_topk_w.clone(), dc.num_tokens_per_expert.clone())
        if first is None:
            first = got
            assert_rows_equal(got[0].cpu().numpy().view(np.uint16), want["recv_x"], "recv_x")
            assert_rows_equal(got[1].cpu().numpy(), lay["slot"], "slot")
            assert_rows_equal(got[2].cpu().numpy(), want["recv_src"], "recv_src")
            assert_rows_equal(got[4].cpu().numpy(), lay["num_tokens_per_expert"], "counts")
        else:
            for a, b in zip(got, first):
                assert torch.equal(a, b), i
    assert int(dc.status.item()) == 0
