"""Dispatch and combine with each rank's receive rows in an allocation of its
own (ep_dispatch_regions, ep_combine_regions), against the CPU oracle.

Region r must hold exactly what the one-buffer dispatch writes to the global
rows [rank_offset[r], rank_offset[r+1]): the oracle's receive rows of that
range, bit for bit (bf16 rows, FP8 codes and scales, metadata), and nothing
beyond its capacity; the combine reading the regions must equal the oracle's
combine of the same rows laid out in one buffer."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import make_bf16, make_inputs, make_routing

from gpu_util import SENT_BF16, SENT_I32, SENT_U8, assert_rows_equal, to_dev_bf16, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()


def _regions(counts, H, k, quant, short=None):
    """One separate allocation per rank, sentinel-filled; ``short[r]`` rows fewer
    than the rank needs where given."""
    regs = []
    for r, n in enumerate(counts):
        rows = max(int(n) - (short or {}).get(r, 0), 0)
        i32 = dict(dtype=torch.int32, device="cuda")
        if quant == ep.EP_QUANT_BF16:
            rx = torch.full((rows, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
            rs = None
        else:
            rx = torch.full((rows, H), SENT_U8, dtype=torch.uint8, device="cuda")
            rs = torch.full((rows, H // 128), -7.0, dtype=torch.float32, device="cuda")
        regs.append({"recv_x": rx, "recv_scale": rs,
                     "recv_topk_idx": torch.full((rows, k), SENT_I32, **i32),
                     "recv_topk_w": torch.full((rows, k), -3.0, dtype=torch.float32, device="cuda"),
                     "recv_src": torch.full((rows,), SENT_I32, **i32)})
    return regs


def _check(x, idx, w, E, W, quant, short=None):
    T, H = x.shape
    k = idx.shape[1]
    lay = oracle.layout(idx, E, W)
    off = lay["rank_offset"]
    R = int(off[-1])
    want = oracle.dispatch(x, idx, w, lay["slot"], R, quant)
    counts = np.diff(off)
    regs = _regions(counts, H, k, quant, short)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    slot_d = torch.from_numpy(lay["slot"]).cuda()
    off_d = torch.from_numpy(off).cuda()
    ep.ep_dispatch_regions(to_dev_bf16(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(),
                           slot_d, off_d, regs, quant, st)
    torch.cuda.synchronize()
    over = any(int(counts[r]) > regs[r]["recv_x"].shape[0] for r in range(W))
    assert int(st.item()) == (ep.EP_STATUS_CAPACITY if over else 0)
    for r in range(W):
        g = regs[r]
        n = g["recv_x"].shape[0]
        lo = int(off[r])
        got_x = u16(g["recv_x"]) if quant == ep.EP_QUANT_BF16 else g["recv_x"].cpu().numpy()
        assert_rows_equal(got_x, want["recv_x"][lo:lo + n], f"region {r} rows")
        if quant != ep.EP_QUANT_BF16:
            assert_rows_equal(g["recv_scale"].cpu().numpy().view(np.uint32),
                              want["recv_scale"][lo:lo + n].view(np.uint32), f"region {r} scales")
        assert_rows_equal(g["recv_topk_idx"].cpu().numpy(), want["recv_topk_idx"][lo:lo + n],
                          f"region {r} ids")
        assert_rows_equal(g["recv_topk_w"].cpu().numpy().view(np.uint32),
                          want["recv_topk_w"][lo:lo + n].view(np.uint32), f"region {r} weights")
        assert_rows_equal(g["recv_src"].cpu().numpy(), want["recv_src"][lo:lo + n],
                          f"region {r} sources")

    # combine from per-rank regions of expert outputs (rows past a region's
    # capacity are skipped: the oracle gets a slot table without them)
    rng = np.random.default_rng(T + W)
    y = make_bf16(rng, (R, H))
    y_regs = [to_dev_bf16(y[int(off[r]):int(off[r]) + regs[r]["recv_x"].shape[0]])
              for r in range(W)]
    slot_kept = lay["slot"].copy()
    for r in range(W):
        col = slot_kept[:, r]
        col[(col >= 0) & (col - off[r] >= regs[r]["recv_x"].shape[0])] = -1
    out = torch.full((T, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    st.zero_()
    ep.ep_combine_regions(y_regs, slot_d, off_d, out, st)
    torch.cuda.synchronize()
    assert_rows_equal(u16(out), oracle.combine(y, slot_kept)["out"], "combine")
    assert int(st.item()) == (ep.EP_STATUS_CAPACITY if over else 0)


@pytest.mark.parametrize("name,T", [("tiny", None), ("dsv3", None), ("dsv3_zipf_fp8", None),
                                    ("qwen", 3000), ("decode", None)])
def test_regions_workloads(name, T):
    inp = make_inputs(name, seed=61, T=T)
    cfg = inp["cfg"]
    quant = ep.EP_QUANT_FP8_E4M3_B128 if cfg.quant == "fp8" else ep.EP_QUANT_BF16
    _check(inp["x"], inp["topk_idx"], inp["topk_w"], cfg.E, cfg.W, quant)


@pytest.mark.parametrize("quant", [0, 1])
@pytest.mark.parametrize("T,H,E,k,W", [
    (700, 7168, 256, 8, 8),     # bulk-copy rows (bf16)
    (1500, 256, 64, 6, 32),     # 32 ranks, register rows
    (333, 1024, 48, 5, 6),      # W not a power of two
])
def test_regions_short_capacity_and_invalid_ids(quant, T, H, E, k, W):
    if quant == 1 and H % 128:
        pytest.skip("FP8 needs H % 128 == 0")
    rng = np.random.default_rng(T * W + quant)
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k, "zipf")
    idx[rng.random(idx.shape) < 0.03] = -1
    w = rng.random((T, k), dtype=np.float32)
    # rank 0 and the last rank get fewer rows than they need, rank 1 none at all
    counts = np.diff(oracle.layout(idx, E, W)["rank_offset"])
    short = {0: 7, 1: int(counts[1]), W - 1: 1}
    _check(x, idx, w, E, W, quant, short)


def test_regions_match_the_one_buffer_dispatch():
    """The same routing through ep_dispatch (one buffer) and
    ep_dispatch_regions: region r equals rows [rank_offset[r], rank_offset[r+1])."""
    inp = make_inputs("dsv3", seed=62, T=2048)
    cfg = inp["cfg"]
    dc = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W)
    x = to_dev_bf16(inp["x"])
    idx = torch.from_numpy(inp["topk_idx"]).cuda()
    w = torch.from_numpy(inp["topk_w"]).cuda()
    dc.layout_dispatch(x, idx, w)
    torch.cuda.synchronize()
    off = dc.rank_offset.cpu().numpy()
    regs = _regions(np.diff(off), cfg.H, cfg.k, ep.EP_QUANT_BF16)
    ep.ep_dispatch_regions(x, idx, w, dc.slot, dc.rank_offset, regs)
    out = torch.empty_like(dc.out)
    ep.ep_combine_regions([g["recv_x"] for g in regs], dc.slot, dc.rank_offset, out)
    dc.combine()
    torch.cuda.synchronize()
    for r in range(cfg.W):
        assert torch.equal(regs[r]["recv_x"].view(torch.int16),
                           dc.recv_x[off[r]:off[r + 1]].view(torch.int16)), r
        assert torch.equal(regs[r]["recv_src"], dc.recv_src[off[r]:off[r + 1]]), r
    assert torch.equal(out.view(torch.int16), dc.out.view(torch.int16))
    assert int(dc.status.item()) == 0


@pytest.mark.parametrize("name,T,short", [
    ("dsv3", None, False),            # the dispatch finishes the layout (bulk-copy rows, claims)
    ("dsv3_zipf_fp8", None, False),   # FP8, finishing the layout
    ("qwen", 3000, False),
    ("decode", None, False),          # no finishing below 1024 tokens: layout, then dispatch
    ("tiny", None, False),            # register rows
    ("dsv3", 2048, True),             # regions shorter than their ranks' rows
])
def test_regions_with_layout(name, T, short):
    """ep_dispatch_regions_with_layout against the oracle: every layout output,
    and region r bit for bit (rows, FP8 scales, metadata), twice in a row."""
    inp = make_inputs(name, seed=63, T=T)
    cfg = inp["cfg"]
    quant = ep.EP_QUANT_FP8_E4M3_B128 if cfg.quant == "fp8" else ep.EP_QUANT_BF16
    x, idx, w = inp["x"], inp["topk_idx"], inp["topk_w"]
    Tn, H = x.shape
    k = idx.shape[1]
    lay = oracle.layout(idx, cfg.E, cfg.W)
    off = lay["rank_offset"]
    counts = np.diff(off)
    cut = {0: 5, cfg.W - 1: int(counts[-1]) // 2} if short else None
    regs = _regions(counts, H, k, quant, cut)
    i32 = dict(dtype=torch.int32, device="cuda")
    ne = torch.full((cfg.E,), SENT_I32, **i32)
    nr = torch.full((cfg.W,), SENT_I32, **i32)
    ro = torch.full((cfg.W + 1,), SENT_I32, **i32)
    sl = torch.full((Tn, cfg.W), SENT_I32, **i32)
    ws = torch.zeros(ep.ep_layout_workspace_bytes(Tn, cfg.W, cfg.E), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, **i32)
    xd, idd, wd = to_dev_bf16(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    for _ in range(2):
        ep.ep_dispatch_regions_with_layout(xd, idd, wd, cfg.E, ne, nr, ro, sl, ws, regs, quant, st)
    torch.cuda.synchronize()
    for key, got in (("num_tokens_per_expert", ne), ("num_tokens_per_rank", nr),
                     ("rank_offset", ro), ("slot", sl)):
        assert_rows_equal(got.cpu().numpy(), lay[key], key)
    R = int(off[-1])
    want = oracle.dispatch(x, idx, w, lay["slot"], R, quant)
    over = any(int(counts[r]) > regs[r]["recv_x"].shape[0] for r in range(cfg.W))
    assert int(st.item()) == (ep.EP_STATUS_CAPACITY if over else 0)
    for r in range(cfg.W):
        g = regs[r]
        n = g["recv_x"].shape[0]
        lo = int(off[r])
        got_x = u16(g["recv_x"]) if quant == ep.EP_QUANT_BF16 else g["recv_x"].cpu().numpy()
        assert_rows_equal(got_x, want["recv_x"][lo:lo + n], f"region {r} rows")
        if quant != ep.EP_QUANT_BF16:
            assert_rows_equal(g["recv_scale"].cpu().numpy().view(np.uint32),
                              want["recv_scale"][lo:lo + n].view(np.uint32), f"region {r} scales")
        assert_rows_equal(g["recv_topk_idx"].cpu().numpy(), want["recv_topk_idx"][lo:lo + n],
                          f"region {r} ids")
        assert_rows_equal(g["recv_topk_w"].cpu().numpy().view(np.uint32),
                          want["recv_topk_w"][lo:lo + n].view(np.uint32), f"region {r} weights")
        assert_rows_equal(g["recv_src"].cpu().numpy(), want["recv_src"][lo:lo + n],
                          f"region {r} sources")


@pytest.mark.parametrize("seed", range(12))
def test_regions_with_layout_fuzz(seed):
    """Seeded random shapes (ranks, experts, top-k, batch around the 1024-token
    switch, row sizes, routing with invalid ids) through
    ep_dispatch_regions_with_layout and ep_combine_regions, against the
    oracle."""
    rng = np.random.default_rng(7000 + seed)
    W = int(rng.choice([1, 2, 3, 8, 16, 32]))
    E = W * int(rng.integers(1, 17))
    k = int(rng.integers(1, min(E, 9) + 1))
    T = int(rng.choice([0, 1, 300, 1024, 1025, 2500]))
    H = int(rng.choice([256, 1024, 2048, 7168]))
    quant = int(rng.integers(0, 2))
    idx = make_routing(rng, T, E, k, "zipf" if seed % 2 else "uniform") if T else \
        np.zeros((0, k), np.int32)
    if T:
        idx[rng.random(idx.shape) < 0.02] = -1
    x = make_bf16(rng, (T, H))
    w = rng.standard_normal((T, k)).astype(np.float32)
    lay = oracle.layout(idx, E, W)
    off = lay["rank_offset"]
    counts = np.diff(off)
    regs = _regions(counts, H, k, quant)
    i32 = dict(dtype=torch.int32, device="cuda")
    ne, nr = torch.zeros(E, **i32), torch.zeros(W, **i32)
    ro, sl = torch.zeros(W + 1, **i32), torch.zeros((T, W), **i32)
    ws = torch.zeros(max(ep.ep_layout_workspace_bytes(T, W, E), 16), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, **i32)
    xd = to_dev_bf16(x) if T else torch.zeros((0, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_dispatch_regions_with_layout(xd, torch.from_numpy(idx).cuda(),
                                       torch.from_numpy(w).cuda(), E, ne, nr, ro, sl, ws, regs,
                                       quant, st)
    torch.cuda.synchronize()
    assert int(st.item()) == lay["status"]
    for key, got in (("num_tokens_per_expert", ne), ("num_tokens_per_rank", nr),
                     ("rank_offset", ro), ("slot", sl)):
        assert_rows_equal(got.cpu().numpy(), lay[key], key)
    R = int(off[-1])
    want = oracle.dispatch(x, idx, w, lay["slot"], R, quant)
    for r in range(W):
        g = regs[r]
        n = g["recv_x"].shape[0]
        lo = int(off[r])
        got_x = u16(g["recv_x"]) if quant == ep.EP_QUANT_BF16 else g["recv_x"].cpu().numpy()
        assert_rows_equal(got_x, want["recv_x"][lo:lo + n], f"region {r} rows")
        if quant != ep.EP_QUANT_BF16:
            assert_rows_equal(g["recv_scale"].cpu().numpy().view(np.uint32),
                              want["recv_scale"][lo:lo + n].view(np.uint32), f"region {r} scales")
        assert_rows_equal(g["recv_src"].cpu().numpy(), want["recv_src"][lo:lo + n],
                          f"region {r} sources")
    if T and quant == ep.EP_QUANT_BF16:
        out = torch.full((T, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        st.zero_()
        ep.ep_combine_regions([g["recv_x"] for g in regs], sl, ro, out, st)
        torch.cuda.synchronize()
        assert_rows_equal(u16(out), oracle.combine(want["recv_x"][:R], lay["slot"])["out"],
                          "combine of the regions")
