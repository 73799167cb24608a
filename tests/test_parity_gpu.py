"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element
by element, on the same seeded inputs.  Integer, index and byte outputs and the
bf16 combine (fixed ascending-rank fp32 order) must be bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import (CONFIGS, f32_from_bf16_bits, make_bf16, make_inputs,
                                              make_routing)
from gpu_util import (SENT_BF16, SENT_I32, SENT_U8, assert_rows_equal, run_combine, run_dispatch,
                      run_layout, to_dev_bf16)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _check_layout(idx, E, W):
    want = oracle.layout(idx, E, W)
    got = run_layout(idx, E, W)
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_offset", "slot"):
        assert_rows_equal(got[key], want[key], key)
    assert got["status"] == want["status"]
    return want


def _check_dispatch(inp, lay, cap, quant, with_meta=True):
    want = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], cap, quant)
    got = run_dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], cap, quant,
                       with_meta=with_meta)
    R = min(int(lay["rank_offset"][-1]), cap)
    assert got["status"] == want["status"]
    assert_rows_equal(got["recv_x"][:R], want["recv_x"][:R], "recv_x")
    if quant == ep.EP_QUANT_FP8_E4M3_B128:
        assert_rows_equal(got["recv_scale"][:R].view(np.uint32), want["recv_scale"][:R].view(np.uint32),
                          "recv_scale")
    if with_meta:
        assert_rows_equal(got["recv_topk_idx"][:R], want["recv_topk_idx"][:R], "recv_topk_idx")
        assert_rows_equal(got["recv_topk_w"][:R].view(np.uint32), want["recv_topk_w"][:R].view(np.uint32),
                          "recv_topk_w")
        assert_rows_equal(got["recv_src"][:R], want["recv_src"][:R], "recv_src")
    # rows beyond R are never written
    sent = SENT_BF16 if quant == ep.EP_QUANT_BF16 else SENT_U8
    assert np.all(got["recv_x"][R:] == sent)
    if with_meta:
        assert np.all(got["recv_src"][R:] == SENT_I32)
    return want, got


# ------------------------------------------------------------ all workloads

@pytest.mark.parametrize("name", list(CONFIGS))
def test_workload_parity_full(name):
    """Every output of layout, dispatch and combine, bit for bit, at full size."""
    inp = make_inputs(name, seed=0)
    cfg = inp["cfg"]
    quant = ep.EP_QUANT_FP8_E4M3_B128 if cfg.quant == "fp8" else ep.EP_QUANT_BF16
    lay = _check_layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    cap = ep.ep_max_recv_rows(cfg.T, cfg.k, cfg.W)
    _check_dispatch(inp, lay, cap, quant)
    # combine: random expert outputs (bf16) for every receive row
    y = make_bf16(np.random.default_rng(100), (R, cfg.H))
    want = oracle.combine(y, lay["slot"])
    got = run_combine(y, lay["slot"], cfg.H)
    assert got["status"] == want["status"] == 0
    assert_rows_equal(got["out"], want["out"], "combine out")


@pytest.mark.parametrize("name", ["tiny", "decode", "qwen", "dsv3"])
def test_identity_experts_end_to_end(name):
    """combine(dispatch(x)) with identity experts = bf16(d_t * x), exactly."""
    inp = make_inputs(name, seed=1)
    cfg = inp["cfg"]
    xd = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).cuda()
    idx = torch.from_numpy(inp["topk_idx"]).cuda()
    w = torch.from_numpy(inp["topk_w"]).cuda()
    dc = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W)
    out = dc.step(xd, idx, w)
    torch.cuda.synchronize()
    d = np.array([len({int(e) // cfg.Er for e in row}) for row in inp["topk_idx"]])
    want = torch.from_numpy(f32_from_bf16_bits(inp["x"]) * d[:, None].astype(np.float32)).to(
        torch.bfloat16).view(torch.int16)
    want[want == -32768] = 0        # the sum starts from +0, so x = -0 gives +0
    got = out.cpu()
    assert torch.equal(got.view(torch.int16), want)
    assert dc.status.item() == 0


def test_rank_tagged_experts():
    """y = 2^r * row for rows of rank r: out = bf16(M_t * x), M_t = sum of 2^r."""
    inp = make_inputs("decode", seed=2)
    cfg = inp["cfg"]
    lay = _check_layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    dis = run_dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], R, ep.EP_QUANT_BF16)
    rank_of_row = np.searchsorted(lay["rank_offset"], np.arange(R), side="right") - 1
    yf = f32_from_bf16_bits(dis["recv_x"]) * (2.0 ** rank_of_row)[:, None].astype(np.float32)
    y = torch.from_numpy(yf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = run_combine(y, lay["slot"], cfg.H)
    m = np.array([sum(2 ** r for r in {int(e) // cfg.Er for e in row}) for row in inp["topk_idx"]])
    want = torch.from_numpy(f32_from_bf16_bits(inp["x"]) * m[:, None].astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    want[want == 0x8000] = 0        # the sum starts from +0, so x = -0 gives +0
    assert_rows_equal(got["out"], want, "rank-tagged combine")


def test_combine_golden_order():
    with open(os.path.join(GOLDEN, "combine_order.json")) as f:
        g = json.load(f)
    lay = _check_layout(np.array(g["topk_idx"], np.int32), g["E"], g["W"])
    y = torch.tensor(g["y_by_rank"], dtype=torch.float32)[:, None].expand(-1, 64).to(torch.bfloat16)
    y = y.contiguous().view(torch.int16).numpy().view(np.uint16)
    got = run_combine(y, lay["slot"], 64)
    assert np.all(f32_from_bf16_bits(got["out"]) == np.float32(g["out"]))


def test_golden_hand_example():
    with open(os.path.join(GOLDEN, "layout_combine_tiny.json")) as f:
        g = json.load(f)
    idx = np.array(g["topk_idx"], np.int32)
    got = run_layout(idx, g["E"], g["W"])
    np.testing.assert_array_equal(got["slot"], g["expect"]["slot"])
    np.testing.assert_array_equal(got["rank_offset"], g["expect"]["rank_offset"])
    np.testing.assert_array_equal(got["num_tokens_per_expert"], g["expect"]["num_tokens_per_expert"])
    assert got["status"] & ep.EP_STATUS_BAD_EXPERT
    # combine needs H % 8 == 0: pad the 2-column rows with zeros
    y = np.zeros((6, 8), np.float32)
    y[:, :2] = np.array(g["combine"]["y"], np.float32)
    yb = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out = run_combine(yb, got["slot"], 8)["out"]
    outf = f32_from_bf16_bits(out)[:, :2]
    np.testing.assert_array_equal(outf, np.array(g["combine"]["out"], np.float32))
    np.testing.assert_array_equal(np.signbit(outf), np.array(g["combine"]["out_sign_bits_negative"]))


# ------------------------------------------------------------ shapes and edges

@pytest.mark.parametrize("T,H,E,k,W", [
    (0, 256, 16, 4, 4),        # empty
    (1, 8, 4, 2, 2),           # one token, one 16-byte chunk per row
    (257, 264, 64, 6, 8),      # ragged tokens (one past a chunk) and ragged columns
    (1000, 7168, 256, 8, 8),   # several layout chunks, not a multiple of anything
    (333, 4096, 128, 8, 8),
    (300, 512, 64, 16, 32),    # W = 32: up to 16 destinations (two groups of 8)
    (200, 136, 7, 3, 1),       # W = 1, odd E
    (513, 1024, 96, 5, 3),     # W not a power of two
])
def test_shapes_bf16(T, H, E, k, W):
    rng = np.random.default_rng(T * 7 + H)
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k) if T else np.zeros((0, k), np.int32)
    w = rng.random((T, k), dtype=np.float32)
    inp = {"x": x, "topk_idx": idx, "topk_w": w}
    lay = _check_layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    cap = max(R, 1)
    _check_dispatch(inp, lay, cap, ep.EP_QUANT_BF16)
    y = make_bf16(rng, (cap, H))
    want = oracle.combine(y, lay["slot"])["out"]
    got = run_combine(y, lay["slot"], H)["out"]
    assert_rows_equal(got, want, "combine")


@pytest.mark.parametrize("T,H,E,k,W", [(1, 128, 8, 2, 2), (257, 384, 64, 6, 8), (64, 7168, 256, 8, 8),
                                       (100, 1024, 64, 16, 32), (2000, 7168, 256, 8, 8),
                                       (1500, 1024, 64, 16, 32), (1025, 384, 48, 3, 6),
                                       (9000, 640, 64, 4, 8)])
def test_shapes_fp8(T, H, E, k, W):
    rng = np.random.default_rng(T + H)
    x = make_bf16(rng, (T, H), scale=5.0)
    idx = make_routing(rng, T, E, k)
    w = rng.random((T, k), dtype=np.float32)
    lay = _check_layout(idx, E, W)
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, int(lay["rank_offset"][-1]),
                    ep.EP_QUANT_FP8_E4M3_B128)


@pytest.mark.parametrize("T,H,E,k,W", [(2048, 7168, 256, 8, 8), (3001, 512, 64, 6, 8),
                                       (4096, 1024, 64, 16, 32), (2500, 2048, 96, 5, 3),
                                       (6000, 4096, 128, 8, 8)])
def test_fp8_large_batches(T, H, E, k, W):
    """Large FP8 batches, ragged and Zipf-skewed, with and without a capacity
    overflow."""
    rng = np.random.default_rng(T * 3 + H)
    x = make_bf16(rng, (T, H), scale=5.0)
    idx = make_routing(rng, T, E, k, "zipf" if T % 2 else "uniform")
    w = rng.random((T, k), dtype=np.float32)
    lay = _check_layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, R, ep.EP_QUANT_FP8_E4M3_B128)
    want, got = _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, R - 300,
                                ep.EP_QUANT_FP8_E4M3_B128)
    assert got["status"] & ep.EP_STATUS_CAPACITY


def test_fp8_large_batch_unaligned_scales():
    """recv_scale only 4-byte aligned (the C ABI's rule for index and scale
    arrays): every scale lands at its place."""
    rng = np.random.default_rng(44)
    T, H, E, k, W = 3000, 1024, 64, 8, 8
    x = make_bf16(rng, (T, H))
    idx = make_routing(rng, T, E, k)
    w = rng.random((T, k), dtype=np.float32)
    lay = oracle.layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    want = oracle.dispatch(x, idx, w, lay["slot"], R, ep.EP_QUANT_FP8_E4M3_B128)
    nb = H // 128
    flat = torch.full((R * nb + 1,), -7.0, dtype=torch.float32, device="cuda")
    rs = flat[1:].view(R, nb)
    rx = torch.full((R, H), 0xA5, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_dispatch(to_dev_bf16(x), torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), W,
                   torch.from_numpy(lay["slot"]).cuda(), rx, None, None, None, rs,
                   ep.EP_QUANT_FP8_E4M3_B128, st)
    torch.cuda.synchronize()
    assert_rows_equal(rx.cpu().numpy(), want["recv_x"], "recv_x")
    assert_rows_equal(rs.cpu().numpy().view(np.uint32), want["recv_scale"].view(np.uint32), "recv_scale")
    assert int(st.item()) == 0


def test_fp8_special_blocks():
    """Zero and -0 blocks, the smallest bf16 subnormal (subnormal fp32 scale),
    the largest bf16 values, exact +-448*2^j values, exact e4m3 ties."""
    rng = np.random.default_rng(21)
    T, H = 8, 1024
    xs = rng.standard_normal((T, H)).astype(np.float32)
    xs[0, :128] = 0.0
    xs[0, 128:256] = -0.0
    xs[1, :128] = 0.0
    xs[1, 7] = 2.0 ** -133
    xs[1, 128:256] = 2.0 ** -133 * rng.integers(-1, 2, 128)
    xs[2, :] = 3.3e38 * np.sign(rng.standard_normal(H))
    xs[3, :128] = 448.0 * 2.0 ** rng.integers(-20, 20, 128)
    # ties of e4m3 after scaling: amax 56 -> scale 0.125, codes of 8*x
    xs[4, :128] = 0.0
    xs[4, 0] = 56.0
    xs[4, 1:9] = [1.0625, 1.1875, -1.0625, 0.0029296875, 1.5 * 2 ** -10, 2.0 ** -12, 2.0 ** -13, 3 * 2.0 ** -13]
    xs[5, :] = rng.standard_normal(H).astype(np.float32) * 1e-30
    xs[6, :] = rng.standard_normal(H).astype(np.float32) * 2.0 ** rng.integers(-60, 60, H)
    x = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx = np.tile(np.array([[0, 5]], np.int32), (T, 1))
    w = np.ones((T, 2), np.float32)
    lay = _check_layout(idx, 8, 4)
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, int(lay["rank_offset"][-1]),
                    ep.EP_QUANT_FP8_E4M3_B128)


def test_fp8_many_values_match_oracle_encoder():
    """Codes for 8M random normal values across many binades."""
    rng = np.random.default_rng(22)
    T, H = 2048, 8192
    xs = (rng.standard_normal((T, H)) * 2.0 ** rng.integers(-30, 30, (T, 1))).astype(np.float32)
    x = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    lay = _check_layout(idx, 1, 1)
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, T, ep.EP_QUANT_FP8_E4M3_B128)


def test_fp8_values_at_e4m3_rounding_boundaries():
    """Values whose quotient x / scale falls on, or within a few fp32 ulps of, a
    midpoint between two e4m3 values (and on exact e4m3 values), where a
    quotient that is not correctly rounded would pick the wrong code."""
    rng = np.random.default_rng(23)
    tab = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    fin = np.unique(np.abs(tab[np.isfinite(tab)])).astype(np.float64)
    mids = (fin[1:] + fin[:-1]) / 2
    targets = np.concatenate([mids, fin])                     # quotients to aim at
    T, H = 1536, 1024
    xs = np.zeros((T, H), np.float32)
    for t in range(T):
        # block scale 2^j exactly: amax = 448 * 2^j; other values x = target * 2^j, so
        # x / scale lands on the target up to the bf16 rounding of x
        j = int(rng.integers(-20, 20))
        blk = rng.choice(targets, H) * 2.0 ** j
        blk[::128] = 448.0 * 2.0 ** j
        blk *= np.where(rng.random(H) < 0.5, -1.0, 1.0)
        xs[t] = blk
    x = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # nudge half of the normal values by one bf16 ulp either way (never zeros,
    # which would turn into NaN patterns)
    nudge = rng.integers(-1, 2, x.shape).astype(np.int32)
    nudge[:, ::128] = 0
    expo = x & 0x7F80
    nudge[(expo == 0) | (expo == 0x7F80)] = 0
    x = (x.astype(np.int32) + nudge * (rng.random(x.shape) < 0.5)).astype(np.uint16)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    lay = _check_layout(idx, 1, 1)
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, T, ep.EP_QUANT_FP8_E4M3_B128)


def test_fp8_every_significand_ratio():
    """bf16 values have 8-bit significands, so x / scale = 448 * x / amax lands
    exactly on e4m3 midpoints far more often than real-valued data would.  One
    block per (amax significand, exponent gap d, sign pattern): the amax is
    m_a * 2^E, the other 127 values are every other significand m * 2^(E - d),
    so every significand ratio m / m_a at 13 gaps is quantised once."""
    rng = np.random.default_rng(24)
    blocks = []
    mant = np.arange(128, 256, dtype=np.float64)
    for m_a in range(128, 256):
        for d in range(0, 13):
            E = int(rng.integers(-30, 30))
            vals = mant * 2.0 ** (E - 7 - d)              # m * 2^(E - d), with m/128 in [1, 2)
            vals = vals[vals != m_a * 2.0 ** (E - 7 - d)] if d == 0 else vals[:127]
            vals = vals[:127]
            blk = np.concatenate([[m_a * 2.0 ** (E - 7)], vals])
            sign = np.where(rng.random(128) < 0.5, -1.0, 1.0)
            blocks.append(blk * sign)
    xs = np.array(blocks, np.float32).reshape(-1, 1024)  # 8 blocks per row
    x = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    T = x.shape[0]
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    lay = _check_layout(idx, 1, 1)
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": w}, lay, T, ep.EP_QUANT_FP8_E4M3_B128)


def test_invalid_expert_ids_are_ignored_and_flagged():
    rng = np.random.default_rng(31)
    T, E, k, W, H = 500, 64, 6, 8, 256
    idx = make_routing(rng, T, E, k)
    idx[rng.random(idx.shape) < 0.1] = -5
    idx[rng.random(idx.shape) < 0.05] = E
    idx[7, :] = 1000                      # a token with no valid id
    lay = _check_layout(idx, E, W)
    assert lay["status"] & oracle.STATUS_BAD_EXPERT
    x = make_bf16(rng, (T, H))
    _check_dispatch({"x": x, "topk_idx": idx, "topk_w": rng.random((T, k), dtype=np.float32)}, lay,
                    max(int(lay["rank_offset"][-1]), 1), ep.EP_QUANT_BF16)
    y = make_bf16(rng, (int(lay["rank_offset"][-1]), H))
    got = run_combine(y, lay["slot"], H)["out"]
    assert_rows_equal(got, oracle.combine(y, lay["slot"])["out"], "combine")
    assert np.all(got[7] == 0)            # no rows: +0


def test_capacity_overflow_flags_and_skips():
    inp = make_inputs("tiny", seed=41)
    cfg = inp["cfg"]
    lay = _check_layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    cap = R - 50
    want, got = _check_dispatch(inp, lay, cap, ep.EP_QUANT_BF16)
    assert got["status"] & ep.EP_STATUS_CAPACITY
    y = make_bf16(np.random.default_rng(42), (R, cfg.H))
    g = run_combine(y, lay["slot"], cfg.H, cap=cap)
    w = oracle.combine(y[:cap], lay["slot"], cap=cap)
    assert g["status"] == w["status"] == ep.EP_STATUS_CAPACITY
    assert_rows_equal(g["out"], w["out"], "combine under capacity")


def test_dispatch_without_metadata_outputs():
    inp = make_inputs("tiny", seed=43)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    _check_dispatch(inp, lay, int(lay["rank_offset"][-1]), ep.EP_QUANT_BF16, with_meta=False)


@pytest.mark.parametrize("T,E,k,W", [(8192, 256, 8, 8), (8193, 256, 8, 8), (20000, 64, 6, 8),
                                     (50000, 128, 8, 32), (30000, 96, 20, 3)])
def test_layout_large_batches(T, E, k, W):
    """Token counts on both sides of the one-CTA layout's limit (8192): the
    larger ones go through the two-kernel layout with its workspace."""
    idx = make_routing(np.random.default_rng(T + k), T, E, k, "zipf" if T % 2 else "uniform")
    idx[np.random.default_rng(T).random(idx.shape) < 0.01] = -2
    _check_layout(idx, E, W)


@pytest.mark.parametrize("k,E,W", [(20, 64, 8), (8, 256, 8), (3, 48, 6)])
def test_layout_unaligned_and_wide_rows(k, E, W):
    """topk_idx rows that are not 16-byte aligned, and k > 16 (scalar id loads)."""
    rng = np.random.default_rng(k * 100 + E)
    T = 777
    idx = make_routing(rng, T, E, k)
    flat = torch.zeros(T * k + 1, dtype=torch.int32, device="cuda")
    flat[1:] = torch.from_numpy(idx.ravel()).cuda()
    dev_idx = flat[1:].view(T, k)               # 4-byte aligned only
    assert dev_idx.data_ptr() % 16 != 0
    want = oracle.layout(idx, E, W)
    i32 = dict(dtype=torch.int32, device="cuda")
    ne, nr = torch.empty(E, **i32), torch.empty(W, **i32)
    off, slot = torch.empty(W + 1, **i32), torch.empty(T, W, **i32)
    ws = torch.empty(ep.ep_layout_workspace_bytes(T, W, E), dtype=torch.uint8, device="cuda")
    ep.ep_dispatch_layout(dev_idx, E, W, ne, nr, off, slot, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slot.cpu().numpy(), want["slot"])
    np.testing.assert_array_equal(ne.cpu().numpy(), want["num_tokens_per_expert"])
    np.testing.assert_array_equal(off.cpu().numpy(), want["rank_offset"])


def test_deterministic_bytes():
    inp = make_inputs("decode", seed=44)
    cfg = inp["cfg"]
    a = run_layout(inp["topk_idx"], cfg.E, cfg.W)
    b = run_layout(inp["topk_idx"], cfg.E, cfg.W)
    np.testing.assert_array_equal(a["slot"], b["slot"])
    R = int(a["rank_offset"][-1])
    y = make_bf16(np.random.default_rng(45), (R, cfg.H))
    o1 = run_combine(y, a["slot"], cfg.H)["out"]
    o2 = run_combine(y, a["slot"], cfg.H)["out"]
    np.testing.assert_array_equal(o1, o2)


def test_host_errors_through_binding():
    inp = make_inputs("tiny", seed=46)
    cfg = inp["cfg"]
    dc = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W)
    idx = torch.from_numpy(inp["topk_idx"]).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    with pytest.raises(ep.EPError) as e:   # shapes fit W = 3, but E % W != 0
        ep.ep_dispatch_layout(idx, cfg.E, 3, dc.num_tokens_per_expert, torch.zeros(3, **i32),
                              torch.zeros(4, **i32), torch.zeros(cfg.T, 3, **i32), dc.workspace,
                              dc.status)
    assert e.value.code == ep.EP_ERR_INVALID_ARG
    small = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch_layout(idx, cfg.E, cfg.W, dc.num_tokens_per_expert, dc.num_tokens_per_rank,
                              dc.rank_offset, dc.slot, small, dc.status)
    assert e.value.code == ep.EP_ERR_WORKSPACE
    x = torch.zeros(cfg.T, cfg.H + 8, dtype=torch.bfloat16, device="cuda")[:, 1:cfg.H + 1]
    with pytest.raises(ValueError):
        ep.ep_dispatch(x, idx, idx.float(), cfg.W, dc.slot, dc.recv_x)      # not contiguous


@pytest.mark.parametrize("name,T,W", [("tiny", None, None), ("dsv3", None, None), ("qwen", 3000, None),
                                      ("tiny", 200, 1)])
def test_localize_expert_ids(name, T, W):
    """ep_localize_expert_ids after dispatch against the oracle's local ids."""
    inp = make_inputs(name, seed=51, T=T)
    cfg = inp["cfg"]
    W = W or cfg.W
    idx = inp["topk_idx"].copy()
    idx[np.random.default_rng(52).random(idx.shape) < 0.02] = -1
    lay = oracle.layout(idx, cfg.E, W)
    R = int(lay["rank_offset"][-1])
    cap = R + 5
    dis = oracle.dispatch(inp["x"], idx, inp["topk_w"], lay["slot"], cap)
    want = oracle.localize_ids(dis["recv_topk_idx"], cfg.E, W, lay["rank_offset"])
    ids = torch.from_numpy(dis["recv_topk_idx"]).cuda()
    off = torch.from_numpy(lay["rank_offset"]).cuda()
    ep.ep_localize_expert_ids(ids, off, cfg.E, W)
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    assert_rows_equal(got[:R], want[:R], "local ids")
    np.testing.assert_array_equal(got[R:], dis["recv_topk_idx"][R:])   # rows beyond R untouched
