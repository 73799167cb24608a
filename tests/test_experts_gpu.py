"""Expert-major path on the GPU against the CPU oracle, bit for bit:
ep_dispatch_layout_experts (both its one-CTA and its chunked kernels),
ep_dispatch into the expert-major rows (bf16 and FP8), and
ep_combine_weighted (expert-major with the gate weights, and rank-major)."""
import numpy as np
import pytest
import torch

import combine_ep_dispatch_gb300 as ep
import oracle
from combine_ep_dispatch_gb300.inputs import f32_from_bf16_bits, make_bf16, make_inputs, make_routing
from gpu_util import SENT_BF16, SENT_I32, assert_rows_equal, run_dispatch, to_dev_bf16, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def run_layout_experts(topk_idx: np.ndarray, E: int, idx_dev=None) -> dict:
    T, k = topk_idx.shape
    if idx_dev is None:
        idx_dev = torch.from_numpy(np.ascontiguousarray(topk_idx, np.int32)).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    ne = torch.full((E,), SENT_I32, **i32)
    off = torch.full((E + 1,), SENT_I32, **i32)
    slot = torch.full((T, k), SENT_I32, **i32)
    ws = torch.full((max(ep.ep_layout_experts_workspace_bytes(T, k, E), 16),), 0x5A,
                    dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, **i32)
    ep.ep_dispatch_layout_experts(idx_dev, E, ne, off, slot, ws, st)
    torch.cuda.synchronize()
    return {"num_tokens_per_expert": ne.cpu().numpy(), "expert_offset": off.cpu().numpy(),
            "slot": slot.cpu().numpy(), "status": int(st.item())}


def run_combine_weighted(y: np.ndarray, slot: np.ndarray, w: np.ndarray, H: int,
                         cap: int | None = None) -> dict:
    T = slot.shape[0]
    yd = to_dev_bf16(y)
    if cap is not None and cap < yd.shape[0]:
        yd = yd[:cap].contiguous()
    out = torch.full((T, H), SENT_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.ep_combine_weighted(yd, torch.from_numpy(np.ascontiguousarray(slot, np.int32)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda(), out, st)
    torch.cuda.synchronize()
    return {"out": u16(out), "status": int(st.item())}


def _check_layout(idx, E, idx_dev=None):
    want = oracle.layout_experts(idx, E)
    got = run_layout_experts(idx, E, idx_dev)
    for key in ("num_tokens_per_expert", "expert_offset", "slot"):
        assert_rows_equal(got[key], want[key], key)
    assert bool(got["status"] & ep.EP_STATUS_BAD_EXPERT) == bool(want["status"] & oracle.STATUS_BAD_EXPERT)
    return want


# ------------------------------------------------------------------ layout

@pytest.mark.parametrize("T,E,k", [
    (0, 256, 8), (1, 256, 8), (5, 16, 2), (128, 256, 8), (1023, 256, 8), (1024, 256, 8),
    (1024, 1024, 8),                          # one CTA, largest expert count
    (1025, 256, 8),                           # 8200 pairs: chunked kernels, ragged last chunk
    (4096, 256, 8), (4096, 128, 8), (9000, 64, 6), (2000, 1500, 4), (3000, 4096, 8),
    (700, 96, 9), (40000, 256, 8),
])
def test_layout_experts_matches_oracle(T, E, k):
    rng = np.random.default_rng(T * 7 + E + k)
    idx = make_routing(rng, T, E, k, "zipf" if (T + E) % 2 else "uniform") if T else \
        np.zeros((0, k), np.int32)
    _check_layout(idx, E)


@pytest.mark.parametrize("T", [300, 5000])
def test_layout_experts_invalid_and_repeated_ids(T):
    rng = np.random.default_rng(T)
    E, k = 128, 8
    idx = make_routing(rng, T, E, k)
    idx[rng.random(idx.shape) < 0.05] = -1
    idx[rng.random(idx.shape) < 0.05] = E + 3
    dup = rng.random(T) < 0.2                 # the same expert twice in a token
    idx[dup, 3] = idx[dup, 2]
    idx[: min(T, 40)] = 7                      # one expert in every column of 40 tokens
    want = _check_layout(idx, E)
    assert want["status"] & oracle.STATUS_BAD_EXPERT


def test_layout_experts_unaligned_ids():
    """topk_idx starting 4 bytes past a 16-byte boundary."""
    rng = np.random.default_rng(5)
    T, E, k = 3001, 256, 8
    idx = make_routing(rng, T, E, k)
    buf = torch.zeros(T * k + 1, dtype=torch.int32, device="cuda")
    buf[1:] = torch.from_numpy(idx.reshape(-1)).cuda()
    _check_layout(idx, E, idx_dev=buf[1:].view(T, k))


def test_layout_experts_large_batch():
    rng = np.random.default_rng(11)
    T, E, k = 120000, 256, 8
    _check_layout(make_routing(rng, T, E, k, "zipf"), E)


# --------------------------------------------------------- dispatch + combine

def _expert_major_round_trip(name, quant, seed):
    inp = make_inputs(name, seed=seed)
    cfg = inp["cfg"]
    idx, w = inp["topk_idx"], inp["topk_w"]
    lay = _check_layout(idx, cfg.E)
    R = int(lay["expert_offset"][-1])
    dis = oracle.dispatch(inp["x"], idx, w, lay["slot"], R, quant=quant)
    got = run_dispatch(inp["x"], idx, w, lay["slot"], R, quant)
    assert_rows_equal(got["recv_x"], dis["recv_x"], "recv_x")
    for key in ("recv_topk_idx", "recv_topk_w", "recv_src"):
        assert_rows_equal(got[key], dis[key], key)
    if quant == ep.EP_QUANT_FP8_E4M3_B128:
        assert_rows_equal(got["recv_scale"], dis["recv_scale"], "recv_scale")
    return inp, lay, dis, R


@pytest.mark.parametrize("name", ["tiny", "decode", "dsv3"])
def test_expert_major_bf16_dispatch_and_weighted_combine(name):
    inp, lay, dis, R = _expert_major_round_trip(name, ep.EP_QUANT_BF16, seed=21)
    cfg = inp["cfg"]
    # expert e's output: its rows scaled by (1 + e mod 3) / 2 (exact in bf16)
    expert_of_row = np.searchsorted(lay["expert_offset"], np.arange(R), side="right") - 1
    f = (1.0 + (expert_of_row % 3)) / 2.0
    y = oracle.bf16_from_f32((f32_from_bf16_bits(dis["recv_x"]) * f[:, None]).astype(np.float32))
    want = oracle.combine_weighted(y, lay["slot"], inp["topk_w"])
    got = run_combine_weighted(y, lay["slot"], inp["topk_w"], cfg.H)
    assert_rows_equal(got["out"], want["out"], "out")
    assert got["status"] == 0


def test_expert_major_fp8_dispatch():
    _expert_major_round_trip("dsv3_zipf_fp8", ep.EP_QUANT_FP8_E4M3_B128, seed=22)


# ---------------------------------------------------------- weighted combine

@pytest.mark.parametrize("T,C,H", [(1, 1, 8), (37, 5, 136), (300, 8, 7168), (1500, 8, 2048),
                                   (5000, 8, 512), (64, 32, 256)])
def test_combine_weighted_random_tables(T, C, H):
    """Random slot tables (repeats, -1 holes) and weights over a wide range,
    half the tokens with cancelling columns whose result shows each FMA's
    single rounding and the column order."""
    rng = np.random.default_rng(T + C + H)
    R = max(2 * T, 4)
    y = make_bf16(rng, (R, H), scale=2.0)
    slot = rng.integers(-1, R, size=(T, C)).astype(np.int32)
    w = (rng.standard_normal((T, C)) * rng.choice([1e-3, 1.0, 50.0], size=(T, C))).astype(np.float32)
    if C >= 3:
        big = (rng.uniform(1.0, 2.0, size=T) * 2.0**20).astype(np.float32)
        for t in range(0, T, 2):
            slot[t, 1] = slot[t, 0] = rng.integers(0, R)
            w[t, 0], w[t, 1] = big[t], -big[t]
            w[t, 2] = np.float32(big[t] * 2.0**-25 * rng.uniform(0.5, 2.0))
    want = oracle.combine_weighted(y, slot, w)
    got = run_combine_weighted(y, slot, w, H)
    assert_rows_equal(got["out"], want["out"], "out")


def test_combine_weighted_unit_weights_equal_plain_combine():
    inp = make_inputs("dsv3", seed=23)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    y = make_bf16(np.random.default_rng(24), (R, cfg.H), scale=3.0)
    ones = np.ones(lay["slot"].shape, np.float32)
    got = run_combine_weighted(y, lay["slot"], ones, cfg.H)
    assert_rows_equal(got["out"], oracle.combine(y, lay["slot"])["out"], "out")


def test_combine_weighted_capacity():
    rng = np.random.default_rng(25)
    T, C, H, R = 400, 8, 256, 1000
    y = make_bf16(rng, (R, H))
    slot = rng.integers(-1, R, size=(T, C)).astype(np.int32)
    w = rng.random((T, C), dtype=np.float32)
    want = oracle.combine_weighted(y[:900], slot, w, cap=900)
    got = run_combine_weighted(y, slot, w, H, cap=900)
    assert_rows_equal(got["out"], want["out"], "out")
    assert got["status"] & ep.EP_STATUS_CAPACITY


def test_combine_weighted_empty_batch():
    got = run_combine_weighted(make_bf16(np.random.default_rng(0), (4, 64)),
                               np.zeros((0, 8), np.int32), np.zeros((0, 8), np.float32), 64)
    assert got["out"].shape == (0, 64) and got["status"] == 0


@pytest.mark.parametrize("name", ["tiny", "dsv3"])
def test_combine_weighted_rank_scaled_experts_closed_form(name):
    """The fused expert epilogue of the pages' combine test (rank r's rows
    scaled by 1 + r) as a weighted rank-major combine of identity experts:
    out[t] = bf16(S_t * x[t]) with S_t = sum over r in D(t) of (1 + r).  x has
    8 significant bits and S_t at most 6, so every product and sum is exact in
    fp32 and the only rounding is the final bf16 one, taken here from
    PyTorch's cast (the dsv3 inputs hold a -0, which the sum from +0 turns
    into +0)."""
    inp = make_inputs(name, seed=4)
    cfg = inp["cfg"]
    dc = ep.DispatchCombine(cfg.T, cfg.H, cfg.E, cfg.k, cfg.W)
    x = to_dev_bf16(inp["x"])
    idx = torch.from_numpy(inp["topk_idx"]).cuda()
    dc.layout_dispatch(x, idx, torch.from_numpy(inp["topk_w"]).cuda())
    slot = dc.slot
    wr = (torch.arange(cfg.W, dtype=torch.float32, device="cuda") + 1.0).expand(cfg.T, cfg.W).contiguous()
    out = dc.combine(dc.recv_x, wr)
    torch.cuda.synchronize()
    S = ((slot >= 0).float() * wr).sum(dim=1, keepdim=True)
    # the sum starts from +0, so a -0 input gives +0 (the combine's reading of signed zero)
    want = (0.0 + x.float() * S).cpu().to(torch.bfloat16)
    assert torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))
    assert int(dc.status.item()) == 0
