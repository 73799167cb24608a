"""Pins of the oracle's layout, dispatch and combine against hand-worked fixtures,
an independent restatement by sorting on tiny routings (brute force over every
routing), closed forms and invariants.  CPU only."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from combine_ep_dispatch_gb300.inputs import (CONFIGS, f32_from_bf16_bits, make_bf16, make_inputs,
                                              make_routing)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(vals) -> np.ndarray:
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _restated_layout(topk_idx, E, W):
    """Independent restatement: collect the distinct (rank, token) pairs, sort them
    rank-major then token, and number them; counts by direct tallies."""
    T, k = topk_idx.shape
    Er = E // W
    pairs = sorted({(int(e) // Er, t) for t in range(T) for e in topk_idx[t] if 0 <= e < E})
    slot = -np.ones((T, W), np.int32)
    for row, (r, t) in enumerate(pairs):
        slot[t, r] = row
    per_rank = np.array([sum(1 for (r, _) in pairs if r == q) for q in range(W)], np.int32)
    per_exp = np.array([int(np.sum(topk_idx == e)) for e in range(E)], np.int32)
    off = np.concatenate([[0], np.cumsum(per_rank)]).astype(np.int32)
    bad = bool(np.any((topk_idx < 0) | (topk_idx >= E)))
    return per_exp, per_rank, off, slot, bad


# ------------------------------------------------------------------ layout

def test_layout_golden_hand_example():
    g = _golden("layout_combine_tiny.json")
    idx = np.array(g["topk_idx"], np.int32)
    lay = oracle.layout(idx, g["E"], g["W"])
    ex = g["expect"]
    np.testing.assert_array_equal(lay["num_tokens_per_expert"], ex["num_tokens_per_expert"])
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], ex["num_tokens_per_rank"])
    np.testing.assert_array_equal(lay["rank_offset"], ex["rank_offset"])
    np.testing.assert_array_equal(lay["slot"], ex["slot"])
    assert bool(lay["status"] & oracle.STATUS_BAD_EXPERT) == ex["status_bad_expert"]


@pytest.mark.parametrize("k", [1, 2])
def test_layout_bruteforce_every_tiny_routing(k):
    E, W = 4, 2
    ids = [-1, 0, 1, 2, 3, 4]          # includes both kinds of out-of-range id
    n = 0
    for T in range(0, 4):
        for flat in itertools.product(ids, repeat=T * k):
            idx = np.array(flat, np.int32).reshape(T, k)
            lay = oracle.layout(idx, E, W)
            pe, pr, off, slot, bad = _restated_layout(idx, E, W)
            assert np.array_equal(lay["num_tokens_per_expert"], pe)
            assert np.array_equal(lay["num_tokens_per_rank"], pr)
            assert np.array_equal(lay["rank_offset"], off)
            assert np.array_equal(lay["slot"], slot)
            assert bool(lay["status"] & oracle.STATUS_BAD_EXPERT) == bad
            n += 1
    assert n == sum(len(ids) ** (T * k) for T in range(4))


def test_layout_random_mid_size_matches_restatement():
    rng = np.random.default_rng(5)
    for T, E, W, k in [(37, 12, 3, 3), (100, 64, 8, 6), (64, 32, 32, 4), (50, 7, 1, 2)]:
        idx = make_routing(rng, T, E, k)
        idx[rng.random(idx.shape) < 0.05] = E + 3    # a few invalid ids
        lay = oracle.layout(idx, E, W)
        pe, pr, off, slot, bad = _restated_layout(idx, E, W)
        np.testing.assert_array_equal(lay["slot"], slot)
        np.testing.assert_array_equal(lay["num_tokens_per_expert"], pe)
        np.testing.assert_array_equal(lay["rank_offset"], off)
        assert bool(lay["status"]) == bad


@pytest.mark.parametrize("name", list(CONFIGS))
def test_layout_invariants_on_workloads(name):
    cfg = CONFIGS[name]
    rng = np.random.default_rng(0)
    idx = make_routing(rng, cfg.T, cfg.E, cfg.k, cfg.routing, cfg.zipf_s)
    lay = oracle.layout(idx, cfg.E, cfg.W)
    slot = lay["slot"]
    # pre-dedup counts sum to T*k (all ids valid)
    assert lay["num_tokens_per_expert"].sum() == cfg.T * cfg.k
    assert lay["status"] == 0
    # per-token copies equal the number of distinct destination ranks
    d = np.array([len({int(e) // cfg.Er for e in row}) for row in idx])
    np.testing.assert_array_equal((slot >= 0).sum(axis=1), d)
    R = int(d.sum())
    assert lay["rank_offset"][-1] == R == lay["num_tokens_per_rank"].sum()
    # the slots of each rank are its row range, increasing in token order
    for r in range(cfg.W):
        s = slot[:, r][slot[:, r] >= 0]
        np.testing.assert_array_equal(s, np.arange(lay["rank_offset"][r], lay["rank_offset"][r + 1]))


def test_zipf_routing_is_skewed_towards_rank0():
    cfg = CONFIGS["dsv3_zipf_fp8"]
    idx = make_routing(np.random.default_rng(0), cfg.T, cfg.E, cfg.k, "zipf", cfg.zipf_s)
    lay = oracle.layout(idx, cfg.E, cfg.W)
    nr = lay["num_tokens_per_rank"]
    assert nr[0] == nr.max() and nr[0] > 0.95 * cfg.T
    assert np.all(np.diff(lay["num_tokens_per_expert"][:8]) <= 0) or nr[0] > nr[-1]


# ---------------------------------------------------------------- dispatch

def test_dispatch_bf16_rows_are_source_rows():
    inp = make_inputs("tiny", seed=7)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    dis = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], R)
    src = dis["recv_src"]
    assert np.all(src >= 0)
    np.testing.assert_array_equal(dis["recv_x"], inp["x"][src])
    np.testing.assert_array_equal(dis["recv_topk_idx"], inp["topk_idx"][src])
    np.testing.assert_array_equal(dis["recv_topk_w"].view(np.uint32), inp["topk_w"][src].view(np.uint32))
    # rows ordered by (rank, token): region r holds ascending tokens, all routed to r
    for r in range(cfg.W):
        a, b = lay["rank_offset"][r], lay["rank_offset"][r + 1]
        toks = src[a:b]
        assert np.all(np.diff(toks) > 0)
        assert all(r in {int(e) // cfg.Er for e in inp["topk_idx"][t]} for t in toks)
    # copies per token = number of distinct destination ranks
    d = np.array([len({int(e) // cfg.Er for e in row}) for row in inp["topk_idx"]])
    np.testing.assert_array_equal(np.bincount(src, minlength=cfg.T), d)


def test_dispatch_capacity_overflow_flags_and_skips():
    inp = make_inputs("tiny", seed=8)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    cap = R - 17
    dis = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], cap, fill=0xABCD)
    assert dis["status"] & oracle.STATUS_CAPACITY
    full = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], R)
    np.testing.assert_array_equal(dis["recv_x"], full["recv_x"][:cap])


def test_dispatch_fp8_golden_block():
    g = _golden("fp8_block.json")
    H = g["H"]
    xs = np.zeros(H, np.float32)
    for i, v in g["x"].items():
        xs[int(i)] = v
    x = _bf16(xs).reshape(1, H)
    assert np.array_equal(f32_from_bf16_bits(x)[0], xs)    # fixture values exact in bf16
    idx = np.array([[0]], np.int32)
    w = np.ones((1, 1), np.float32)
    slot = np.array([[0]], np.int32)
    dis = oracle.dispatch(x, idx, w, slot, 1, oracle.QUANT_FP8)
    assert dis["recv_scale"][0, 0] == np.float32(g["scale"])
    want = np.zeros(H, np.uint8)
    for i, c in g["codes"].items():
        want[int(i)] = c
    np.testing.assert_array_equal(dis["recv_x"][0], want)


def test_dispatch_fp8_quotient_golden_block():
    """A block whose scale is not a power of two: the IEEE quotient x/scale
    lands exactly on e4m3 midpoints (ties to even), while x times the rounded
    reciprocal of the scale lands one fp32 ulp above them and rounds up."""
    g = _golden("fp8_quotient_block.json")
    H = g["H"]
    xs = np.zeros(H, np.float32)
    for i, v in g["x"].items():
        xs[int(i)] = v
    x = _bf16(xs).reshape(1, H)
    assert np.array_equal(f32_from_bf16_bits(x)[0], xs)    # fixture values exact in bf16
    dis = oracle.dispatch(x, np.array([[0]], np.int32), np.ones((1, 1), np.float32),
                          np.array([[0]], np.int32), 1, oracle.QUANT_FP8)
    assert hex(int(dis["recv_scale"][0, 0:1].view(np.uint32)[0])) == g["scale_bits"]
    want = np.zeros(H, np.uint8)
    for i, c in g["codes"].items():
        want[int(i)] = c
    np.testing.assert_array_equal(dis["recv_x"][0], want)
    # the fixture tells the two quotients apart: the reciprocal form's codes differ
    assert any(g["codes"][i] != g["codes_if_reciprocal_multiply"][i] for i in g["codes"])


def test_dispatch_fp8_codes_match_library_cast_of_ieee_quotient():
    """1M values in blocks of N(0,1) * 2^j (non-power-of-two scales): the
    oracle's scales equal numpy's fp32 amax / 448 bit for bit, and its codes
    equal PyTorch's float8_e4m3fn cast of numpy's fp32 quotient x / scale,
    saturated at +-448 (the library cast does not saturate).  About 0.1% of the
    codes change when the quotient is taken as x * (1 / scale)."""
    rng = np.random.default_rng(2024)
    T, H = 128, 8192
    nb = H // 128
    xs = rng.standard_normal((T, H)).astype(np.float32)
    xs *= np.repeat(2.0 ** rng.integers(-24, 24, (T, nb)), 128, axis=1).astype(np.float32)
    x = _bf16(xs)
    xf = f32_from_bf16_bits(x)
    slot = np.arange(T, dtype=np.int32).reshape(T, 1)
    dis = oracle.dispatch(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32), slot, T,
                          oracle.QUANT_FP8)
    amax = np.abs(xf.reshape(T, nb, 128)).max(axis=2)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    np.testing.assert_array_equal(dis["recv_scale"].view(np.uint32), scale.view(np.uint32))
    assert np.all(scale > 0)
    q = (xf / np.repeat(scale, 128, axis=1)).astype(np.float32)
    want = torch.from_numpy(np.clip(q, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(dis["recv_x"], want)
    rcp = (xf * np.repeat((np.float32(1.0) / scale).astype(np.float32), 128, axis=1)).astype(np.float32)
    other = torch.from_numpy(np.clip(rcp, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.count_nonzero(other != want) > 100    # the sweep separates the two readings


def test_dispatch_fp8_closed_forms():
    rng = np.random.default_rng(11)
    T, H = 6, 512
    xs = rng.standard_normal((T, H)).astype(np.float32)
    # token 1: a block of +-448*2^j exact values; token 2: an all-zero block and a
    # block of -0; token 3: a block whose only non-zero is the smallest bf16
    # subnormal, so that the scale is an fp32 subnormal
    xs[1, :128] = 448.0 * 2.0 ** rng.integers(-12, -4, 128) * np.where(rng.random(128) < 0.5, -1, 1)
    xs[2, 128:256] = 0.0
    xs[2, 256:384] = -0.0
    xs[3, 0:128] = 0.0
    xs[3, 5] = 2.0 ** -133                   # smallest bf16 subnormal
    x = _bf16(xs)
    idx = np.arange(T, dtype=np.int32).reshape(T, 1)
    w = np.ones((T, 1), np.float32)
    slot = np.arange(T, dtype=np.int32).reshape(T, 1)
    dis = oracle.dispatch(x, idx, w, slot, T, oracle.QUANT_FP8)
    q, sc = dis["recv_x"], dis["recv_scale"]
    xf = f32_from_bf16_bits(x)
    # scale = amax/448 with amax = max |x| (exact)
    amax = np.abs(xf.reshape(T, H // 128, 128)).max(axis=2)
    np.testing.assert_array_equal(sc, (amax / np.float32(448.0)).astype(np.float32))
    # exact +-448*2^j values dequantise exactly
    deq = oracle.f32_from_e4m3(q[1, :128]) * sc[1, 0]
    np.testing.assert_array_equal(deq, xf[1, :128])
    # zero blocks give a zero scale and all-zero codes, even for -0 inputs
    assert sc[2, 1] == 0 and sc[2, 2] == 0
    assert not q[2, 128:384].any()
    # subnormal scale: 2^-133/448 = 146.29 * 2^-149 rounds to 146 * 2^-149, and
    # 2^-133 / that = 2^16/146 = 448.9 saturates to 448 (code 0x7E)
    assert sc[3, 0] == np.float32(146 * 2.0**-149)
    assert q[3, 5] == 0x7E and np.count_nonzero(q[3, :128]) == 1
    # dequantisation error <= half an e4m3 ulp of the code's binade, times scale,
    # plus the rounding of x/scale to fp32
    tab_codes = q.astype(np.int64)
    deq_all = oracle.f32_from_e4m3(q).astype(np.float64) * np.repeat(sc, 128, axis=1)
    e = (tab_codes >> 3) & 15
    ulp = np.where(e == 0, 2.0**-9, 2.0 ** (np.maximum(e, 1) - 10))
    bound = 0.5 * ulp * np.repeat(sc, 128, axis=1) + np.abs(xf) * 2.0**-23
    assert np.all(np.abs(deq_all - xf) <= bound + 1e-45)


# ----------------------------------------------------------------- combine

def test_combine_golden_hand_example():
    g = _golden("layout_combine_tiny.json")
    lay = oracle.layout(np.array(g["topk_idx"], np.int32), g["E"], g["W"])
    c = g["combine"]
    y = _bf16(c["y"])
    out = oracle.combine(y, lay["slot"])["out"]
    outf = f32_from_bf16_bits(out)
    np.testing.assert_array_equal(outf, np.array(c["out"], np.float32))
    np.testing.assert_array_equal(np.signbit(outf), np.array(c["out_sign_bits_negative"]))


def test_combine_fixed_ascending_rank_order():
    g = _golden("combine_order.json")
    idx = np.array(g["topk_idx"], np.int32)
    lay = oracle.layout(idx, g["E"], g["W"])
    y = _bf16(np.array(g["y_by_rank"], np.float32)[:, None] * np.ones((1, 8), np.float32))
    out = f32_from_bf16_bits(oracle.combine(y, lay["slot"])["out"])
    assert np.all(out == np.float32(g["out"]))
    assert g["out_if_descending"] != g["out"]


def _d_and_mask(idx, Er):
    d = np.array([len({int(e) // Er for e in row}) for row in idx])
    m = np.array([sum(2 ** r for r in {int(e) // Er for e in row}) for row in idx])
    return d, m


@pytest.mark.parametrize("name", ["tiny", "decode", "qwen"])
def test_combine_identity_experts_is_d_times_x(name):
    inp = make_inputs(name, seed=3)
    cfg = inp["cfg"]
    run = oracle.run_all(inp)
    d, _ = _d_and_mask(inp["topk_idx"], cfg.Er)
    want = _bf16(f32_from_bf16_bits(inp["x"]).astype(np.float64) * d[:, None])   # exact product
    want[want == 0x8000] = 0      # the sum starts from +0: a -0 input sums to +0
    np.testing.assert_array_equal(run["combine"]["out"], want)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_combine_rank_tagged_experts(name):
    """Expert output of a row of rank r = 2^r * the row (exact in bf16), so the
    sum is M_t * x with M_t = sum of 2^r over the token's ranks: exact in fp32,
    and it shows which ranks were gathered."""
    inp = make_inputs(name, seed=4)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    dis = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_w"], lay["slot"], R)
    rank_of_row = np.searchsorted(lay["rank_offset"], np.arange(R), side="right") - 1
    y = _bf16(f32_from_bf16_bits(dis["recv_x"]) * (2.0 ** rank_of_row)[:, None])
    out = oracle.combine(y, lay["slot"])["out"]
    _, m = _d_and_mask(inp["topk_idx"], cfg.Er)
    want = _bf16(f32_from_bf16_bits(inp["x"]).astype(np.float64) * m[:, None])
    want[want == 0x8000] = 0
    np.testing.assert_array_equal(out, want)


def test_combine_random_rows_within_fp32_error_bound():
    inp = make_inputs("tiny", seed=9)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    y = make_bf16(np.random.default_rng(10), (R, cfg.H), scale=3.0)
    out = f32_from_bf16_bits(oracle.combine(y, lay["slot"])["out"]).astype(np.float64)
    yf = f32_from_bf16_bits(y).astype(np.float64)
    s = np.zeros((cfg.T, cfg.H))
    a = np.zeros((cfg.T, cfg.H))
    for t in range(cfg.T):
        rows = lay["slot"][t][lay["slot"][t] >= 0]
        s[t] = yf[rows].sum(axis=0)
        a[t] = np.abs(yf[rows]).sum(axis=0)
    d = (lay["slot"] >= 0).sum(axis=1)[:, None]
    bound = 2.0**-8 * np.abs(s) + 2.0 * d * 2.0**-24 * a
    assert np.all(np.abs(out - s) <= bound)
    # and the bound is not vacuous: most outputs are the correctly rounded sum
    assert np.mean(out == f32_from_bf16_bits(_bf16(s.astype(np.float32)))) > 0.95


def test_combine_capacity_rows_are_skipped_and_flagged():
    inp = make_inputs("tiny", seed=12)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    y = make_bf16(np.random.default_rng(13), (R, cfg.H))
    res = oracle.combine(y[: R - 5], lay["slot"], cap=R - 5)
    assert res["status"] & oracle.STATUS_CAPACITY
    slot = lay["slot"].copy()
    slot[slot >= R - 5] = -1
    np.testing.assert_array_equal(res["out"], oracle.combine(y, slot)["out"])


def test_localize_ids_golden_hand_example():
    """Hand-worked on the layout fixture (E=8, W=4, two experts per rank): rows
    0-1 are rank 0 (tokens 0, 2), rows 2-3 rank 1 (tokens 0, 3), row 4 rank 2
    (token 1), row 5 rank 3 (token 2)."""
    g = _golden("layout_combine_tiny.json")
    idx = np.array(g["topk_idx"], np.int32)
    lay = oracle.layout(idx, g["E"], g["W"])
    dis = oracle.dispatch(np.zeros((5, 8), np.uint16), idx, np.ones((5, 2), np.float32), lay["slot"], 6)
    local = oracle.localize_ids(dis["recv_topk_idx"], g["E"], g["W"], lay["rank_offset"])
    want = [[0, -1],    # token 0 [0, 3] on rank 0: 0 -> 0, 3 lives on rank 1
            [-1, 1],    # token 2 [7, 1] on rank 0: 1 -> 1
            [-1, 1],    # token 0 on rank 1: 3 -> 3 - 2 = 1
            [-1, 0],    # token 3 [9, 2] on rank 1: 9 invalid, 2 -> 0
            [1, 0],     # token 1 [5, 4] on rank 2: 5 -> 1, 4 -> 0
            [1, -1]]    # token 2 [7, 1] on rank 3: 7 -> 1
    np.testing.assert_array_equal(local, want)


def test_localize_ids_restatement_random():
    rng = np.random.default_rng(61)
    T, E, W, k = 300, 48, 6, 5
    idx = make_routing(rng, T, E, k)
    idx[rng.random(idx.shape) < 0.05] = -4
    lay = oracle.layout(idx, E, W)
    R = int(lay["rank_offset"][-1])
    dis = oracle.dispatch(make_bf16(rng, (T, 8)), idx, rng.random((T, k), dtype=np.float32), lay["slot"], R)
    local = oracle.localize_ids(dis["recv_topk_idx"], E, W, lay["rank_offset"])
    Er = E // W
    for t in range(T):
        for r in range(W):
            s = lay["slot"][t, r]
            if s < 0:
                continue
            want = [e - r * Er if 0 <= e < E and e // Er == r else -1 for e in idx[t]]
            assert list(local[s]) == want
            assert any(v >= 0 for v in want)      # a row is only sent to a rank hosting an expert
