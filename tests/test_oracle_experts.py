"""Pins of the oracle's expert-major layout and weighted combine against a
hand-worked fixture, a restatement by stable sorting, brute force over every tiny
routing, and an exact rational evaluation of the fused multiply-add chain.  CPU
only."""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from combine_ep_dispatch_gb300.inputs import f32_from_bf16_bits, make_bf16, make_inputs, make_routing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(vals) -> np.ndarray:
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _sorted_layout(topk_idx, E):
    """Restatement: number the valid (token, column) pairs in the order of a
    stable sort on the expert id; counts by tallies, offsets by cumulative sum."""
    T, k = topk_idx.shape
    flat = topk_idx.reshape(-1).astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    pos = np.nonzero(valid)[0]
    order = pos[np.argsort(flat[pos], kind="stable")]
    slot = -np.ones(T * k, np.int32)
    slot[order] = np.arange(order.size, dtype=np.int32)
    ne = np.bincount(flat[valid], minlength=E).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(ne)]).astype(np.int32)
    return ne, off, slot.reshape(T, k), bool(np.any(~valid))


# ------------------------------------------------------------ expert layout

def test_layout_experts_golden_hand_example():
    g = _golden("layout_experts_tiny.json")
    lay = oracle.layout_experts(np.array(g["topk_idx"], np.int32), g["E"])
    ex = g["expect"]
    np.testing.assert_array_equal(lay["num_tokens_per_expert"], ex["num_tokens_per_expert"])
    np.testing.assert_array_equal(lay["expert_offset"], ex["expert_offset"])
    np.testing.assert_array_equal(lay["slot"], ex["slot"])
    assert bool(lay["status"] & oracle.STATUS_BAD_EXPERT) == ex["status_bad_expert"]


@pytest.mark.parametrize("T,k", [(3, 2), (2, 3), (4, 1)])
def test_layout_experts_bruteforce_every_tiny_routing(T, k):
    """Every routing of T tokens over ids -1..E (both ends invalid), duplicates
    within a token included."""
    E = 3
    ids = list(range(-1, E + 1))
    for flat in itertools.product(ids, repeat=T * k):
        idx = np.array(flat, np.int32).reshape(T, k)
        lay = oracle.layout_experts(idx, E)
        ne, off, slot, bad = _sorted_layout(idx, E)
        np.testing.assert_array_equal(lay["slot"], slot)
        np.testing.assert_array_equal(lay["num_tokens_per_expert"], ne)
        np.testing.assert_array_equal(lay["expert_offset"], off)
        assert bool(lay["status"] & oracle.STATUS_BAD_EXPERT) == bad


@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_layout_experts_random_matches_sorting(dist):
    rng = np.random.default_rng(71)
    T, E, k = 3000, 96, 6
    idx = make_routing(rng, T, E, k, dist)
    idx[rng.random(idx.shape) < 0.03] = E + 2
    dup = rng.random(T) < 0.1           # the same expert twice in a token
    idx[dup, 1] = idx[dup, 0]
    lay = oracle.layout_experts(idx, E)
    ne, off, slot, bad = _sorted_layout(idx, E)
    np.testing.assert_array_equal(lay["slot"], slot)
    np.testing.assert_array_equal(lay["expert_offset"], off)
    assert bool(lay["status"] & oracle.STATUS_BAD_EXPERT) == bad


@pytest.mark.parametrize("name", ["tiny", "dsv3", "qwen"])
def test_layout_experts_agrees_with_rank_layout(name):
    """Per-expert counts equal the rank layout's; the rows of rank r are the
    range offset[r*Er] .. offset[(r+1)*Er]; every valid pair has its own row,
    and within an expert rows follow token order."""
    inp = make_inputs(name, seed=5)
    cfg = inp["cfg"]
    idx = inp["topk_idx"]
    ex = oracle.layout_experts(idx, cfg.E)
    rk = oracle.layout(idx, cfg.E, cfg.W)
    np.testing.assert_array_equal(ex["num_tokens_per_expert"], rk["num_tokens_per_expert"])
    valid = (idx >= 0) & (idx < cfg.E)
    s = ex["slot"][valid]
    assert np.array_equal(np.sort(s), np.arange(valid.sum()))
    e = idx[valid]
    assert np.all((s >= ex["expert_offset"][e]) & (s < ex["expert_offset"][e + 1]))
    tok = np.nonzero(valid)[0]
    order = np.argsort(s)
    e_sorted, t_sorted = e[order], tok[order]
    same = e_sorted[1:] == e_sorted[:-1]
    assert np.all(t_sorted[1:][same] >= t_sorted[:-1][same])
    per_rank_pairs = np.add.reduceat(ex["num_tokens_per_expert"], np.arange(0, cfg.E, cfg.Er))
    np.testing.assert_array_equal(np.diff(ex["expert_offset"][::cfg.Er]), per_rank_pairs)


# -------------------------------------------------------- weighted combine

def _fraction_of_f32(v) -> Fraction:
    return Fraction(float(np.float32(v)))


def _round_f32(q: Fraction) -> np.float32:
    """Correctly rounded fp32 of an exact rational (ties to even) by search over
    the neighbours of a first guess; finite, normal-range values only."""
    f = np.float32(float(q))
    best = None
    for c in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        d = abs(Fraction(float(c)) - q)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(c).view(np.uint32)) & 1) == 0):
            best = (d, np.float32(c))
    return best[1]


def _fma_chain_exact(y, slot, w):
    """The combine by exact rationals: per token and column, acc = RN32(w*y + acc)
    with the product never rounded; +0 start; bf16 RNE at the end via torch."""
    T, C = slot.shape
    H = y.shape[1]
    yf = f32_from_bf16_bits(y)
    out = np.zeros((T, H), np.float32)
    for t in range(T):
        for h in range(H):
            acc = np.float32(0.0)
            for c in range(C):
                s = slot[t, c]
                if s < 0:
                    continue
                # acc never holds -0: it starts at +0 and an exact zero rounds to +0
                acc = _round_f32(_fraction_of_f32(w[t, c]) * _fraction_of_f32(yf[s, h]) + _fraction_of_f32(acc))
            out[t, h] = acc
    return _bf16(out)


def test_combine_weighted_golden_hand_example():
    g = _golden("layout_experts_tiny.json")
    lay = oracle.layout_experts(np.array(g["topk_idx"], np.int32), g["E"])
    c = g["combine"]
    out = oracle.combine_weighted(_bf16(c["y"]), lay["slot"], np.array(c["topk_w"], np.float32))["out"]
    np.testing.assert_array_equal(f32_from_bf16_bits(out), np.array(c["out"], np.float32))


def test_combine_weighted_rounds_each_step_once():
    s = _golden("layout_experts_tiny.json")["single_rounding"]
    w = np.array(s["w_bits"], np.uint32).view(np.float32)
    out = oracle.combine_weighted(_bf16(s["y"]), np.array(s["slot"], np.int32), w)["out"]
    got = f32_from_bf16_bits(out)[0]
    assert got[0] == np.float32(s["out"][0])
    assert got[0] != np.float32(s["out_if_product_rounded_first"][0])


def _cancelling_case(rng, T, C, H, R):
    """Random slots and weights; in every other token columns 0 and 1 hold the
    same row with weights W and -W and column 2 a weight near W * 2^-25.  Then
    column 1 leaves exactly the rounding error of the column-0 product, which is
    as large as the column-2 term: the result shows whether each product enters
    unrounded and whether the columns are taken in ascending order."""
    y = make_bf16(rng, (R, H), scale=2.0)
    slot = rng.integers(-1, R, size=(T, C)).astype(np.int32)
    w = (rng.standard_normal((T, C)) * rng.choice([1e-3, 1.0, 50.0], size=(T, C))).astype(np.float32)
    big = (rng.uniform(1.0, 2.0, size=T) * 2.0**20).astype(np.float32)
    for t in range(0, T, 2):
        slot[t, 1] = slot[t, 0] = rng.integers(0, R)
        slot[t, 2] = rng.integers(0, R)
        w[t, 0], w[t, 1] = big[t], -big[t]
        w[t, 2] = np.float32(big[t] * 2.0**-25 * rng.uniform(0.5, 2.0))
    return y, slot, w


def test_combine_weighted_matches_exact_rational_chain():
    rng = np.random.default_rng(81)
    y, slot, w = _cancelling_case(rng, T=32, C=5, H=32, R=40)
    got = oracle.combine_weighted(y, slot, w)["out"]
    np.testing.assert_array_equal(got, _fma_chain_exact(y, slot, w))


def test_combine_weighted_unit_weights_is_plain_combine():
    """fma(1, y, acc) rounds y + acc once, exactly as the plain combine's add."""
    inp = make_inputs("tiny", seed=14)
    cfg = inp["cfg"]
    lay = oracle.layout(inp["topk_idx"], cfg.E, cfg.W)
    R = int(lay["rank_offset"][-1])
    y = make_bf16(np.random.default_rng(15), (R, cfg.H), scale=4.0)
    ones = np.ones(lay["slot"].shape, np.float32)
    np.testing.assert_array_equal(oracle.combine_weighted(y, lay["slot"], ones)["out"],
                                  oracle.combine(y, lay["slot"])["out"])


def test_combine_weighted_capacity_rows_are_skipped_and_flagged():
    rng = np.random.default_rng(16)
    T, C, H, R = 30, 4, 8, 50
    y = make_bf16(rng, (R, H))
    slot = rng.integers(-1, R, size=(T, C)).astype(np.int32)
    w = rng.random((T, C), dtype=np.float32)
    res = oracle.combine_weighted(y[:40], slot, w, cap=40)
    assert res["status"] & oracle.STATUS_CAPACITY
    cut = slot.copy()
    cut[cut >= 40] = -1
    np.testing.assert_array_equal(res["out"], oracle.combine_weighted(y, cut, w)["out"])


def test_expert_major_round_trip_power_of_two_weights():
    """Dispatch into the expert-major layout, expert output = the row itself,
    weights 2^-j: every product and partial sum is exact, so the combine is
    bf16(sum_j 2^-j x_t) over the token's valid columns."""
    inp = make_inputs("decode", seed=6)
    cfg = inp["cfg"]
    idx = inp["topk_idx"]
    lay = oracle.layout_experts(idx, cfg.E)
    R = int(lay["expert_offset"][-1])
    w = np.broadcast_to((2.0 ** -np.arange(cfg.k)).astype(np.float32), idx.shape).copy()
    dis = oracle.dispatch(inp["x"], idx, w, lay["slot"], R)
    np.testing.assert_array_equal(dis["recv_src"][lay["slot"]], np.arange(cfg.T)[:, None].repeat(cfg.k, 1))
    out = oracle.combine_weighted(dis["recv_x"], lay["slot"], w)["out"]
    xf = f32_from_bf16_bits(inp["x"]).astype(np.float64)
    m = ((idx >= 0) & (idx < cfg.E)) * w
    want = _bf16(xf * m.sum(axis=1)[:, None])
    want[want == 0x8000] = 0
    np.testing.assert_array_equal(out, want)
