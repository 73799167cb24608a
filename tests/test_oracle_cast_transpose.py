"""Pins of the oracle's FP8 cast and transposed cast of the expert-major rows:
a hand-worked fixture, the codes against PyTorch's float8_e4m3fn cast of the
fp32 products, the transposed blocks against a numpy transpose of the cast,
and the amax against numpy.  CPU only."""
import json
import os

import numpy as np
import torch

import oracle
from combine_ep_dispatch_gb300.inputs import f32_from_bf16_bits, make_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals) -> np.ndarray:
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _codes_by_torch(q: np.ndarray) -> np.ndarray:
    """e4m3 codes (round to nearest even) by PyTorch's cast; magnitudes above
    448 saturate to +-448 first (the encoder's rule, pinned separately)."""
    q = np.clip(q.astype(np.float32), -448.0, 448.0)
    return torch.from_numpy(np.ascontiguousarray(q)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_cast_transpose_golden_hand_example():
    with open(os.path.join(GOLDEN, "cast_transpose_tiny.json")) as f:
        g = json.load(f)
    res = oracle.cast_transpose(_bf16(g["y"]), np.array(g["expert_offset"], np.int32),
                                np.array(g["scale"], np.float32))
    np.testing.assert_array_equal(res["out_c"], np.array(g["out_c"], np.uint8))
    np.testing.assert_array_equal(res["out_t"], np.array(g["out_t"], np.uint8).ravel())
    np.testing.assert_array_equal(res["amax"], np.array(g["amax"], np.float32))


def test_cast_transpose_random_against_torch_and_numpy():
    rng = np.random.default_rng(91)
    E, H = 9, 96
    n = rng.integers(0, 40, size=E)
    n[3] = 0
    n[5] = 16
    off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    R = int(off[-1])
    y = make_bf16(rng, (R, H), scale=3.0)
    y[rng.random(y.shape) < 0.01] = 0x8000          # some -0
    scale = (2.0 ** rng.uniform(-4, 8, size=E)).astype(np.float32)   # some products saturate
    amax0 = (rng.random(E) * 2).astype(np.float32)
    res = oracle.cast_transpose(y, off, scale, amax0)
    yf = f32_from_bf16_bits(y)
    tb = 0
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        q = (yf[rows] * scale[e]).astype(np.float32)        # IEEE fp32 products
        codes = _codes_by_torch(q)
        np.testing.assert_array_equal(res["out_c"][rows], codes)
        ld = (n[e] + 15) // 16 * 16
        block = res["out_t"][tb:tb + H * ld].reshape(H, ld)
        np.testing.assert_array_equal(block[:, :n[e]], codes.T)
        assert np.all(block[:, n[e]:] == 0)
        tb += H * ld
        want = max(amax0[e], float(np.abs(yf[rows]).max()) if n[e] else 0.0)
        assert res["amax"][e] == np.float32(want)
    assert tb == res["out_t"].size == oracle.cast_transpose_t_bytes(off, H)
