"""Pins of the oracle's number encoders (bf16 and FP8 e4m3) against things other
than the oracle: PyTorch's CPU casts (library routines), an exhaustive
nearest-value search over the e4m3 value table, and the format's closed forms."""
import numpy as np
import pytest
import torch

import oracle


def _torch_bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _torch_e4m3_codes(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_table() -> np.ndarray:
    """Value of each code 0..255 decoded by PyTorch (NaN codes stay NaN)."""
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()


# ------------------------------------------------------------------- bf16

def test_bf16_random_bit_patterns_match_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    a = bits.view(np.float32)
    a = a[np.isfinite(a)]
    np.testing.assert_array_equal(oracle.bf16_from_f32(a), _torch_bf16_bits(a))


def test_bf16_all_ties_and_neighbours_match_torch():
    hi = np.arange(0, 1 << 16, dtype=np.uint32)
    for low in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF, 0x0001):
        bits = (hi << 16) | np.uint32(low)
        a = bits.view(np.float32)
        a = a[np.isfinite(a)]
        np.testing.assert_array_equal(oracle.bf16_from_f32(a), _torch_bf16_bits(a))


def test_bf16_ties_go_to_even_closed_form():
    # 1 + 2^-8 lies half way between 1 and 1 + 2^-7: ties to the even 1.0
    # 1 + 3*2^-8 lies half way between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6
    a = np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8)], np.float32)
    np.testing.assert_array_equal(oracle.bf16_from_f32(a), np.array([0x3F80, 0x3F82, 0xBF80], np.uint16))


# ------------------------------------------------------------------- e4m3

def test_e4m3_table_closed_form():
    """The decoded value of every finite code from the format's definition."""
    tab = _e4m3_table()
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(tab[c])
            continue
        v = m * 2.0**-9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert tab[c] == (-v if s else v), c
    assert tab[0x7E] == 448.0 and tab[0x01] == 2.0**-9 and tab[0x08] == 2.0**-6


def test_e4m3_roundtrip_all_codes():
    tab = _e4m3_table()
    codes = np.array([c for c in range(256) if not np.isnan(tab[c])], np.uint8)
    back = oracle.e4m3_from_f32(tab[codes])
    np.testing.assert_array_equal(back, codes)
    np.testing.assert_array_equal(oracle.f32_from_e4m3(codes), tab[codes])


def _sweep_values(rng) -> np.ndarray:
    """fp32 values with |v| <= 448: every (sign, exponent, top 11 mantissa bits)
    with several low-bit fills, plus all the e4m3 midpoints and their neighbours."""
    hi = np.arange(0, 1 << 20, dtype=np.uint32) << 12
    lows = [np.uint32(0), np.uint32(0x800), np.uint32(0x7FF), np.uint32(0x801), np.uint32(0xFFF)]
    parts = [hi | lo for lo in lows]
    parts.append(hi | rng.integers(0, 1 << 12, size=hi.size, dtype=np.uint32))
    a = np.concatenate(parts).view(np.float32)
    tab = _e4m3_table()
    fin = np.unique(np.abs(tab[np.isfinite(tab)]))
    mids = ((fin[1:].astype(np.float64) + fin[:-1]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    m = np.concatenate([mids, up, dn])
    a = np.concatenate([a, m, -m])
    a = a[np.isfinite(a)]
    return a[np.abs(a) <= 448.0]


def test_e4m3_matches_torch_cast_within_range():
    a = _sweep_values(np.random.default_rng(2))
    assert a.size > 3_000_000
    np.testing.assert_array_equal(oracle.e4m3_from_f32(a), _torch_e4m3_codes(a))


def test_e4m3_every_nonnegative_pattern_up_to_448_matches_torch():
    """Every fp32 bit pattern from +0 to 448 (1.14e9 values, in chunks)
    against PyTorch's float8_e4m3fn cast; negative values on a stride-7
    subsample of the same range (the sign only sets bit 7)."""
    lim = int(np.float32(448.0).view(np.uint32))
    chunk = 1 << 24
    for start in range(0, lim + 1, chunk):
        bits = np.arange(start, min(start + chunk, lim + 1), dtype=np.uint32)
        a = bits.view(np.float32)
        assert np.array_equal(oracle.e4m3_from_f32(a), _torch_e4m3_codes(a)), start
        neg = (bits[::7] | np.uint32(0x80000000)).view(np.float32)
        assert np.array_equal(oracle.e4m3_from_f32(neg), _torch_e4m3_codes(neg)), start


def _e4m3_nearest_bruteforce(a: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 value by exhaustive search over the value table in
    float64; ties to the code with an even mantissa; magnitudes >= 448 saturate."""
    tab = _e4m3_table().astype(np.float64)
    pos_codes = np.array([c for c in range(127)], np.int64)     # 0x00..0x7E
    pos_vals = tab[pos_codes]
    mag = np.abs(a.astype(np.float64))
    d = np.abs(mag[:, None] - pos_vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = (pos_codes[None, :] & 1) == 0
    n_cand = cand.sum(axis=1)
    pick = np.where(n_cand[:, None] > 1, cand & even, cand)
    code = pos_codes[np.argmax(pick, axis=1)]
    code = np.where(mag >= 448.0, 0x7E, code)
    sign = np.signbit(a).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def test_e4m3_matches_exhaustive_nearest_value():
    rng = np.random.default_rng(3)
    a = _sweep_values(rng)
    sample = np.concatenate([rng.choice(a, 150_000, replace=False),
                             np.array([1000.0, -1e30, 464.0, 470.0, 449.0, -450.0], np.float32)])
    np.testing.assert_array_equal(oracle.e4m3_from_f32(sample), _e4m3_nearest_bruteforce(sample))


def test_e4m3_all_midpoints_tie_to_even():
    tab = _e4m3_table()
    fin = np.unique(np.abs(tab[np.isfinite(tab)])).astype(np.float64)  # +0 once
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (fin[1:] + fin[:-1]) / 2)  # exact in fp32
    codes = oracle.e4m3_from_f32(mids)
    assert np.all((codes & 1) == 0)
    lo = oracle.e4m3_from_f32(fin[:-1].astype(np.float32))
    hi = oracle.e4m3_from_f32(fin[1:].astype(np.float32))
    assert np.all((codes == lo) | (codes == hi))


def test_e4m3_saturation_and_signed_zero():
    a = np.array([448.0, 449.0, 464.0, 1e9, -1e9, -464.0, 0.0, -0.0, 2.0**-10, -(2.0**-10)], np.float32)
    # 2^-10 is a quarter of the smallest subnormal 2^-9: rounds to (signed) zero
    np.testing.assert_array_equal(
        oracle.e4m3_from_f32(a), np.array([0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x00, 0x80, 0x00, 0x80], np.uint8))
