"""Pins of the oracle's codecs against the format specifications, library
conversions and brute force (no GPU)."""
import os

import numpy as np
import pytest
import torch

from oracle import codecs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n").split("\t") for ln in f if ln.strip() and not ln.startswith("#")]


def test_e2m1_decode_matches_ocp_table():
    for code, value in _rows("e2m1_values.txt"):
        got = float(codecs.e2m1_decode(int(code)))
        assert got == float(value)
        assert np.signbit(got) == value.startswith("-")


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = codecs.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_landmarks():
    for _, hexcode, value in _rows("e4m3_limits.txt"):
        assert float(codecs.e4m3_decode(int(hexcode, 16))) == float(value)
        assert int(codecs.e4m3_encode(float(value))) == int(hexcode, 16)


def _brute_encode(v, decode, ncodes, signbit):
    """Nearest finite code by exhaustive search; ties to the even code;
    saturating."""
    out = []
    cand = [(c, decode(c)) for c in range(ncodes)]
    cand = [(c, float(x)) for c, x in cand if np.isfinite(x) and not np.signbit(x)]
    vmax = max(x for _, x in cand)
    for x in np.atleast_1d(v):
        m = min(abs(float(x)), vmax)
        best = min(cand, key=lambda cx: (abs(cx[1] - m), cx[0] % 2))
        out.append(best[0] | (signbit if np.signbit(x) else 0))
    return np.array(out, dtype=np.uint8)


def test_e2m1_encode_brute_force_and_ties():
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.default_rng(1)
    v = np.concatenate([grid, -grid, mids, -mids, rng.uniform(-8, 8, 500), [7.0, -100.0, 6.0001]])
    got = codecs.e2m1_encode(v)
    ref = _brute_encode(v, lambda c: codecs.e2m1_decode(c), 8, 0x8)
    assert np.array_equal(got, ref)
    # Ties go to the even code: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2,
    # 2.5 -> 2, 3.5 -> 4, 5 -> 4.
    assert list(codecs.e2m1_encode(mids)) == [0, 2, 2, 4, 4, 6, 6]


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.uniform(-464, 464, 4000),
        np.exp2(rng.uniform(-12, 8.8, 4000)),
        codecs.e4m3_decode(np.arange(0, 0x7F)),
    ]).astype(np.float32)
    mids = (codecs.e4m3_decode(np.arange(1, 0x7F)) + codecs.e4m3_decode(np.arange(0, 0x7E))) / 2
    v = np.concatenate([v, mids.astype(np.float32)])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.e4m3_encode(v.astype(np.float64))
    assert np.array_equal(got, ref)
    # satfinite: beyond the largest finite value the code is 448, never NaN
    assert list(codecs.e4m3_encode([470.0, 1e9, -1e30])) == [0x7E, 0x7E, 0xFE]
    # brute force over a slice of the range, including subnormal ties
    w = np.concatenate([np.arange(0, 40) * 2.0**-11, rng.uniform(0, 2, 200)])
    assert np.array_equal(codecs.e4m3_encode(w), _brute_encode(w, lambda c: codecs.e4m3_decode(c), 128, 0x80))


def test_bf16_round_matches_torch_from_fp32():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-6, 6, 5000), [0.0, 1.0, -3.0]])
    v = v.astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(codecs.round_to_bf16(v.astype(np.float64)), ref)
    bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codecs.bf16_bits_to_f64(bits), ref)
    assert np.array_equal(codecs.bf16_bits(ref), bits)


def test_bf16_round_from_fp64_is_single_rounding():
    # 1 + 2^-8 + 2^-30 lies just above the bf16 midpoint 1 + 2^-8 between 1
    # and 1 + 2^-7: one rounding gives 1 + 2^-7; a detour through fp32 would
    # first land exactly on the midpoint and then tie to even 1.0.
    x = 1.0 + 2.0**-8 + 2.0**-30
    assert codecs.round_to_bf16(x) == 1.0 + 2.0**-7
    assert codecs.round_to_bf16(1.0 + 2.0**-8) == 1.0  # exact tie -> even
    assert codecs.round_to_bf16(1.0 + 3 * 2.0**-8) == 1.0 + 2 * 2.0**-7  # tie -> even


def test_nibble_pack_order():
    codes = np.array([1, 2, 3, 4], dtype=np.uint8)
    assert list(codecs.pack_nibbles(codes)) == [0x21, 0x43]
    assert np.array_equal(codecs.unpack_nibbles(codecs.pack_nibbles(codes)), codes)


@pytest.mark.parametrize("n", [2, 16, 64])
def test_nibble_roundtrip(n):
    b = np.random.default_rng(n).integers(0, 256, (3, n), dtype=np.uint8)
    assert np.array_equal(codecs.pack_nibbles(codecs.unpack_nibbles(b)), b)
