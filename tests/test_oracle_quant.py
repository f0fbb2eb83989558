"""Pins of the oracle's NVFP4 quantizer (no GPU)."""
import os

import numpy as np
import pytest

from oracle import codecs, quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _worked():
    d = {}
    with open(os.path.join(GOLDEN, "nvfp4_block_worked.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, v = ln.rstrip("\n").split("\t")
                d[k] = v.split()
    return d


def test_worked_block():
    d = _worked()
    v = np.array([float(x) for x in d["values"]], dtype=np.float32)
    q, sf = quant.quantize_blocks(v[None, :], 1.0)
    assert list(q[0]) == [int(c) for c in d["codes"]]
    assert int(sf[0, 0]) == int(d["sf"][0], 16)


def test_zero_block_and_underflow():
    v = np.zeros((2, 32), dtype=np.float32)
    v[1, 16:] = 1e-30  # amax * g / 6 below half the smallest e4m3 subnormal
    q, sf = quant.quantize_blocks(v, 1.0)
    assert not q.any() and not sf.any()


def test_saturation():
    v = np.full((1, 16), 1e6, dtype=np.float32)
    v[0, 0] = -3e6
    q, sf = quant.quantize_blocks(v, 1.0)
    assert sf[0, 0] == 0x7E  # 448
    assert q[0, 0] == 0xF  # -6
    # 1e6 / 448 = 2232 -> saturates to 6 as well
    assert (q[0, 1:] == 0x7).all()


@pytest.mark.parametrize("j", [-3, 1, 4])
def test_power_of_two_scaling_invariance(j):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((4, 64)).astype(np.float32)
    q0, sf0 = quant.quantize_blocks(v, 8.0)
    q1, sf1 = quant.quantize_blocks(v, 8.0 * 2.0**j)
    assert np.array_equal(q0, q1)
    assert np.array_equal(codecs.e4m3_decode(sf1), codecs.e4m3_decode(sf0) * 2.0**j)


def test_representable_blocks_round_trip():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 16, (8, 16)).astype(np.uint8)
    codes[:, 0] = 7  # amax = 6 * scale exactly
    scale = codecs.e4m3_decode(rng.integers(0x20, 0x60, 8))
    v = codecs.e2m1_decode(codes) * scale[:, None]
    q, sf = quant.quantize_blocks(v.astype(np.float32), 1.0)
    assert np.array_equal(codecs.e4m3_decode(sf[:, 0]), scale)
    assert np.array_equal(codecs.e2m1_decode(q), codecs.e2m1_decode(codes))


def test_error_within_half_step():
    """Brute-force: every code is the nearest e2m1 value to v * g / sf."""
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((16, 64)) * 3).astype(np.float32)
    g = np.float32(37.5)
    q, sf = quant.quantize_blocks(v, g)
    s = codecs.e4m3_decode(np.repeat(sf, 16, axis=1))
    t = v.astype(np.float64) * g / s
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    best = np.abs(np.abs(t)[..., None] - grid).min(-1)
    got = np.abs(np.abs(t) - np.abs(codecs.e2m1_decode(q)))
    assert (got <= best + 1e-6 * np.abs(t) + 1e-12).all()
    # sf is the e4m3 nearest to amax * g / 6
    amax = np.abs(v.reshape(16, 4, 16)).max(-1).astype(np.float64)
    target = amax * g / 6
    grid8 = codecs.e4m3_decode(np.arange(0, 0x7F))
    near = np.abs(target[..., None] - grid8).min(-1)
    assert (np.abs(codecs.e4m3_decode(sf) - target) <= near + 1e-9 * target).all()


def test_pack_layout():
    v = np.arange(16, dtype=np.float32)[None, :] / 3
    q, _ = quant.quantize_blocks(v, 1.0)
    p, _ = quant.quantize_rows_packed(v, 1.0)
    assert np.array_equal(p[0] & 0xF, q[0, 0::2]) and np.array_equal(p[0] >> 4, q[0, 1::2])


def _rel_dist_to_midpoints(x, grid):
    """Relative distance of each |x| to the nearest rounding boundary (the
    midpoints between consecutive representable magnitudes)."""
    mids = (grid[1:] + grid[:-1]) / 2.0
    ax = np.abs(np.asarray(x, dtype=np.float64))
    i = np.clip(np.searchsorted(mids, ax), 1, len(mids) - 1)
    d = np.minimum(np.abs(ax - mids[i - 1]), np.abs(ax - mids[i]))
    return d / np.maximum(ax, np.finfo(np.float64).tiny)


@pytest.mark.parametrize("kind,g", [("bf16", 531.7), ("bf16", 2.25), ("h", 97.3), ("h", 1.0)])
def test_fp32_order_agrees_with_exact_definition(kind, g):
    """The oracle quantizer takes its decisions in fp32, in the kernel's
    operation order (s = fp32(amax g)/6, inv = g/sf, t = v inv). Held against
    the definition evaluated exactly (fp64: sf = e4m3(amax g / 6), q =
    e2m1(v g / sf)): they agree on every block scale and code except where the
    exact quotient lies within 2^-20 (relative) of a rounding boundary; there
    they differ by at most one code step, and such elements are at most 1e-3
    of all."""
    rng = np.random.default_rng(11)
    if kind == "bf16":
        v = codecs.bf16_bits_to_f64(
            (np.frombuffer(rng.standard_normal(1 << 18).astype(np.float32).tobytes(), np.uint32) >> 16)
            .astype(np.uint16)).astype(np.float32)
    else:  # fp32 values shaped like the SwiGLU output: heavy-tailed
        a, b = rng.standard_normal((2, 1 << 18))
        v = (a / (1.0 + np.exp(-a)) * b * 37.0).astype(np.float32)
    v = v.reshape(-1, 256)
    g32 = np.float32(g)
    q, sf = quant.quantize_blocks(v, g32)

    blocks = v.astype(np.float64).reshape(v.shape[0], -1, 16)
    s_exact = np.max(np.abs(blocks), axis=-1) * float(g32) / 6.0
    sf_exact = codecs.e4m3_encode(s_exact)
    sfv = codecs.e4m3_decode(sf_exact)
    with np.errstate(divide="ignore", invalid="ignore"):
        t_exact = np.where(sfv[..., None] > 0, blocks * float(g32) / sfv[..., None], 0.0)
    q_exact = np.where(sfv[..., None] > 0, codecs.e2m1_encode(t_exact), 0).astype(np.uint8).reshape(v.shape)

    e4m3_grid = np.unique(np.abs(codecs.e4m3_decode(np.arange(256))[np.isfinite(codecs.e4m3_decode(np.arange(256)))]))
    e2m1_grid = np.unique(np.abs(codecs.e2m1_decode(np.arange(16))))
    near_sf = _rel_dist_to_midpoints(s_exact, e4m3_grid) < 2.0**-20
    near_q = (_rel_dist_to_midpoints(t_exact, e2m1_grid) < 2.0**-20) | near_sf[..., None]
    near_q = near_q.reshape(v.shape)

    sf_diff = sf != sf_exact
    assert not (sf_diff & ~near_sf).any()
    assert (np.abs(sf.astype(int) - sf_exact.astype(int))[sf_diff] <= 1).all()
    mag = lambda c: np.abs(codecs.e2m1_decode(c))  # noqa: E731
    step = lambda c: np.searchsorted(e2m1_grid, mag(c))  # noqa: E731
    q_diff = (q & 0x7) != (q_exact & 0x7)
    assert not (q_diff & ~near_q).any()
    assert (np.abs(step(q) - step(q_exact))[q_diff] <= 1).all()
    assert q_diff.mean() <= 1e-3
