"""Pins of the oracle's prepared layout and the expert-TP layout identity
(no GPU)."""
import numpy as np
import pytest

from oracle import layout


def _raw(E, H, I, seed=0):
    rng = np.random.default_rng(seed)
    return {
        "w13": rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8),
        "w13_sf": rng.integers(0, 256, (E, 2 * I, H // 16), dtype=np.uint8),
        "w2": rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
        "w2_sf": rng.integers(0, 256, (E, H, I // 16), dtype=np.uint8),
    }


def test_round_trip():
    raw = _raw(3, 256, 192)
    p = layout.prepare(raw["w13"], raw["w13_sf"], raw["w2"], raw["w2_sf"])
    back = layout.unprepare(p)
    for k in raw:
        assert np.array_equal(back[k], raw[k])


def test_scale_atom_bytes_by_index():
    """Scalar index arithmetic for a few scales, against the vectorised
    packer: prepared row r, block b lands in atom (r // 128, b // 4) at byte
    16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4."""
    E, H, I = 2, 256, 128
    raw = _raw(E, H, I, seed=1)
    p = layout.prepare(raw["w13"], raw["w13_sf"], raw["w2"], raw["w2_sf"])
    for e, r, b in [(0, 0, 0), (1, 33, 5), (0, 127, 15), (1, 200, 9), (0, 255, 3)]:
        src = 16 * (r // 32) + r % 32 if r % 32 < 16 else I + 16 * (r // 32) + r % 32 - 16
        byte = 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4
        assert p["w13_sf"][e, r // 128, b // 4, byte] == raw["w13_sf"][e, src, b]
        assert np.array_equal(p["w13"][e, r], raw["w13"][e, src])
    for e, r, b in [(0, 5, 7), (1, 130, 2), (1, 255, 7)]:
        byte = 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4
        assert p["w2_sf"][e, r // 128, b // 4, byte] == raw["w2_sf"][e, r, b]


def test_gate_up_granules():
    I = 64
    src = layout.w13_source_row(np.arange(2 * I), I)
    assert list(src[:32]) == list(range(16)) + list(range(64, 80))
    assert list(src[32:64]) == list(range(16, 32)) + list(range(80, 96))
    assert sorted(src) == list(range(2 * I))


@pytest.mark.parametrize("I,tp", [(256, 2), (512, 4), (512, 8), (2048, 8)])
def test_tp_slice_layout_identity(I, tp):
    """The expert_tp page: a TP slice of the converted layout is, byte for
    byte, the converted layout of the TP slice (I' % 64 == 0, H % 128 == 0)."""
    E, H = 2, 256
    raw = _raw(E, H, I, seed=I + tp)
    p = layout.prepare(raw["w13"], raw["w13_sf"], raw["w2"], raw["w2_sf"])
    for r in range(tp):
        s = layout.raw_slice(raw, r, tp)
        want = layout.prepare(s["w13"], s["w13_sf"], s["w2"], s["w2_sf"])
        got = layout.prepared_slice_view(p, r, tp)
        for k in want:
            assert np.array_equal(got[k], want[k]), (k, r)


def test_identity_needs_whole_atoms():
    """With I' % 64 != 0 a slice of the scale atoms is not the slice's own
    layout (the slice does not even have one)."""
    assert layout.unsupported(1, 256, 96) is not None
    assert layout.unsupported(1, 192, 128) is not None
    assert layout.unsupported(1, 256, 128) is None
    with pytest.raises(ValueError):
        layout.prepare(*(_raw(1, 256, 96)[k] for k in ("w13", "w13_sf", "w2", "w2_sf")))
