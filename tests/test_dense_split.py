"""Host model of the dense projection's stream-K work split (no GPU).

For few tokens, dense_bf16_kernel cuts the (tile, K = 64 step) space,
tile-major, into one contiguous range per CTA: CTA c takes steps
[c W / G, (c + 1) W / G) of W = tiles * KC. A range splits into segments,
one per tile it touches. A segment covering a whole tile is stored directly.
Otherwise it writes an fp32 partial into its CTA's slot 0 (the CTA's first
tile) or slot 1 (its last). A tile's partials are summed by the last of its
segments to arrive, over the CTAs c_first..c_last that touch it, found as the
largest c with floor(c W / G) <= x. This model checks the properties the
kernel relies on for every shape class it can meet."""
import pytest


def segments(c, G, tiles, KC):
    W = tiles * KC
    x, end = c * W // G, (c + 1) * W // G
    out = []
    while x < end:
        t = x // KC
        e = min(end, (t + 1) * KC)
        out.append((t, x - t * KC, e - t * KC))
        x = e
    return out


def cta_of(x, W, G):
    return ((x + 1) * G + W - 1) // W - 1


def check_split(tiles, KC, slots):
    W = tiles * KC
    G = min(W, slots)  # the host never launches more CTAs than steps
    cover, writes, whole = {}, {}, {}
    for c in range(G):
        segs = segments(c, G, tiles, KC)
        assert segs, "every CTA has work"
        first_tile = (c * W // G) // KC
        for t, k0, k1 in segs:
            for k in range(k0, k1):
                assert (t, k) not in cover
                cover[(t, k)] = c
            if k0 == 0 and k1 == KC:
                whole[t] = whole.get(t, 0) + 1
            else:
                slot = 2 * c + (0 if t == first_tile else 1)
                assert 0 <= slot < 2 * G
                writes.setdefault(t, []).append(slot)
    assert len(cover) == W  # every step once
    all_slots = [s for v in writes.values() for s in v]
    assert len(all_slots) == len(set(all_slots))  # no slot serves two tiles
    for t in range(tiles):
        cf, cl = cta_of(t * KC, W, G), cta_of((t + 1) * KC - 1, W, G)
        assert 0 <= cf <= cl < G
        assert cover[(t, 0)] == cf and cover[(t, KC - 1)] == cl
        if t in whole:  # one CTA owns the tile: stored directly, no counter
            assert whole[t] == 1 and cf == cl and t not in writes
        else:
            got = writes[t]
            # the counter's target is the number of CTAs touching the tile
            assert len(got) == cl - cf + 1
            # the reducer's slots (CTA order) are exactly the written ones
            want = [2 * c + (0 if t == (c * W // G) // KC else 1) for c in range(cf, cl + 1)]
            assert sorted(want) == sorted(got)


@pytest.mark.parametrize("KC", [1, 2, 3, 5, 16, 32, 80, 81])
@pytest.mark.parametrize("slots", [1, 2, 7, 40, 152, 304])
def test_split_covers_each_step_once_and_the_fix_up_finds_every_partial(KC, slots):
    for tiles in list(range(1, 45)) + [80, 120, 607]:
        check_split(tiles, KC, slots)


def test_pooler_decode_shape():
    """T = 8 through 5120 x 5120: 40 tiles of 80 steps over 304 CTAs, so
    each CTA takes 10 or 11 steps and a tile is shared by 8 or 9 CTAs."""
    check_split(40, 80, 304)
    counts = [len(segments(c, 304, 40, 80)) for c in range(304)]
    assert max(counts) == 2
