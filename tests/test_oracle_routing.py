"""Pins of the oracle's routing metadata (no GPU)."""
import numpy as np
import pytest

from oracle import routing
from nvfp4_mixture_experts_route_gb300 import inputs


def brute(ids, E, tile):
    """Sort routes by (expert, expanded index); pad each expert's run."""
    T, K = ids.shape
    flat = ids.reshape(-1)
    js = [j for j in range(T * K) if flat[j] >= 0]
    js.sort(key=lambda j: (flat[j], j))
    e2p = -np.ones(T * K, dtype=np.int64)
    p2t = []
    tiles = []
    for e in range(E):
        run = [j for j in js if flat[j] == e]
        if not run:
            continue
        start = len(p2t)
        for j in run:
            e2p[j] = len(p2t)
            p2t.append(j // K)
        while len(p2t) % tile:
            p2t.append(-1)
        for _ in range((len(p2t) - start) // tile):
            tiles.append((e, start + len(run)))
    return e2p.reshape(T, K), p2t, tiles


CASES = [
    ("uniform", 16, 8, 128, 4, 32),
    ("zipf", 64, 8, 128, 8, 32),
    ("uniform", 3, 2, 8, 2, 32),
    ("zipf", 300, 8, 16, 8, 64),
]


@pytest.mark.parametrize("dist,T,K,E,_,tile", CASES)
def test_against_brute_force(dist, T, K, E, _, tile):
    rng = np.random.default_rng(T)
    ids = inputs.draw_topk(rng, T, E, K, dist)
    m = routing.route_metadata(ids, E, tile)
    e2p, p2t, tiles = brute(ids, E, tile)
    assert np.array_equal(m["expanded_to_permuted"], e2p)
    P = len(m["permuted_to_token"])
    assert np.array_equal(m["permuted_to_token"][: len(p2t)], p2t)
    assert (m["permuted_to_token"][len(p2t):] == -1).all()
    n = m["totals"][0]
    assert n == len(tiles) and m["totals"][1] == len(p2t) <= P
    assert [tuple(x) for x in zip(m["tile_expert"][:n], m["tile_row_limit"][:n])] == tiles
    assert (m["tile_expert"][n:] == -1).all() and (m["tile_row_limit"][n:] == -1).all()


def test_invariants_random():
    rng = np.random.default_rng(11)
    E, tile = 32, 32
    ids = inputs.draw_topk(rng, 50, E, 6, "zipf")
    ids[3, 2] = -1
    ids[7] = -1
    m = routing.route_metadata(ids, E, tile)
    counts, off = m["expert_counts"], m["expert_offsets"]
    live = ids.reshape(-1) >= 0
    assert counts.sum() == live.sum()
    assert (off % tile == 0).all() and off[0] == 0 and off[-1] == m["totals"][1]
    e2p = m["expanded_to_permuted"].reshape(-1)
    assert (e2p[~live] == -1).all()
    # bijection between live routes and non-padding rows
    rows = e2p[live]
    assert len(np.unique(rows)) == len(rows)
    p2t = m["permuted_to_token"]
    assert set(np.nonzero(p2t >= 0)[0]) == set(rows)
    assert (p2t[rows] == np.nonzero(live)[0] // 6).all()
    # an expert's rows are increasing in the expanded index
    flat = ids.reshape(-1)
    for e in range(E):
        r = e2p[flat == e]
        assert (np.diff(r) > 0).all()
        if len(r):
            assert r[0] == off[e] and r[-1] == off[e] + counts[e] - 1


def test_all_routes_one_expert_and_single_token():
    ids = np.full((40, 1), 5, dtype=np.int32)
    m = routing.route_metadata(ids, 8, 32)
    assert list(m["expert_counts"]) == [0, 0, 0, 0, 0, 40, 0, 0]
    assert list(m["totals"]) == [2, 64]
    assert list(m["tile_expert"][:2]) == [5, 5] and list(m["tile_row_limit"][:2]) == [40, 40]
    m1 = routing.route_metadata(np.array([[3, 0]], dtype=np.int32), 8, 32)
    assert list(m1["expanded_to_permuted"][0]) == [32, 0]
    assert list(m1["totals"]) == [2, 64]


def test_all_unrouted():
    m = routing.route_metadata(-np.ones((4, 2), dtype=np.int32), 8, 32)
    assert list(m["totals"]) == [0, 0]
    assert (m["expanded_to_permuted"] == -1).all() and (m["permuted_to_token"] == -1).all()


def test_bad_id_refused():
    with pytest.raises(ValueError):
        routing.route_metadata(np.array([[0, 8]], dtype=np.int32), 8, 32)
    with pytest.raises(ValueError):
        routing.route_metadata(np.array([[-2, 1]], dtype=np.int32), 8, 32)


@pytest.mark.parametrize("T,K,E,tile", [(8, 8, 128, 32), (64, 8, 128, 32), (8192, 8, 128, 128), (1, 1, 4, 32)])
def test_padded_bound_holds(T, K, E, tile):
    """max_padded_rows (the flashinfer_ops page's gemm2_rows bound) covers the
    worst case: every expert holding one route beyond a multiple of tile."""
    P = routing.max_padded_rows(T, K, E, tile)
    R = T * K
    F = min(E, R)
    # adversarial: F experts with 1 route, the rest on one expert
    ids = np.zeros(R, dtype=np.int32)
    ids[:F] = np.arange(F)
    m = routing.route_metadata(ids.reshape(T, K), E, tile)
    assert m["totals"][1] <= P
    # exact at the extremes where it is attained
    if R - F == 0:
        assert m["totals"][1] == P
