"""Host model of the one-launch expert GEMMs' schedule (no GPU).

The kernel deals units round-robin over a grid of G resident CTAs, each CTA
taking its units in order: the n1 = tiles * tw1 GEMM1 units (route tile
u // tw1) first, then the tiles * tw2 GEMM2 units (route tile (u - n1) // tw2).
A GEMM2 unit may start only once every GEMM1 unit of its route tile has
finished (the per-tile completion counter). This model runs that schedule in
discrete steps, one unit per CTA per step, and checks that it always
completes: a waited-for GEMM1 unit is earlier in its own CTA's order than any
GEMM2 unit, so no CTA can wait on a unit that waits on it."""
import pytest


def run_schedule(tiles: int, tw1: int, tw2: int, G: int, work1: int = 20, work2: int = 8) -> int:
    """Simulated steps until every unit is done; raises on a stall."""
    n1, n2 = tiles * tw1, tiles * tw2
    n = n1 + n2
    G = min(G, n)
    queues = [list(range(c, n, G)) for c in range(G)]
    left = [0] * G  # remaining work of the CTA's current unit
    pos = [0] * G
    done1 = [0] * tiles  # finished GEMM1 units per route tile
    finished = 0
    steps = 0
    while finished < n:
        progressed = False
        completed = []  # GEMM1 units finished in this step: visible from the next
        for c in range(G):
            if pos[c] >= len(queues[c]):
                continue
            u = queues[c][pos[c]]
            if left[c] == 0:  # not started: may it start?
                if u >= n1 and done1[(u - n1) // tw2] < tw1:
                    continue  # waiting on the tile's counter
                left[c] = work1 if u < n1 else work2
            left[c] -= 1
            progressed = True
            if left[c] == 0:
                if u < n1:
                    completed.append(u // tw1)
                pos[c] += 1
                finished += 1
        for tau in completed:
            done1[tau] += 1
        steps += 1
        if not progressed:
            raise RuntimeError(f"stalled with {n - finished} units left")
    return steps


@pytest.mark.parametrize("tiles,tw1,tw2,G", [
    (1, 2, 2, 456),        # one route tile: GEMM2 units wait on GEMM1 units running alongside
    (53, 32, 40, 456),     # decode b=8 (tile_m = 32)
    (96, 32, 40, 456),     # decode b=64 Zipf
    (64, 32, 40, 304),     # 64-row tiles, two CTAs per SM
    (575, 32, 40, 304),    # prefill-sized
    (7, 3, 5, 2),          # few CTAs, many units each
    (3, 1, 1, 1),          # a single CTA
])
def test_schedule_completes(tiles, tw1, tw2, G):
    steps = run_schedule(tiles, tw1, tw2, G)
    n1, n2 = tiles * tw1, tiles * tw2
    # never slower than the busiest CTA doing all of its units back to back
    # plus one GEMM1 unit of waiting per GEMM2 unit of the CTA at most
    g = min(G, n1 + n2)
    per_cta = max(
        sum(20 if u < n1 else 8 for u in range(c, n1 + n2, g)) for c in range(g)
    )
    assert steps <= per_cta + 20 * (n2 // g + 1)


def test_a_grid_larger_than_the_units_is_trimmed():
    assert run_schedule(2, 2, 2, 1000) > 0


def test_waiting_really_happens_with_one_tile():
    """With one route tile and more CTAs than units, every GEMM2 unit waits
    for GEMM1 units running on other CTAs: the run takes at least one GEMM1
    unit plus one GEMM2 unit."""
    assert run_schedule(1, 4, 4, 8) >= 20 + 8
