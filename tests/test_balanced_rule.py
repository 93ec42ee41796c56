"""The balanced split's partition rule (MLA_DECODE_UNIFORM_SEGMENTS's default in
the C header), as restated for the parity tests and for the benchmark's byte
accounting: both restatements agree, and the rule has the properties the
kernel relies on -- every unit's tiles covered once, in order, by at most S
parts, and chunks whose positions (tiles plus one overhead position per unit
with tiles) differ by at most one."""
import numpy as np
import pytest

import bench
from parity import balanced_parts


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        u = int(rng.integers(1, 60))
        kind = rng.integers(0, 4, u)
        tiles = np.where(kind == 0, 0, np.where(kind == 1, rng.integers(1, 6, u), rng.integers(1, 400, u)))
        yield [int(t) for t in tiles], int(rng.integers(2, 24)), int(rng.integers(1, 200))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rule_covers_every_tile_once_within_s_parts(seed):
    for tiles, S, grid in _cases(300, seed):
        parts = balanced_parts(tiles, S, grid)
        for u, t in enumerate(tiles):
            pl = parts[u]
            assert len(pl) <= S
            if t == 0:
                assert pl == []
                continue
            assert pl[0][0] == 0 and pl[-1][1] == t
            assert all(a < b for a, b in pl)
            assert all(pl[k][1] == pl[k + 1][0] for k in range(len(pl) - 1))


@pytest.mark.parametrize("seed", [3, 4])
def test_chunks_differ_by_at_most_one_position(seed):
    for tiles, S, grid in _cases(300, seed):
        V = sum(t + 1 for t in tiles if t > 0)
        if V == 0:
            continue
        need = max(-(-max(tiles) // (S - 1)), 1)
        n = min(grid, max(V // need, 1))
        sizes = [(c + 1) * V // n - c * V // n for c in range(n)]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= need
        # tiles of every unit's parts plus the overhead positions, chunk by
        # chunk, add up to the chunk sizes
        per_chunk = [0] * n
        bounds = [c * V // n for c in range(n + 1)]
        chunk = lambda x: next(c for c in range(n) if bounds[c] <= x < bounds[c + 1])
        parts = balanced_parts(tiles, S, grid)
        pos = 0
        for u, t in enumerate(tiles):
            if t == 0:
                continue
            per_chunk[chunk(pos)] += 1  # the overhead position
            start = pos + 1
            for a, b in parts[u]:
                per_chunk[chunk(start + a)] += b - a
            pos = start + t
        assert per_chunk == sizes


def test_a_chunk_crossing_a_unit_start_holds_one_tile_less():
    # 4 units of 10 tiles on 4 chunks: 44 positions, 11 each; chunk 0 takes
    # unit 0 whole (overhead + 10 tiles), every chunk one unit
    assert balanced_parts([10, 10, 10, 10], 4, 4) == {u: [(0, 10)] for u in range(4)}
    # 2 units of 20 tiles on 3 chunks: 42 positions, 14 each; unit 0 (positions
    # 1..20) is cut 13 + 7, unit 1 (22..41) 6 + 14: the middle chunk holds
    # unit 1's overhead position and 13 tiles (7 + 6)
    assert balanced_parts([20, 20], 4, 3) == {0: [(0, 13), (13, 20)], 1: [(0, 6), (6, 20)]}


def test_benchmark_accounting_uses_the_same_rule():
    for tiles, S, grid in _cases(200, 5):
        ref = balanced_parts(tiles, S, grid)
        got = bench._balanced_parts(tiles, S, grid)
        assert [ref[u] for u in range(len(tiles))] == got
