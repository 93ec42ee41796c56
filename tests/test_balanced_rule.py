"""The balanced split's partition rule (MLA_DECODE_UNIFORM_SEGMENTS's default in
the C header), as restated for the parity tests and for the benchmark's byte
accounting: both restatements agree, and the rule has the properties the
kernel relies on -- every unit's tiles covered once, in order, by at most S
parts, and chunks that differ by at most one tile."""
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
def test_chunks_differ_by_at_most_one_tile(seed):
    for tiles, S, grid in _cases(300, seed):
        T = sum(tiles)
        if T == 0:
            continue
        need = max(-(-max(tiles) // (S - 1)), 1)
        n = min(grid, max(T // need, 1))
        sizes = [(c + 1) * T // n - c * T // n for c in range(n)]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= need
        # the parts of all units, chunk by chunk, add up to the chunk sizes
        per_chunk = [0] * n
        start = 0
        bounds = [c * T // n for c in range(n + 1)]
        for u, t in enumerate(tiles):
            for a, b in balanced_parts(tiles, S, grid)[u]:
                c = next(c for c in range(n) if bounds[c] <= start + a < bounds[c + 1])
                per_chunk[c] += b - a
            start += t
        assert per_chunk == sizes


def test_benchmark_accounting_uses_the_same_rule():
    for tiles, S, grid in _cases(200, 5):
        ref = balanced_parts(tiles, S, grid)
        got = bench._balanced_parts(tiles, S, grid)
        assert [ref[u] for u in range(len(tiles))] == got
