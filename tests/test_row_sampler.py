"""CPU check of the row sampler the sampled GPU parity checks use: it must hold the first
and last rows of both CTAs of every 256-row pair tile (where the masks of "Chapter 13: The
Blocked Matmul Kernel", section 13.2, act at tile edges) and of every 128-row tile."""
from gpu_util import sample_rows


def test_sample_rows_cover_tile_edges():
    for M in (8192, 16384, 1000, 257):
        rows = set(sample_rows(M, n_random=0))
        for t0 in range(0, M, 128):
            assert {r for r in (t0, t0 + 127) if r < M} <= rows
        assert M - 1 in rows


def test_sample_rows_random_part():
    rows = sample_rows(8192, n_random=256)
    assert len(rows) >= 8192 // 256 * 4 + 100 and rows == sorted(set(rows))
    assert all(0 <= r < 8192 for r in rows)
