"""Host-only checks of the persistent tile schedule (data-parallel rounds plus the
split-K share of the last rounds): every (tile, K-block) unit is computed exactly once,
every partial sum is added by exactly one owner, owners gather exactly the workers that
cover the rest of their tile, and shares are balanced."""
import itertools

import pytest

import dense_tiled_gemm_05_gb300 as g
from dense_tiled_gemm_05_gb300 import build as gbuild

FULL, PARTIAL, OWNER = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def built():
    gbuild.build()


def check(tiles, kb, slots, stream_k=True):
    sched = g.schedule(tiles, kb, slots, stream_k)
    covered = {}
    whole_total = sum(w for w, _ in sched)
    # round-robin whole tiles: slot s gets s, s + slots, ...
    for s, (whole, _) in enumerate(sched):
        for i in range(whole):
            t = s + i * slots
            for k in range(kb):
                assert (t, k) not in covered
                covered[(t, k)] = s
    partial_of = {}
    owners = {}
    work = []
    for s, (whole, segs) in enumerate(sched):
        units = 0
        for i, (t, b, e, role, f, l) in enumerate(segs):
            assert 0 <= b < e <= kb and whole_total <= t < tiles
            units += e - b
            for k in range(b, e):
                assert (t, k) not in covered, (t, k)
                covered[(t, k)] = s
            if i > 0:  # walked backwards: each piece ends where the previous one began
                assert (t, e) == (segs[i - 1][0], kb) or (t == segs[i - 1][0] - 1 and e == kb)
            if role == PARTIAL:
                assert e < kb and i == 0, "only a share's first piece lacks its tile's end"
                partial_of[s] = t
            elif role == OWNER:
                assert b > 0 and e == kb and i == len(segs) - 1
                owners[t] = (s, f, l, b)
            else:
                assert b == 0 and e == kb and f == l == -1
        work.append(units + whole * kb)
    assert len(covered) == tiles * kb
    # every partial is gathered by the owner of its tile, in increasing worker order, and an
    # owner only waits for workers numbered below it
    gathered = set()
    for t, (s, f, l, b) in owners.items():
        assert l == s - 1 and f <= l
        for src in range(f, l + 1):
            assert partial_of.get(src) == t
            gathered.add(src)
        # the sources cover exactly the start of the tile
        assert all(covered[(t, k)] in range(f, l + 1) for k in range(0, b))
    assert gathered == set(partial_of)
    if stream_k and tiles % slots and tiles * kb >= slots:
        assert max(work) - min(work) <= kb + 1  # the split share is balanced to a unit
    return sched


@pytest.mark.parametrize("tiles,kb,slots", [(256, 64, 76), (64, 128, 76), (1024, 128, 76),
                                            (5, 3, 2), (7, 1, 3), (3, 10, 8), (1, 5, 4),
                                            (152, 17, 76), (2, 2, 76)])
def test_schedule_covers_every_unit_once(tiles, kb, slots):
    check(tiles, kb, slots, True)
    check(tiles, kb, slots, False)


def test_schedule_exhaustive_small():
    for tiles, kb, slots in itertools.product(range(1, 13), range(1, 7), range(1, 9)):
        check(tiles, kb, slots, True)


def test_headline_shapes():
    # bf16 4096^3 on 76 clusters: 2 whole rounds, then 104 tiles shared as K-blocks.
    sched = check(256, 64, 76)
    assert all(w == 2 for w, _ in sched)
    # 8192^3: 12 whole rounds, the last 112 tiles shared.
    assert all(w == 12 for w, _ in check(1024, 128, 76))
    # skinny 16384 x 128: 64 tiles on 76 workers, all shared.
    assert all(w == 0 for w, _ in check(64, 128, 76))
    # tiles that fill whole rounds need no split.
    assert all(not segs for _, segs in check(152, 64, 76))
    assert g.lib().gemm_schedule_segments(4, 0, 2, 1, 0, None, None, 0) == -1


def test_idle_split_pieces_per_tile():
    # Few tiles with long K-loops are split over as many clusters as the planner gives
    # them (about sqrt(K-blocks / 4) pieces a tile): every unit once, and no owner gathers
    # more than that many partials less one.
    import torch

    def t(shape, layout="row"):
        if layout == "row":
            return torch.empty(shape, dtype=torch.bfloat16)
        return torch.empty(shape[::-1], dtype=torch.bfloat16).t()

    for M, N, K, cap in [(256, 256, 8192, 6), (1024, 128, 8192, 6), (128, 128, 32768, 11),
                         (128, 128, 65536, 16)]:
        p = g.plan(t((M, K)), t((K, N), "col"), sm_count=152)
        tiles, kb, slots = p["grid_m"] * p["grid_n"], p["k_iters"], p["ctas"] // 2
        assert p["split_tiles"] == tiles and slots == min(76, cap * tiles), (M, N, K, p)
        sched = check(tiles, kb, slots, True)
        for whole, segs in sched:
            assert whole == 0
            for (_, _, _, role, f, l) in segs:
                if role == OWNER:
                    assert l - f + 1 <= cap - 1
