"""Model check of the tile order of the grouped products (no GPU).

The device builds every CTA's tile sequence from the expert offsets: the groups are split in
two streams (groups of more than 256 rows, and the rest, in the products whose B operand is
an expert weight), the two streams are merged in proportion, and inside a group the tiles run
N-tile major, M-tile minor, a group of more than 16 M tiles (with K of at least 4096) in
panels of 16 M tiles. The functions below restate that arithmetic (the quotient and remainder
merge of the cursor, the panel decode of a tile's index inside its group) and check, over
many random shapes, that the CTAs together visit every (group, M tile, N tile) exactly once
and that a panel's tiles are contiguous in the group's order.
"""
import random

import pytest

HEAVY_ROWS = 256
PANEL = 16


def group_tiles(mt, nt, local, panel, K):
    """(mi, ni) of the tile with index `local` in its group of mt x nt tiles."""
    if panel <= 0 or mt <= panel or K < 4096:
        ni, mi = divmod(local, mt)
        return mi, ni
    p, r0 = divmod(local, panel * nt)
    pm = min(panel, mt - p * panel)
    ni, rem = divmod(r0, pm)
    return p * panel + rem, ni


def cta_tiles(counts, stream_of, first, stride):
    """The merged positions a CTA visits: tile = first, first + stride, ...; position i is
    stream 0's iff floor((i + 1) n0 / tot) > floor(i n0 / tot) (the cursor's test r + n0 >= tot
    on the carried quotient q = floor(i n0 / tot) and remainder r)."""
    n = [sum(c for c, s in zip(counts, stream_of) if s == k) for k in (0, 1)]
    tot = n[0] + n[1]
    out = []
    tile = first
    while tile < tot:
        q, r = divmod(tile * n[0], tot) if tot else (0, 0)
        s0 = r + n[0] >= tot
        j = q if s0 else tile - q
        out.append((0 if s0 else 1, j))
        tile += stride
    return out


@pytest.mark.parametrize("seed", range(40))
def test_every_tile_is_visited_once(seed):
    rng = random.Random(seed)
    E = rng.randint(1, 40)
    rows = [rng.choice([0, 1, 64, 65, 128, 200, 256, 257, 900, 2048, 2100, 4500]) for _ in range(E)]
    nt = rng.randint(1, 12)
    K = rng.choice([2048, 7680])
    bm = 128
    mts = [(r + bm - 1) // bm for r in rows]
    counts = [mt * nt for mt in mts]
    stream_of = [1 if r > HEAVY_ROWS else 0 for r in rows]
    # each stream's groups keep their order: start of group g within its stream
    start = {}
    run = [0, 0]
    for g, (c, s) in enumerate(zip(counts, stream_of)):
        start[g] = (s, run[s])
        run[s] += c
    by_stream = {0: [], 1: []}
    for g in range(E):
        by_stream[stream_of[g]].append(g)
    seen = set()
    ctas = rng.choice([1, 7, 152])
    for cta in range(ctas):
        for s, j in cta_tiles(counts, stream_of, cta, ctas):
            g = next(g for g in by_stream[s] if start[g][1] <= j < start[g][1] + counts[g])
            local = j - start[g][1]
            mi, ni = group_tiles(mts[g], nt, local, PANEL, K)
            assert 0 <= mi < mts[g] and 0 <= ni < nt
            key = (g, mi, ni)
            assert key not in seen
            seen.add(key)
    assert len(seen) == sum(counts)


@pytest.mark.parametrize("mt,nt", [(17, 16), (32, 30), (40, 8), (16, 5), (1, 3), (100, 7)])
def test_panels_are_contiguous_and_n_major_inside(mt, nt):
    order = [group_tiles(mt, nt, i, PANEL, 7680) for i in range(mt * nt)]
    assert sorted(order) == [(m, n) for m in range(mt) for n in range(nt)]
    for p0 in range(0, mt, PANEL):
        pm = min(PANEL, mt - p0)
        block = order[p0 * nt:(p0 + pm) * nt]
        assert {m for m, _ in block} == set(range(p0, p0 + pm))
        # N-tile major: the first pm tiles share N tile 0, the next pm N tile 1, ...
        assert [n for _, n in block] == [n for n in range(nt) for _ in range(pm)]
    # a short K keeps the plain N-major order over the whole group
    plain = [group_tiles(mt, nt, i, PANEL, 2048) for i in range(mt * nt)]
    assert plain == [(m, n) for n in range(nt) for m in range(mt)]
