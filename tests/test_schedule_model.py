"""Host-side model of the kernel's work partition (whole tiles round robin,
then the stream-K tail cut into equal k-block ranges), checked for the
properties the kernel relies on: every k-block of every tile is computed by
exactly one unit, the per-tile contributor count and first contributor agree
with the ranges, and a unit needs at most two workspace slots."""
import random


def bound(u, iters, sk_units):
    return u * iters // sk_units


def unit_of(it, iters, sk_units):
    return ((it + 1) * sk_units - 1) // iters


def work(unit, units, T, KB, dp_tiles, sk_units):
    out = []
    t = unit
    while t < dp_tiles:
        out.append((t, 0, KB, -1, 1, unit))
        t += units
    iters = (T - dp_tiles) * KB
    if sk_units and unit < sk_units:
        x, x_end = bound(unit, iters, sk_units), bound(unit + 1, iters, sk_units)
        while x < x_end:
            tt = x // KB
            t0, t1 = tt * KB, tt * KB + KB
            e = min(x_end, t1)
            first = unit_of(t0, iters, sk_units)
            splits = unit_of(t1 - 1, iters, sk_units) - first + 1
            out.append((dp_tiles + tt, x - t0, e - t0, tt, splits, first))
            x = e
    return out


def schedule(T, KB, U):
    sk_tiles = (T % U if T % U else U) if T >= U else T
    dp = T - sk_tiles
    usk = min(U, sk_tiles * KB // 16)
    if usk > 4 * sk_tiles:
        usk = 4 * sk_tiles
    return (U if dp > 0 else usk), dp, usk


def test_partition_properties():
    rng = random.Random(0)
    cases = [(1024, 128, 76), (256, 64, 76), (240, 65, 76), (4, 8, 76), (6, 6, 76),
             (2048, 128, 152), (7, 1, 76), (77, 3, 76), (152, 64, 76)]
    cases += [(rng.randint(1, 600), rng.randint(1, 200), rng.randint(2, 160)) for _ in range(300)]
    for T, KB, U in cases:
        units, dp, usk = schedule(T, KB, U)
        if usk < 2:
            continue
        assert dp % U == 0
        cover = {}
        slots = {}
        for u in range(units):
            for (tile, kb0, kb1, sk_tile, splits, first) in work(u, units, T, KB, dp, usk):
                assert 0 <= kb0 < kb1 <= KB
                for kb in range(kb0, kb1):
                    assert (tile, kb) not in cover
                    cover[(tile, kb)] = u
                if sk_tile >= 0:
                    assert first <= u < first + splits
                    if splits == 1:
                        assert (kb0, kb1) == (0, KB)   # a tile of its own: no workspace
                    else:
                        # only the first and last tiles of a range are shared
                        slot = 0 if bound(u, (T - dp) * KB, usk) // KB == sk_tile else 1
                        assert (u, slot) not in slots
                        slots[(u, slot)] = sk_tile
        assert len(cover) == T * KB, (T, KB, U)
        # contributor counts per tail tile match the ranges
        for tt in range(T - dp):
            owners = {cover[(dp + tt, kb)] for kb in range(KB)}
            iters = (T - dp) * KB
            first = unit_of(tt * KB, iters, usk)
            last = unit_of(tt * KB + KB - 1, iters, usk)
            assert owners == set(range(first, last + 1))


def test_whole_pieces_of_few_tall_tiles():
    """Fewer tiles than units (the swapped-roles kernels on C with few rows):
    every tile is cut into the same whole number of k-pieces, T * floor(U / T)
    units with at least 16 k-blocks each.  Then each unit holds exactly one
    piece of one tile, each tile has exactly `pieces` contributors, and the
    pieces of a tile are consecutive units."""
    rng = random.Random(1)
    cases = [(64, 128, 152), (128, 256, 152), (96, 128, 152), (32, 64, 152), (64, 33, 152)]
    cases += [(rng.randint(1, 151), rng.randint(16, 400), 152) for _ in range(300)]
    for T, KB, U in cases:
        pieces = min(U // T, KB // 16)
        if pieces < 2:
            continue
        usk = T * pieces
        iters = T * KB
        seen = {}
        for u in range(usk):
            items = work(u, usk, T, KB, 0, usk)
            assert len(items) == 1, (T, KB, U, u, items)
            tile, kb0, kb1, sk_tile, splits, first = items[0]
            assert splits == pieces and first == (u // pieces) * pieces
            assert kb1 - kb0 >= 16
            seen.setdefault(tile, []).append((kb0, kb1))
        assert sorted(seen) == list(range(T))
        for tile, ranges in seen.items():
            ranges.sort()
            assert ranges[0][0] == 0 and ranges[-1][1] == KB
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
