"""Host-side models of two pieces of the kernels' arithmetic on indices,
checked for the properties the kernels rely on (the GPU tests check the
kernels themselves against the oracle):

* the k-slices of a split-K cluster: the slices [r KB / S, (r + 1) KB / S)
  of the S ranks partition a tile's KB k-blocks, none empty when KB >= S;
* the swapped-roles store: lane l of a warp holds column l of C and the
  values of rows 0 .. R-1; within each group of eight lanes a three-step
  butterfly (at distance d = 4, 2, 1 a lane swaps with lane ^ d the four
  values whose index differs from its own lane index in bit d; every step
  over all 8 x 8 blocks) leaves lane (g, j) holding row 8b + j, columns
  8g .. 8g + 7 of block b, which it writes as one 16-byte store.  Every
  element of the tile is then written exactly once, at its own place.
"""
import itertools
import random


def k_slice(r, S, KB):
    return r * KB // S, (r + 1) * KB // S


def test_k_slices_partition_every_tile():
    for S in (2, 4):
        for KB in range(1, 300):
            covered = []
            for r in range(S):
                k0, k1 = k_slice(r, S, KB)
                assert 0 <= k0 <= k1 <= KB
                if KB >= S:
                    assert k1 > k0, (S, KB, r)
                covered.extend(range(k0, k1))
            assert covered == list(range(KB)), (S, KB)


def butterfly(v):
    """v[lane][i]: lane's value for row i (R rows, R % 8 == 0).  Returns
    x[lane][b][k] after the three steps, as the kernel computes it."""
    lanes, R = len(v), len(v[0])
    x = [[[v[l][8 * b + k] for k in range(8)] for b in range(R // 8)] for l in range(lanes)]
    for d in (4, 2, 1):
        new = [[blk[:] for blk in lane] for lane in x]
        for l in range(lanes):
            j = l & 7
            upper = (j & d) != 0
            partner = l ^ d
            pj = partner & 7
            for b in range(R // 8):
                for k0 in range(8):
                    if k0 & d:
                        continue
                    k1 = k0 | d
                    # what the partner sends: its x[k0] if it is the upper lane, else x[k1]
                    sent = x[partner][b][k0] if (pj & d) else x[partner][b][k1]
                    if upper:
                        new[l][b][k0] = sent
                    else:
                        new[l][b][k1] = sent
        x = new
    return x


def test_butterfly_transposes_every_block():
    for R in (8, 16, 32, 64):
        # value encodes (row, column)
        v = [[(i, l) for i in range(R)] for l in range(32)]
        x = butterfly(v)
        for l, b, k in itertools.product(range(32), range(R // 8), range(8)):
            g, j = l >> 3, l & 7
            assert x[l][b][k] == (8 * b + j, 8 * g + k), (R, l, b, k)


def test_store_pattern_writes_each_element_once():
    rng = random.Random(5)
    for _ in range(200):
        R = rng.choice((8, 16, 32, 64))
        n_warp = 32 * rng.randrange(0, 8)     # the warp's first column of C
        m0 = R * rng.randrange(0, 4)          # the block's first row of C
        M = rng.randrange(1, m0 + R + 9)      # rows of C
        N = 8 * rng.randrange(1, (n_warp + 40) // 8 + 1)   # columns of C, a multiple of 8
        v = [[(m0 + i, n_warp + l) for i in range(R)] for l in range(32)]
        x = butterfly(v)
        written = {}
        for l in range(32):
            j = l & 7
            n = n_warp + l - j                # first of the lane group's eight columns
            for b in range(R // 8):
                m = m0 + 8 * b + j
                if m < M and n < N:           # the kernel's store condition
                    for k in range(8):
                        key = (m, n + k)
                        assert key not in written
                        written[key] = x[l][b][k]
        want = {(m, n): (m, n) for m in range(m0, min(M, m0 + R))
                for n in range(n_warp, min(N, n_warp + 32))}
        assert written == want, (R, n_warp, m0, M, N)


def test_half_tiles_of_a_split_pair_cover_the_tile():
    """Rank r of a swapped-roles pair finishes accumulator columns (rows of
    C) [r BN/2, (r+1) BN/2) and receives the other rank's partial of them."""
    for BN in (16, 32, 64):
        H = BN // 2
        own = [list(range(r * H, (r + 1) * H)) for r in (0, 1)]
        sent = [list(range((r ^ 1) * H, ((r ^ 1) + 1) * H)) for r in (0, 1)]
        assert sorted(own[0] + own[1]) == list(range(BN))
        assert sent[0] == own[1] and sent[1] == own[0]
        assert H % 8 == 0          # the store works in blocks of eight rows
