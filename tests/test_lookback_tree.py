"""The 32-ary look-back tree of the single-pass scans, replayed on the CPU with
the kernels' index arithmetic: tile j publishes its sum as node (0, j); a tile
whose index ends in 31 at level L also publishes the sum of its 32-node group
as node (L + 1, j >> 5(L+1)); the carry into tile j is, for every level L
below `levels`, the sum of the siblings m - d .. m - 1 of its level-L ancestor
m = j >> 5L, d = m mod 32.  Node (L, m) lives at word off_L + m, off_0 = 0,
off_{L+1} = off_L + count_L, count_{L+1} = count_L >> 5.  For any tile count
the carry must be the sum of every tile before j, and no node may be read
before it is written or land outside 2 * tiles words."""
import pytest

MAX_LEVELS = 4


def levels_of(tiles):
    levels = 1
    while levels < MAX_LEVELS and ((tiles - 1) >> (5 * levels)) != 0:
        levels += 1
    return levels


def replay(tiles, publish_top):
    """Publish in ticket order and check each tile's carry; publish_top: the
    forms that also publish parents at level `levels` (harmless extra words)."""
    levels = levels_of(tiles)
    words = {}
    value = [(7 * j) % 13 + 1 for j in range(tiles)]
    prefix = 0
    for j in range(tiles):
        # look-back of tile j: every node it reads was published before
        carry, off, count = 0, 0, tiles
        for L in range(levels):
            m = j >> (5 * L)
            d = m & 31
            for s in range(m - d, m):
                assert (off + s) in words, (tiles, j, L, s)
                carry += words[off + s]
            off += count
            count >>= 5
        assert carry == prefix, (tiles, j)
        prefix += value[j]
        # publish tile j and every parent it completes
        words[j] = value[j]
        own, off, count, m = value[j], 0, tiles, j
        L = 0
        while (L + 1 < levels or (publish_top and L < levels)) and (m & 31) == 31:
            own = sum(words[off + s] for s in range(m - 31, m + 1))
            nxt = off + count
            assert nxt + (m >> 5) < 2 * tiles
            words[nxt + (m >> 5)] = own
            off, count, m, L = nxt, count >> 5, m >> 5, L + 1


@pytest.mark.parametrize("tiles", [1, 2, 31, 32, 33, 63, 64, 1023, 1024, 1025, 1056, 32767, 32768, 32769, 40000])
@pytest.mark.parametrize("publish_top", [False, True])
def test_lookback_carries_are_prefix_sums(tiles, publish_top):
    replay(tiles, publish_top)


def test_levels_cover_the_tiles():
    for tiles in (1, 32, 33, 1024, 1025, 32768, 32769, 1 << 20):
        L = levels_of(tiles)
        assert 32 ** L >= tiles or L == MAX_LEVELS
