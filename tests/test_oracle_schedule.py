"""Pins for the oracle's schedule readings (storage_align, Stream-K split)."""
import pytest

from oracle import schedule


def test_storage_align_worked_values():
    # Values worked by hand from the stride loop printed in the leiblog.wang
    # storage_align answer (Technical index): stride starts at 1, innermost
    # first; an aligned dim gets stride += (factor + offset - stride % factor) % factor.
    # fp16 [128][32] with (32, 8) on dim 0: 32 + (32+8-0)%32 = 40.
    assert schedule.storage_align_strides([128, 32], [(32, 8), None]) == [40, 1]
    # fp32 [8][128] with (32, 4) on dim 0: 128 + 4 = 132.
    assert schedule.storage_align_strides([8, 128], [(32, 4), None]) == [132, 1]
    # already congruent: 40 + (32+8-8)%32 = 40.
    assert schedule.storage_align_strides([4, 40], [(32, 8), None]) == [40, 1]
    # 3-D, align on the middle dim: 5 + (4+1-1)%4 = 5; outer = 5*3 = 15.
    assert schedule.storage_align_strides([2, 3, 5], [None, (4, 1), None]) == [15, 5, 1]
    # no alignment: plain packed strides.
    assert schedule.storage_align_strides([7, 3, 5], [None, None, None]) == [15, 5, 1]


@pytest.mark.parametrize("shape,factor,offset", [
    ([128, 32], 32, 8), ([64, 77], 16, 3), ([8, 128], 32, 4), ([3, 1], 8, 7)])
def test_storage_align_invariants(shape, factor, offset):
    inner = shape[1]
    s = schedule.storage_align_strides(shape, [(factor, offset), None])[0]
    assert s % factor == offset % factor          # congruence the knob asks for
    assert inner <= s < inner + factor            # smallest such stride >= extent


@pytest.mark.parametrize("W,G", [(128, 128), (2048, 152), (100, 7), (7, 7), (1, 1), (6400, 152)])
def test_streamk_ranges_cover_exactly_once(W, G):
    ranges = schedule.streamk_ranges(W, G)
    assert ranges[0][0] == 0 and ranges[-1][1] == W
    for (b0, e0), (b1, _) in zip(ranges, ranges[1:]):
        assert e0 == b1
    sizes = [e - b for b, e in ranges]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("dp,sk,I,G", [(0, 16, 8, 128), (0, 32, 64, 152),
                                       (304, 224, 128, 152), (2048, 0, 128, 152),
                                       (0, 5, 3, 4), (10, 3, 7, 4)])
def test_streamk_units_partition_every_iteration(dp, sk, I, G):
    units = schedule.streamk_units(dp, sk, I, G)
    seen = {}
    for c, lst in enumerate(units):
        for tile, k0, k1 in lst:
            assert 0 <= k0 < k1 <= I
            for k in range(k0, k1):
                assert (tile, k) not in seen
                seen[(tile, k)] = c
            if tile < dp:
                assert (k0, k1) == (0, I) and tile % G == c
    assert len(seen) == (dp + sk) * I


@pytest.mark.parametrize("T,I,s", [(32, 64, 4), (16, 8, 4), (1, 256, 8), (5, 3, 2), (7, 17, 8)])
def test_cluster_split_partitions_every_iteration(T, I, s):
    units = schedule.cluster_split_units(T, I, s)
    assert len(units) == T * s
    seen = set()
    for c, lst in enumerate(units):
        (tile, k0, k1), = lst
        assert tile == c // s and 0 <= k0 <= k1 <= I
        seen.update((tile, k) for k in range(k0, k1))
    assert len(seen) == T * I
