"""Plain readings of the two scheduling rules the pages state.  Test
infrastructure only (see the package docstring).

``storage_align_strides`` follows the stride loop quoted in the leiblog.wang
post answering what ``storage_align(factor, offset)`` does (Technical index,
the Zhihu-answer post on shared-memory bank conflicts): walk the dimensions
from innermost to outermost with a running stride that starts at 1; where a
dimension carries an alignment, raise the stride to the next value congruent
to ``offset`` modulo ``factor``; that is the dimension's stride; then multiply
the running stride by the dimension's extent.

``streamk_units`` is the reading of the Stream-K post on the same index
(reproducing "Stream-K: Work-centric Parallel Decomposition for Dense
Matrix-Matrix Multiplication on the GPU"): the k-axis work of all output tiles
is laid end to end as one iteration space and cut into equal contiguous
ranges, one per CTA, so that no SM is left without work when the tile count
is small.  The page gives no further detail; the reading taken is: range r of
G covers iterations floor(r*W/G) .. floor((r+1)*W/G)-1 of the W iterations;
a range is cut where it crosses a tile boundary; tiles ahead of the split
region (``dp_tiles``) are handed out whole, tile c + u*G to CTA c.
"""
from __future__ import annotations


def storage_align_strides(shape, aligns):
    """Strides (in elements, outermost first) of a buffer of ``shape`` whose
    dimension d carries ``aligns[d] = (factor, offset)`` or None."""
    stride = 1
    rstrides = []
    for dim in range(len(shape) - 1, -1, -1):
        al = aligns[dim] if dim < len(aligns) else None
        if al is not None and al[0] != 0:
            factor, offset = al
            stride = stride + (factor + offset - stride % factor) % factor
        rstrides.append(stride)
        stride = stride * shape[dim]
    return list(reversed(rstrides))


def streamk_ranges(total_iters: int, ctas: int):
    """[begin, end) of each CTA's share of ``total_iters`` MAC iterations."""
    return [(r * total_iters // ctas, (r + 1) * total_iters // ctas)
            for r in range(ctas)]


def cluster_split_units(tiles: int, iters_per_tile: int, split: int):
    """Plain k-split of every tile into `split` equal contiguous ranges, one
    per CTA of the tile's cluster: CTA c owns tile c // split and k-blocks
    floor(r*I/split) .. floor((r+1)*I/split)-1, r = c % split."""
    out = []
    for c in range(tiles * split):
        t, r = divmod(c, split)
        out.append([(t, r * iters_per_tile // split, (r + 1) * iters_per_tile // split)])
    return out


def streamk_units(dp_tiles: int, sk_tiles: int, iters_per_tile: int, ctas: int):
    """Work units of every CTA, in the order each CTA processes them.

    Returns a list (one per CTA) of lists of (tile, k_begin, k_end): first the
    whole tiles of the data-parallel region (tile c, c+G, ... < dp_tiles), then
    the pieces of the CTA's equal share of the split region, whose tiles are
    numbered dp_tiles .. dp_tiles+sk_tiles-1.
    """
    out = []
    total = sk_tiles * iters_per_tile
    ranges = streamk_ranges(total, ctas) if total > 0 else [(0, 0)] * ctas
    for c in range(ctas):
        units = []
        t = c
        while t < dp_tiles:
            units.append((t, 0, iters_per_tile))
            t += ctas
        x, end = ranges[c]
        while x < end:
            tile = x // iters_per_tile
            k0 = x % iters_per_tile
            k1 = min(iters_per_tile, k0 + (end - x))
            units.append((dp_tiles + tile, k0, k1))
            x += k1 - k0
        out.append(units)
    return out
