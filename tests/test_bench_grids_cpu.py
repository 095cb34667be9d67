"""The measurement grids behind the backward's choices (bench.py --variant-table,
--split-table, --key-split-table): their sizes as quoted in the documentation and
the property each grid is meant to cover."""

import bench


def test_variant_grid():
    pts = bench.variant_grid()
    assert len(pts) == 306
    assert {d for d, _, _, _ in pts} == {64, 96, 128}
    assert all(bh * n * n <= 1 << 32 for _, _, bh, n in pts)
    assert len(set(pts)) == len(pts)


def test_split_grid_has_few_key_tiles():
    pts = bench.split_grid()
    assert len(pts) == 64
    for bh, n, d, causal, variant in pts:
        assert variant == (5 if d <= 128 else 7)
        # fewer 128-key tiles than two waves of 152 SMs: the regime the query split serves
        assert bh * (n // 128) < 304


def test_key_split_grid_has_few_query_tiles():
    pts = bench.key_split_grid()
    assert len(pts) == 130
    assert {d for _, _, d, _ in pts} == {64, 128, 192, 256, 384}
    for bh, n, d, causal in pts:
        items = (n // 128) * (2 if d == 384 else 1) * bh  # the dQ kernel's work items
        assert items < 304
        assert not (d == 384 and n == 16384)
