"""Host logic of the ZeRO-2 streaming driver that needs no GPU: how a flat
model is cut into buckets."""

import pytest

from zero_gradient_reduce_gb300 import streaming


@pytest.mark.parametrize("n,B", [(1, 1), (10, 4), (12, 4), (123_578_112, 13_107_200),
                                 (6_574_178_304, 134_217_728), (5, 100)])
def test_buckets_tile_the_model_in_order(n, B):
    bounds = streaming.bucket_bounds(n, B)
    assert bounds[0][0] == 0 and bounds[-1][1] == n
    assert all(a[1] == b[0] for a, b in zip(bounds, bounds[1:]))
    assert all(0 < hi - lo <= B for lo, hi in bounds)
    assert all(hi - lo == B for lo, hi in bounds[:-1])
    assert len(bounds) == -(-n // B)


@pytest.mark.parametrize("n,B", [(0, 4), (4, 0), (-1, 3)])
def test_bucket_sizes_must_be_positive(n, B):
    with pytest.raises(ValueError):
        streaming.bucket_bounds(n, B)
