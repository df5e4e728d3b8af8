"""Pins of the oracle's in-place cache refresh, CPU only: against numpy fancy indexing of the
state before the step (positions < len) with the rest of every row kept, on parent patterns
that make in-place writing hazardous (swaps, cycles, one parent for all, identity)."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("pattern", [[0, 0, 0, 0], [1, 0, 3, 2], [1, 2, 3, 0], [3, 3, 1, 1], [0, 1, 2, 3],
                                     [2, 2, 2, 0]])
def test_inplace_equals_the_gather_of_the_old_state(pattern):
    g = np.random.default_rng(sum(pattern))
    layers, batch, k, heads, max_len, head_dim, length = 2, 3, 4, 2, 6, 5, 4
    cache = g.standard_normal((layers, batch * k, heads, max_len, head_dim)).astype(np.float16)
    parent = np.array([pattern, pattern[::-1], [0, 1, 2, 3]], np.int32)
    new = oracle.cache_refresh_inplace(cache, parent, length)
    src_rows = (np.arange(batch)[:, None] * k + parent).reshape(-1)
    want = cache.copy()
    want[:, :, :, :length] = cache[:, src_rows, :, :length]
    assert np.array_equal(new.view(np.int16), want.view(np.int16))


def test_inplace_matches_out_of_place_on_the_copied_positions():
    g = np.random.default_rng(7)
    shape = (3, 8, 2, 5, 4)
    cache = g.standard_normal(shape).astype(np.float16)
    parent = g.integers(0, 4, (2, 4)).astype(np.int32)
    new = oracle.cache_refresh_inplace(cache, parent, 5)
    out = oracle.cache_reorder(cache, parent, 5)
    assert np.array_equal(new.view(np.int16), out.view(np.int16))


def test_bad_parent_is_rejected():
    cache = np.zeros((1, 2, 1, 2, 2), np.float16)
    with pytest.raises(ValueError):
        oracle.cache_refresh_inplace(cache, np.array([[0, 2]], np.int32), 1)
