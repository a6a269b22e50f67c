"""The fp64 oracle against its pins (no GPU)."""
import math

import numpy as np
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_block_partial_rejects_empty_and_mismatched():
    # The worked example raises on an empty or length-mismatched block, and the merge
    # raises when there is no block at all.
    with pytest.raises(ValueError):
        oracle.block_partial([], [])
    with pytest.raises(ValueError):
        oracle.block_partial([0.0, 1.0], [1.0])
    with pytest.raises(ValueError):
        oracle.merge_blocks([])


def test_merge_weights_in_unit_interval():
    w = oracle.merge_weights([120.0, 0.0, -5.0, 119.0])
    assert abs(math.fsum(w) - 1.0) < 1e-15
    assert all(0.0 <= x <= 1.0 for x in w)


def test_split_ranges():
    assert oracle.split_ranges(3, 2) == [(0, 2), (2, 3)]
    assert [b - a for a, b in oracle.split_ranges(257, 4)] == [65, 65, 65, 62]
    # Splits at or beyond the sequence length are empty.
    assert oracle.split_ranges(5, 4, capacity=16) == [(0, 4), (4, 5), (8, 8), (12, 12)]


def test_rejects_bad_arguments(lib):
    q = np.zeros((1, 3, 4), np.float32)
    k = np.zeros((1, 2, 4, 4), np.float32)
    with pytest.raises(ValueError):          # Hq not a multiple of Hkv
        oracle.decode(q, k, k, np.array([4], np.int32), lib=lib)
    q = np.zeros((1, 2, 4), np.float32)
    with pytest.raises(ValueError):          # seq_len beyond capacity
        oracle.decode(q, k, k, np.array([5], np.int32), lib=lib)
    with pytest.raises(ValueError):          # block-table id outside the pool
        oracle.decode(q, k, k, np.array([3], np.int32),
                      block_table=np.array([[7]], np.int32), page_size=4, lib=lib)


def test_rows_subset_matches_full(lib):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 4, 8)).astype(np.float32)
    k = rng.standard_normal((2, 2, 9, 8)).astype(np.float32)
    v = rng.standard_normal((2, 2, 9, 8)).astype(np.float32)
    lens = np.array([9, 4], np.int32)
    o, l = oracle.decode(q, k, v, lens, lib=lib)
    o2, l2 = oracle.decode(q, k, v, lens, rows=[5, 0], lib=lib)
    assert np.array_equal(o2[1, 1], o[1, 1]) and np.array_equal(o2[0, 0], o[0, 0])
    assert np.isnan(o2[0, 1]).all() and np.isnan(l2[1, 0])
