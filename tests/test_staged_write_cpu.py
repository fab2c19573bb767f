"""CPU pins of the staged-write oracle ("Model Runner V2 设计文档", section
"4. StagedWriteTensor"): the page's usage example, a hand-worked overlap, element-by-element
brute force and invalid writes."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "staged_write_example.json")


def test_oracle_reproduces_the_pages_usage_example():
    g = json.load(open(GOLDEN))
    base = np.zeros(g["shape"], dtype=np.int32)
    out = oracle.staged_write_apply(base, [(r, s, v) for r, s, v in g["writes"]])
    expect = np.zeros_like(base)
    for r, c, val in g["expected_nonzero"]:
        expect[r, c] = val
    assert np.array_equal(out, expect)


def test_oracle_later_write_wins_on_overlap():
    """Closed form by hand: row 1 of a 3x6 tensor of 9s; [1,2,3,4] at column 0, then
    [7,8] at column 2, then [5] at column 5."""
    base = np.full((3, 6), 9, dtype=np.int32)
    out = oracle.staged_write_apply(base, [(1, 0, [1, 2, 3, 4]), (1, 2, [7, 8]), (1, 5, [5])])
    assert out[1].tolist() == [1, 2, 7, 8, 9, 5]
    assert (out[[0, 2]] == 9).all()
    # and the reverse order keeps the long write
    out = oracle.staged_write_apply(base, [(1, 2, [7, 8]), (1, 0, [1, 2, 3, 4])])
    assert out[1].tolist() == [1, 2, 3, 4, 9, 9]


@pytest.mark.parametrize("dtype", [np.int32, np.int64, np.float32, np.int16, np.uint8])
def test_oracle_against_element_by_element_brute_force(dtype):
    rng = np.random.default_rng(31)
    for _ in range(20):
        R, C = rng.integers(1, 6), rng.integers(1, 9)
        base = rng.integers(0, 100, size=(R, C)).astype(dtype)
        writes = []
        for _ in range(rng.integers(0, 6)):
            r = int(rng.integers(R))
            s = int(rng.integers(C))
            n = int(rng.integers(0, C - s + 1))
            writes.append((r, s, rng.integers(0, 100, size=n).astype(dtype)))
        ref = base.copy()
        for r, s, v in writes:  # one element at a time, in staging order
            for i, x in enumerate(v):
                ref[r, s + i] = x
        assert np.array_equal(oracle.staged_write_apply(base, writes), ref)


def test_oracle_rejects_a_write_outside_the_tensor():
    with pytest.raises(ValueError):
        oracle.staged_write_apply(np.zeros((2, 4), np.int32), [(0, 3, [1, 2])])
    with pytest.raises(ValueError):
        oracle.staged_write_apply(np.zeros((2, 4), np.int32), [(2, 0, [1])])
