"""CPU tests of the library's native host staging (pa_staged_pack: merge + pack) that
feeds pa_staged_write_apply ("Model Runner V2 设计文档", section "4. StagedWriteTensor"),
checked against the oracle. No GPU: the packing is host code."""
import numpy as np

import oracle
from paged_kv_cache_107_gb300 import staged


def test_merged_runs_do_not_overlap_and_have_the_same_effect():
    """The host merge turns any staging sequence into disjoint runs; applying those runs in
    any order gives what the oracle gives for the staged sequence."""
    rng = np.random.default_rng(32)
    for trial in range(200):
        R, C = int(rng.integers(1, 5)), int(rng.integers(1, 40))
        base = rng.integers(-50, 50, size=(R, C)).astype(np.int32)
        writes = []
        for _ in range(int(rng.integers(0, 12))):
            r = int(rng.integers(R))
            s = int(rng.integers(C))
            n = int(rng.integers(0, C - s + 1))
            writes.append((r, s, rng.integers(-99, 99, size=n).astype(np.int32)))
        rows = [w[0] for w in writes]
        starts = [w[1] for w in writes]
        lens = [len(w[2]) for w in writes]
        vals = np.concatenate([w[2] for w in writes]) if writes else np.zeros(0, np.int32)
        buf, lay = staged.pack(rows, starts, lens, vals, 4)
        runs = staged.unpack(buf, lay, np.int32)
        cover = {}
        for r, s, v in runs:
            assert len(v) > 0
            for c in range(s, s + len(v)):
                assert (r, c) not in cover, "merged runs overlap"
                cover[(r, c)] = True
        order = rng.permutation(len(runs)) if runs else []
        got = oracle.staged_write_apply(base, [runs[i] for i in order])
        assert np.array_equal(got, oracle.staged_write_apply(base, writes)), trial


def test_pack_layout():
    """Two disjoint writes stay two runs, sorted by row; offsets and values as packed."""
    buf, lay = staged.pack([2, 0], [3, 1], [3, 3], np.array([3, 1, 2, -1, -2, -5], np.int32), 4)
    W = lay.num_writes
    assert W == 2 and lay.num_values == 6 and lay.values_offset % 16 == 0
    assert buf[:8].view(np.int32).tolist() == [0, 2]
    assert buf[8:16].view(np.int32).tolist() == [1, 3]
    assert buf[16:28].view(np.int32).tolist() == [0, 3, 6]
    assert buf[lay.values_offset:].view(np.int32).tolist() == [-1, -2, -5, 3, 1, 2]


def test_pack_joins_touching_and_overlapping_writes():
    buf, lay = staged.pack([1, 1, 1], [0, 4, 2], [4, 2, 3],
                           np.array([1, 2, 3, 4, 5, 6, 7, 8, 9], np.int64), 8)
    runs = staged.unpack(buf, lay, np.int64)
    assert len(runs) == 1
    r, s0, v = runs[0]
    assert (r, s0) == (1, 0) and v.tolist() == [1, 2, 7, 8, 9, 6]


def test_pack_rejects_negative_lengths_and_reports_size():
    import pytest
    import paged_kv_cache_107_gb300 as pk
    with pytest.raises(pk.PagedAttentionError):
        staged.pack([0], [0], [-1], np.zeros(0, np.int32), 4)
    with pytest.raises(pk.PagedAttentionError, match="28 bytes needed"):
        pk.pa_staged_pack([0], [0], [3], np.array([1, 2, 3], np.int32), 4, np.zeros(8, np.uint8))
