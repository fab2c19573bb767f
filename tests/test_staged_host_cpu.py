"""CPU tests of the host staging (merge + pack) that feeds pa_staged_write_apply
("Model Runner V2 设计文档", section "4. StagedWriteTensor"), checked against the oracle."""
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
        runs = staged.merge_runs(writes)
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
    runs = [(2, 3, np.array([3, 1, 2], np.int32)), (0, 1, np.array([-1, -2, -5], np.int32))]
    buf, lay = staged.pack_runs(runs, 4)
    meta = buf[:4 * 7].view(np.int32)
    assert meta[:2].tolist() == [2, 0]
    assert meta[2:4].tolist() == [3, 1]
    assert meta[4:7].tolist() == [0, 3, 6]
    assert lay["values"] % 16 == 0 and lay["num_values"] == 6 and lay["num_writes"] == 2
    assert buf[lay["values"]:].view(np.int32).tolist() == [3, 1, 2, -1, -2, -5]
