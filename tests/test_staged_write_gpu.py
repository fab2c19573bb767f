"""GPU parity of pa_staged_write_apply and StagedWriteTensor against the oracle, bit for
bit ("Model Runner V2 设计文档", section "4. StagedWriteTensor")."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300.staged import StagedWriteTensor

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "staged_write_example.json")


def test_pages_usage_example():
    g = json.load(open(GOLDEN))
    t = StagedWriteTensor(tuple(g["shape"]), dtype=torch.int32)
    for r, s, v in g["writes"]:
        t.stage_write(r, s, v)
    t.apply_write()
    torch.cuda.synchronize()
    assert int(t.dev_err.item()) == 0
    expect = np.zeros(g["shape"], np.int32)
    for r, c, val in g["expected_nonzero"]:
        expect[r, c] = val
    assert np.array_equal(t.gpu.cpu().numpy(), expect)


def test_block_table_update_rounds():
    """A [1024, 1000] int32 table (block ids, -1 padded); each round stages the decode
    step's appends (one new block id for some sequences), a few prefill runs of several
    ids, and overlapping rewrites; rounds follow each other without synchronisation."""
    rng = np.random.default_rng(107400)
    R, C = 1024, 1000
    init = np.full((R, C), -1, np.int32)
    lens = rng.integers(0, 200, size=R)
    for r in range(R):
        init[r, :lens[r]] = rng.integers(0, 1 << 20, size=lens[r])
    t = StagedWriteTensor((R, C), dtype=torch.int32, init=torch.from_numpy(init))
    ref = init.copy()
    for rnd in range(6):
        writes = []
        for r in rng.choice(R, size=256, replace=False):  # decode appends
            if lens[r] < C:
                writes.append((int(r), int(lens[r]), [int(rng.integers(1 << 20))]))
                lens[r] += 1
        for r in rng.choice(R, size=8, replace=False):  # prefill: several new blocks
            n = int(min(C - lens[r], rng.integers(1, 40)))
            if n > 0:
                writes.append((int(r), int(lens[r]), rng.integers(1 << 20, size=n).tolist()))
                lens[r] += n
        for _ in range(4):  # rewrites that overlap earlier writes of this round
            r, s, v = writes[int(rng.integers(len(writes)))]
            writes.append((r, max(0, s - 1), rng.integers(1 << 20, size=len(v) + 1).tolist()))
        for w in writes:
            t.stage_write(*w)
        t.apply_write()
        ref = oracle.staged_write_apply(ref, writes)
    torch.cuda.synchronize()
    assert int(t.dev_err.item()) == 0
    assert np.array_equal(t.gpu.cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", [torch.uint8, torch.int16, torch.int32, torch.float32,
                                   torch.int64])
def test_element_sizes_and_strided_rows(dtype):
    """1-, 2-, 4- and 8-byte elements; the tensor is a column slice of a wider one (row
    stride > columns): columns past the slice stay untouched."""
    rng = np.random.default_rng(int(torch.finfo(dtype).bits if dtype.is_floating_point
                                    else torch.iinfo(dtype).bits))
    R, C, P = 37, 50, 64
    wide = torch.from_numpy(rng.integers(0, 100, size=(R, P)).astype(np.int64)).to(dtype).cuda()
    before = wide.cpu().numpy().copy()
    base = wide[:, :C]
    writes = []
    used = set()
    for _ in range(30):
        r = int(rng.integers(R))
        s = int(rng.integers(C))
        n = int(rng.integers(1, C - s + 1))
        if any((r, c) in used for c in range(s, s + n)):
            continue
        used.update((r, c) for c in range(s, s + n))
        writes.append((r, s, rng.integers(0, 100, size=n)))
    rows = torch.tensor([w[0] for w in writes], dtype=torch.int32, device="cuda")
    starts = torch.tensor([w[1] for w in writes], dtype=torch.int32, device="cuda")
    offs = np.zeros(len(writes) + 1, np.int32)
    offs[1:] = np.cumsum([len(w[2]) for w in writes])
    vals = torch.from_numpy(np.concatenate([w[2] for w in writes]).astype(np.int64)).to(dtype).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pa_staged_write_apply(base, rows, starts, torch.from_numpy(offs).cuda(), vals, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = wide.cpu().numpy()
    ref_slice = oracle.staged_write_apply(before[:, :C], [(r, s, v.astype(before.dtype))
                                                          for r, s, v in writes])
    assert np.array_equal(got[:, :C].view(np.uint8), ref_slice.view(np.uint8))
    assert np.array_equal(got[:, C:].view(np.uint8), before[:, C:].view(np.uint8))


def test_bad_runs_are_flagged_and_skipped():
    """A run past the last column, a row out of range, and decreasing offsets: flagged
    with PA_DEV_ERR_STAGED; only the good runs are written."""
    base = torch.zeros((4, 8), dtype=torch.int32, device="cuda")
    rows = torch.tensor([0, 1, 9, 2], dtype=torch.int32, device="cuda")
    starts = torch.tensor([0, 6, 0, 1], dtype=torch.int32, device="cuda")
    offs = torch.tensor([0, 2, 5, 6, 8], dtype=torch.int32, device="cuda")
    vals = torch.arange(1, 9, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.pa_staged_write_apply(base, rows, starts, offs, vals, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pk.PA_DEV_ERR["staged"]
    expect = np.zeros((4, 8), np.int32)
    expect[0, 0:2] = [1, 2]
    expect[2, 1:3] = [7, 8]
    assert np.array_equal(base.cpu().numpy(), expect)
    # decreasing offsets: nothing out of bounds, flagged
    err.zero_()
    offs_bad = torch.tensor([0, 5, 2, 6, 8], dtype=torch.int32, device="cuda")
    pk.pa_staged_write_apply(base, rows, starts, offs_bad, vals, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pk.PA_DEV_ERR["staged"]


def test_long_runs():
    """Whole-row rewrites of a [512, 4096] int32 tensor: 2M values in 512 runs."""
    rng = np.random.default_rng(107401)
    R, C = 512, 4096
    t = StagedWriteTensor((R, C), dtype=torch.int32)
    writes = [(r, 0, rng.integers(-(1 << 30), 1 << 30, size=C)) for r in range(R)]
    for w in writes:
        t.stage_write(*w)
    t.apply_write()
    torch.cuda.synchronize()
    assert np.array_equal(t.gpu.cpu().numpy(),
                          oracle.staged_write_apply(np.zeros((R, C), np.int32), writes))


@pytest.mark.parametrize("W", [8191, 8192, 20000])
def test_run_counts_around_the_shared_memory_limit(W):
    """Up to 8191 runs the offsets (W+1 entries) sit in shared memory; from 8192 runs
    the search reads them from global memory: both paths give the oracle's result."""
    rng = np.random.default_rng(W)
    R, C = 4096, 64
    t = StagedWriteTensor((R, C), dtype=torch.int32)
    flat = rng.choice(R * C, size=W, replace=False)
    rows, cols = (flat // C).astype(np.int32), (flat % C).astype(np.int32)
    vals = rng.integers(-(1 << 31), 1 << 31, size=W).astype(np.int32)
    t.stage_writes(rows, cols, vals)
    t.apply_write()
    torch.cuda.synchronize()
    assert int(t.dev_err.item()) == 0
    ref = oracle.staged_write_apply(np.zeros((R, C), np.int32),
                                    [(int(r), int(c), [int(v)]) for r, c, v in zip(rows, cols, vals)])
    assert np.array_equal(t.gpu.cpu().numpy(), ref)
