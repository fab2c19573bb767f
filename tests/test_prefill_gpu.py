"""GPU parity of pa_prefill_varlen (tcgen05 path) against the fp64 oracle.

Each case stores the new tokens first (pa_store_kvcache), then runs the prefill, and
compares with the oracle applied after its own store. Tolerance: |o - ref| <= 1e-2 +
1e-2*|ref| (bf16 operands, fp32 accumulation, P rounded to bf16 for the second product)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import (DeviceCase, assert_close, from_bits, oracle_after_store, to_f64)

pytestmark = pytest.mark.gpu


def run_prefill(case, rows=None):
    dc = DeviceCase(case)
    dc.store()
    out = dc.prefill()
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov = oracle_after_store(case)
    dt = case.k_cache.dtype
    got = to_f64(out)
    if rows is None:
        ref = oracle.prefill(case.q, from_bits(ok, dt), from_bits(ov, dt), case.block_tables,
                             case.cu_seqlens_q, case.cu_seqlens_k, causal=case.causal)
        assert np.all(np.isfinite(got))
        assert_close(got, ref, case.name)
    else:
        ref = oracle.prefill(case.q, from_bits(ok, dt), from_bits(ov, dt), case.block_tables,
                             case.cu_seqlens_q, case.cu_seqlens_k, causal=case.causal, rows=rows)
        flat = got.reshape(-1, case.head_dim)[rows]
        assert np.all(np.isfinite(flat))
        assert_close(flat, ref, case.name)
    return dc, out


@pytest.mark.parametrize("cached,new", [
    ([0], [1]), ([0], [5]), ([0], [64]), ([0], [128]), ([0], [129]), ([1], [1]),
    ([255], [1]), ([256], [1]), ([300], [200]), ([0, 17, 256, 1000], [70, 300, 1, 257])])
def test_small_causal(cached, new):
    """No cache, a cache ending mid-block or on a block edge, n = 1 (decode shape),
    several tiles and ragged tails."""
    run_prefill(workloads.prefill_case(cached, new, 16, 8, 128, 256,
                                       seed=800 + sum(cached) + 3 * sum(new)))


@pytest.mark.parametrize("H,Hk", [(8, 8), (16, 8), (32, 8), (64, 8), (4, 1), (16, 16)])
def test_group_sizes(H, Hk):
    """GQA groups of 1, 2, 4 and 8 query heads packed into the 128-row tile."""
    run_prefill(workloads.prefill_case([40, 0, 300], [100, 33, 130], H, Hk, 128, 256,
                                       seed=900 + H + Hk))


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 512])
def test_block_sizes(bs):
    """Boxes of one block (block_size >= 128) or several blocks per 128-key tile."""
    run_prefill(workloads.prefill_case([0, 150, 700], [200, 77, 129], 16, 8, 128, bs,
                                       seed=1000 + bs))


def test_non_causal():
    run_prefill(workloads.prefill_case([0, 37, 256], [50, 91, 300], 16, 8, 128, 256,
                                       seed=1100, causal=False))


def test_single_token_prefill_equals_decode():
    """A prefill of one new token after c cached ones is the decode of that token."""
    case = workloads.prefill_case([0, 99, 256, 511], [1, 1, 1, 1], 16, 8, 128, 256, seed=1200)
    dc, out = run_prefill(case)
    dec = torch.empty_like(dc.q)
    ctx = torch.from_numpy(np.diff(case.cu_seqlens_k).astype(np.int32)).cuda()
    pk.pa_decode(dec, dc.q, dc.k_cache, dc.v_cache, dc.bt, ctx)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_f64(out), to_f64(dec), atol=2e-2, rtol=2e-2)


def test_q_rows_after_an_offset():
    """cu_seqlens_q starting past row 0: the first rows of q and out belong to no sequence.
    The later tiles lie past the host's bound on the batch's rows (num_seqs x max_seqlen_q),
    so their Q rows are copied row by row while the earlier ones come by whole TMA boxes;
    rows outside the sequences are never written."""
    import dataclasses
    base = workloads.prefill_case([0, 130, 700], [200, 77, 129], 16, 8, 128, 256, seed=1250)
    off = 300
    rng = np.random.default_rng(1251)
    lead = torch.from_numpy(rng.standard_normal((off,) + tuple(base.q.shape[1:])).astype(
        np.float32)).to(base.q.dtype)
    case = dataclasses.replace(base, q=torch.cat([lead, base.q]),
                               cu_seqlens_q=(base.cu_seqlens_q + off).astype(np.int32))
    dc = DeviceCase(case)
    dc.store()
    out = dc.prefill()
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    # the oracle takes rows from 0: the same sequences without the leading rows
    ok, ov = oracle_after_store(base)
    ref = oracle.prefill(base.q, from_bits(ok), from_bits(ov), base.block_tables,
                         base.cu_seqlens_q, base.cu_seqlens_k, causal=True)
    got = to_f64(out)
    assert np.all(np.isnan(got[:off])), "rows before the first sequence were written"
    assert np.all(np.isfinite(got[off:]))
    assert_close(got[off:], ref, "q rows after an offset")


def test_prefill_deterministic():
    case = workloads.prefill_case([100, 0], [300, 257], 16, 8, 128, 256, seed=1300)
    dc = DeviceCase(case)
    dc.store()
    a = dc.prefill()
    b = dc.prefill()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_full_chunked_prefill_workload_sampled():
    """Workload 5: 32 sequences, cached U{0..2048}, new U{100..1024}, causal. Every row of
    four sequences plus 2000 random rows are compared with the oracle."""
    case = workloads.workload(5)
    H = case.num_heads
    rng = np.random.default_rng(5)
    total = int(case.cu_seqlens_q[-1])
    rows = set(rng.choice(total * H, 2000, replace=False).tolist())
    for s in (0, 7, 19, 31):
        for t in range(int(case.cu_seqlens_q[s]), int(case.cu_seqlens_q[s + 1])):
            for h in (0, H - 1):
                rows.add(t * H + h)
    run_prefill(case, rows=np.array(sorted(rows), np.int64))


def _sampled_rows(case, n_random, seed, whole=()):
    H = case.num_heads
    rng = np.random.default_rng(seed)
    total = int(case.cu_seqlens_q[-1])
    rows = set(rng.choice(total * H, min(n_random, total * H), replace=False).tolist())
    for s in whole:
        for t in range(int(case.cu_seqlens_q[s]), int(case.cu_seqlens_q[s + 1])):
            for h in range(H):
                rows.add(t * H + h)
    return np.array(sorted(rows), np.int64)


def test_schedule_one_unit_per_cta_beyond_sort_limit():
    """1,100 sequences (more than the in-kernel sort takes): the launcher runs one unit per
    CTA on a (KV head, sequence, pair) grid. Every row is compared."""
    rng = np.random.default_rng(1400)
    cached = rng.integers(0, 41, 1100)
    new = rng.integers(1, 4, 1100)
    run_prefill(workloads.prefill_case(cached, new, 16, 8, 128, 16, seed=1401))


def test_schedule_one_unit_per_cta_head_dim_64_fp16():
    """The same grid at head_dim 64 with IEEE fp16 elements (P in its own tensor-memory
    columns, the next S product issued once the softmax has read the last): every row."""
    rng = np.random.default_rng(1410)
    cached = rng.integers(0, 41, 1100)
    new = rng.integers(1, 4, 1100)
    run_prefill(workloads.prefill_case(cached, new, 16, 8, 64, 16, seed=1411,
                                       dtype=torch.float16))


def test_schedule_persistent_with_many_units_per_cta():
    """8 query heads per KV head (16 positions per tile), 64 sequences of 512 new tokens:
    8,192 units, about 54 per CTA on the persistent grid; sampled rows plus two whole
    sequences."""
    rng = np.random.default_rng(1500)
    cached = rng.integers(0, 301, 64)
    case = workloads.prefill_case(cached, [512] * 64, 64, 8, 128, 256, seed=1501)
    run_prefill(case, rows=_sampled_rows(case, 4000, 1502, whole=(0, 63)))


def test_schedule_one_unit_per_cta_beyond_pair_limit():
    """8 query heads per KV head and up to 900 new tokens over 80 sequences: more possible
    (sequence, pair) entries than the in-kernel sort takes, so one unit per CTA; sampled
    rows plus the longest sequence whole."""
    rng = np.random.default_rng(1600)
    cached = rng.integers(0, 200, 80)
    new = rng.integers(1, 901, 80)
    new[5] = 900
    case = workloads.prefill_case(cached, new, 64, 8, 128, 256, seed=1601)
    run_prefill(case, rows=_sampled_rows(case, 3000, 1602, whole=(5,)))
