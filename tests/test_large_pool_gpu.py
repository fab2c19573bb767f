"""GPU parity with the referenced blocks placed past 2^31 elements (2^32 bytes) of the cache.

A block pool the size a serving engine allocates ("PagedAttention：KV Cache", block
allocation: the pool is sized from the free device memory) holds more rows than a 32-bit
element index reaches. Each case here draws a small workload, copies its pool on the
device to block ids BASE.. of a pool of BASE + nb blocks whose other rows are NaN, shifts
the block tables and slots by BASE, and runs the library on the large pool. The oracle
runs on the small host case: physical block ids do not enter the result, so the outputs
must agree within |o - ref| <= 1e-2 + 1e-2*|ref| and the stored rows bit for bit. Every
row outside the relocated blocks must still be NaN afterwards (nothing written there)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import (DeviceCase, assert_close, bits, from_bits, oracle_after_store,
                               to_f64)

pytestmark = pytest.mark.gpu


def relocate(case):
    """The case on the device, its blocks moved to ids BASE.. of a large NaN pool, BASE
    the smallest multiple of 64 whose first element index is at least 2^31."""
    dc = DeviceCase(case)
    per_block = case.block_size * case.num_kv_heads * case.head_dim
    base = -(-(1 << 31) // per_block)
    base = -(-base // 64) * 64
    assert base * per_block >= 1 << 31 and base * per_block * 2 >= 1 << 32
    nb = case.num_blocks
    shape = (base + nb,) + tuple(case.k_cache.shape[1:])
    for name in ("k_cache", "v_cache"):
        big = torch.full(shape, float("nan"), dtype=case.k_cache.dtype, device=dc.dev)
        big[base:] = getattr(dc, name)
        setattr(dc, name, big)
    bt = dc.bt.clone()
    bt[bt >= 0] += base
    dc.bt = bt
    slots = dc.slots.clone()
    slots[slots >= 0] += base * case.block_size
    dc.slots = slots
    return dc, base


def check_pool(dc, base, ok, ov):
    """The relocated blocks equal the oracle's store; every other row is untouched NaN."""
    for cache, ref in ((dc.k_cache, ok), (dc.v_cache, ov)):
        torch.cuda.synchronize()
        assert bool(torch.isnan(cache[:base]).all()), "a row below the relocated blocks changed"
        assert np.array_equal(bits(cache[base:]), ref)


CASES = [(16, 8, 128), (32, 8, 128), (16, 8, 64)]


@pytest.mark.parametrize("H,Hk,D", CASES)
def test_store_then_decode_past_2_31(H, Hk, D):
    """Store and decode (two launches) on the CUDA-core route (2 query heads per KV head)
    and the tensor-core route (4 per KV head; head_dim 64)."""
    case = workloads.decode_case([1, 257, 2048, 4000, 0, 130], H, Hk, D, 256,
                                 seed=4100 + H + D)
    dc, base = relocate(case)
    dc.store()
    out = dc.decode()
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov = oracle_after_store(case)
    check_pool(dc, base, ok, ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                        case.context_lens)
    assert_close(got, ref, f"decode past 2^31 H={H} Hk={Hk} D={D}")


@pytest.mark.parametrize("H,Hk,D", CASES)
def test_fused_step_past_2_31(H, Hk, D):
    """The fused store + decode step writes the new rows past 2^31 and reads them back."""
    case = workloads.decode_case([3, 256, 1025, 3000, 0], H, Hk, D, 256, seed=4200 + H + D)
    dc, base = relocate(case)
    out = torch.full_like(dc.q, float("nan"))
    pk.pa_decode_step(out, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.slots,
                      dc.bt, dc.ctx, dev_err=dc.err)
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov = oracle_after_store(case)
    check_pool(dc, base, ok, ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                        case.context_lens)
    assert_close(got, ref, f"fused step past 2^31 H={H} Hk={Hk} D={D}")


@pytest.mark.parametrize("D", [128, 64])
def test_store_then_prefill_past_2_31(D):
    """Chunked prefill whose tensor maps address blocks past 2^31 elements."""
    case = workloads.prefill_case([0, 300, 1000], [129, 77, 260], 16, 8, D, 256,
                                  seed=4300 + D)
    dc, base = relocate(case)
    dc.store()
    out = dc.prefill()
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov = oracle_after_store(case)
    check_pool(dc, base, ok, ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.prefill(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                         case.cu_seqlens_q, case.cu_seqlens_k, causal=case.causal)
    assert_close(got, ref, f"prefill past 2^31 D={D}")
