"""GPU parity of pa_store_kvcache against the oracle's store: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import DeviceCase, bits, oracle_after_store

pytestmark = pytest.mark.gpu


def _check_store(case):
    dc = DeviceCase(case)
    dc.store()
    assert dc.dev_err() == 0
    ok, ov = oracle_after_store(case)
    assert np.array_equal(bits(dc.k_cache), ok)
    assert np.array_equal(bits(dc.v_cache), ov)


def test_store_tiny_with_padding_slot():
    """Four tokens, slot_mapping[1] = -1: that token writes nothing."""
    case = workloads.workload(1)
    assert case.slot_mapping[1] == -1
    _check_store(case)


@pytest.mark.parametrize("bs", [16, 256])
def test_store_decode_batch(bs):
    _check_store(workloads.decode_case(list(range(1, 300, 7)), 16, 8, 128, bs, seed=300 + bs))


def test_store_prefill_batch_all_new_tokens():
    case = workloads.prefill_case([0, 100, 256, 1000], [300, 1, 255, 513], 16, 8, 128, 256,
                                  seed=310)
    _check_store(case)


def test_store_unaligned_token_stride_takes_scalar_path():
    """A token stride that is not a multiple of 8 elements goes through the 2-byte path
    and must give the same bytes."""
    case = workloads.decode_case([5, 9, 33], 8, 4, 128, 16, seed=311)
    dev = torch.device("cuda")
    n, hk, d = case.k_new.shape
    padded_k = torch.zeros((n, hk * d + 3), dtype=torch.bfloat16, device=dev)
    padded_v = torch.zeros((n, hk * d + 3), dtype=torch.bfloat16, device=dev)
    padded_k[:, : hk * d] = case.k_new.reshape(n, -1).to(dev)
    padded_v[:, : hk * d] = case.v_new.reshape(n, -1).to(dev)
    k = torch.as_strided(padded_k, (n, hk, d), (hk * d + 3, d, 1))
    v = torch.as_strided(padded_v, (n, hk, d), (hk * d + 3, d, 1))
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    slots = torch.from_numpy(case.slot_mapping).to(dev)
    pk.pa_store_kvcache(k, v, kc, vc, slots)
    torch.cuda.synchronize()
    ok, ov = oracle_after_store(case)
    assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)


def test_store_out_of_range_slot_is_skipped_and_flagged():
    case = workloads.decode_case([4, 4], 8, 8, 128, 16, seed=312)
    case.slot_mapping[1] = case.num_blocks * case.block_size + 7  # beyond the cache
    dc = DeviceCase(case)
    before_k = bits(dc.k_cache).copy()
    dc.store()
    assert dc.dev_err() & pk.PA_DEV_ERR["slot"]
    after_k = bits(dc.k_cache)
    # token 0 landed, token 1 wrote nothing
    flat_b = before_k.reshape(-1, 8 * 128)
    flat_a = after_k.reshape(-1, 8 * 128)
    s0 = int(case.slot_mapping[0])
    assert np.array_equal(flat_a[s0], bits(case.k_new)[0].reshape(-1))
    mask = np.ones(flat_a.shape[0], bool)
    mask[s0] = False
    assert np.array_equal(flat_a[mask], flat_b[mask])


def test_store_zero_tokens_is_a_no_op():
    dev = torch.device("cuda")
    kc = torch.zeros((2, 16, 8, 128), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device=dev)
    pk.pa_store_kvcache(k, k, kc, kc, torch.zeros(0, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()


@pytest.mark.slow
def test_store_full_size_decode_step():
    """Qwen3-0.6B-shaped decode step: 256 new tokens into a 4096-block pool."""
    case = workloads.workload(2)
    dc = DeviceCase(case)
    dc.store()
    assert dc.dev_err() == 0
    ok, ov = oracle_after_store(case)
    # compare only the rows the store may touch plus a sample of the rest
    row = case.num_kv_heads * case.head_dim
    fk = bits(dc.k_cache).reshape(-1, row)
    fv = bits(dc.v_cache).reshape(-1, row)
    ok2, ov2 = ok.reshape(-1, row), ov.reshape(-1, row)
    slots = case.slot_mapping[case.slot_mapping >= 0]
    assert np.array_equal(fk[slots], ok2[slots]) and np.array_equal(fv[slots], ov2[slots])
    rng = np.random.default_rng(0)
    sample = rng.choice(fk.shape[0], 4096, replace=False)
    assert np.array_equal(fk[sample], ok2[sample]) and np.array_equal(fv[sample], ov2[sample])


def test_store_full_chunked_prefill_workload_byte_for_byte():
    """Every one of the chunked-prefill workload's 17,556 new tokens (32 sequences,
    cached U{0..2048}, new U{100..1024}, block size 256, the 4096-block pool) stored in one
    launch, then both whole caches compared byte for byte with the oracle's store.

    The store's grid holds one resident wave of warps (6 blocks of 8 warps per SM), one
    warp per K or V row; 35,112 rows are several per warp, so this is the size that takes
    the kernel's grid-stride loop ("3.6 ModelRunner…", section 2: prepare_prefill builds
    one slot per new token)."""
    case = workloads.workload(5)
    n_tok = int(case.cu_seqlens_q[-1])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 2 * n_tok > sms * 6 * 8, "the case must need more rows than the grid has warps"
    assert np.all(case.slot_mapping >= 0)
    _check_store(case)
