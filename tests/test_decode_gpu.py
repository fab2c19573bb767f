"""GPU parity of pa_decode against the fp64 oracle, element by element.

Every case runs the step in the order the engine does (store of the new token, then
decode over context_lens that include it) and compares with the oracle applied after its
own store. Tolerance: |o - ref| <= 1e-2 + 1e-2*|ref| (bf16 inputs, fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import (DeviceCase, assert_close, bits, from_bits, oracle_after_store,
                               to_f64)

pytestmark = pytest.mark.gpu


def run_case(case, grid_ctas=0, pairs=None, check_store=True):
    dc = DeviceCase(case)
    dc.store()
    out = dc.decode(grid_ctas=grid_ctas)
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov = oracle_after_store(case)
    if check_store:
        assert np.array_equal(bits(dc.k_cache), ok) and np.array_equal(bits(dc.v_cache), ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got)), "non-finite output (a poisoned row was read)"
    if pairs is None:
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens)
        assert_close(got, ref, case.name)
    else:
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens, pairs=pairs)
        assert_close(got.reshape(-1, case.head_dim)[pairs], ref, case.name)
    return dc, out


def test_tiny_workload():
    """B=4, context {1,17,256,300}, H=16, Hk=8, bs=256, permuted physical ids, store of 4
    tokens with one slot = -1."""
    run_case(workloads.workload(1))


@pytest.mark.parametrize("grid", [0, 1, 2, 5, 37, 600])
def test_tiny_any_split_count(grid):
    """The split of the key stream over CTAs does not change the result (beyond fp32
    rounding): one CTA, a few, one tile per CTA."""
    run_case(workloads.workload(1), grid_ctas=grid)


@pytest.mark.parametrize("lens,bs", [
    ([1], 256), ([1], 16), ([15, 16, 17], 16), ([255, 256, 257], 256), ([0, 3, 0], 16),
    ([0], 256), ([31, 1, 64, 100, 2], 32), ([513, 7], 8)])
def test_context_edges(lens, bs):
    """context 1, bs-1, bs, bs+1, empty rows (CUDA-graph padding), tiny blocks."""
    case = workloads.decode_case(lens, 16, 8, 128, bs, seed=400 + sum(lens) + bs)
    run_case(case)


@pytest.mark.parametrize("H,Hk", [(8, 8), (16, 8), (32, 8), (64, 8), (16, 16), (32, 16),
                                  (8, 4), (16, 4), (4, 2), (8, 2), (2, 1), (8, 1), (24, 8),
                                  (40, 8), (48, 8), (56, 8), (12, 4), (5, 1), (14, 2), (32, 2)])
def test_head_layouts(H, Hk):
    """GQA group sizes 1..8 (1 and 2 on CUDA cores when one slab holds every KV head, all
    other layouts on the tensor-core path; 16 is rejected) and KV head slabs of 8, 4, 2, 1
    heads (the slab path with several warps per KV head merges their softmax states)."""
    case = workloads.decode_case([1, 40, 300, 129], H, Hk, 128, 16, seed=500 + H * 7 + Hk)
    if not 1 <= (H // Hk) <= 8:
        with pytest.raises(pk.PagedAttentionError):
            run_case(case)
        return
    for grid in (0, 3):
        run_case(case, grid_ctas=grid)


def test_empty_rows_are_zero():
    case = workloads.decode_case([0, 10, 0, 0, 33], 16, 8, 128, 16, seed=600)
    dc, out = run_case(case)
    o = to_f64(out)
    assert np.all(o[[0, 2, 3]] == 0.0)


@pytest.mark.parametrize("H,Hk,D", [(16, 8, 128), (64, 8, 128), (28, 4, 128), (32, 16, 128),
                                    (16, 8, 64)])
@pytest.mark.parametrize("grid", [0, 7])
def test_run_to_run_bitwise_deterministic(H, Hk, D, grid):
    """The split combine uses the arrival counters only to pick the CTA that combines, in
    CTA order, so repeated launches give the same bits (both decode kernels)."""
    case = workloads.decode_case(list(np.random.default_rng(7).integers(1, 3000, 64)), H, Hk,
                                 D, 256, seed=601, num_blocks=1024)
    dc = DeviceCase(case)
    dc.store()
    a = dc.decode(grid_ctas=grid)
    b = dc.decode(grid_ctas=grid)
    c = dc.decode(grid_ctas=grid)
    torch.cuda.synchronize()
    assert dc.dev_err() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_split_counts_agree_closely():
    """One CTA (no split) vs auto vs many CTAs: the only difference is fp32 rounding in
    the combine, far below bf16 resolution."""
    case = workloads.decode_case(list(np.random.default_rng(8).integers(1, 5000, 20)), 32, 8,
                                 128, 256, seed=602, num_blocks=512)
    dc = DeviceCase(case)
    dc.store()
    outs = [to_f64(dc.decode(grid_ctas=g)) for g in (1, 0, 300, 601)]
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2 * 2.0 ** -8 * (np.abs(outs[0]).max() + 1e-3)


def _ordered_bf16(t):
    """bf16 bit patterns as integers in the order of the values they encode (+0 and -0
    both map to 0), so that adjacent representable values differ by one."""
    b = bits(t).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


SPLIT_GRIDS = (1, 0, 300, 601)  # one CTA (no split), automatic, many CTAs


def _split_outputs(H, Hk, D, seed):
    lens = list(np.random.default_rng(seed).integers(1, 6000, 24)) + [1, 256, 257]
    case = workloads.decode_case(lens, H, Hk, D, 256, seed=seed, num_blocks=1024)
    dc = DeviceCase(case)
    dc.store()
    outs = [dc.decode(grid_ctas=g) for g in SPLIT_GRIDS]
    assert dc.dev_err() == 0
    return case, outs


@pytest.mark.parametrize("H,Hk", [(16, 8), (8, 8), (4, 2)])
def test_split_counts_round_to_adjacent_bf16(H, Hk):
    """CUDA-core kernel (1 or 2 query heads per KV head, probabilities kept in fp32): the
    split-softmax identity is exact, so the split count only changes fp32 rounding (about
    1e-6 relative), far below one bf16 step (2^-8 relative). The bf16 outputs of one CTA,
    the automatic grid and many CTAs are therefore, element by element, the same value or
    adjacent representable values. Near zero the bf16 step is finer than that rounding, so
    two values closer than 1e-5 of their row's largest magnitude also pass."""
    case, outs = _split_outputs(H, Hk, 128, 607 + H + Hk)
    base = _ordered_bf16(outs[0])
    ref = to_f64(outs[0])
    row_max = np.abs(ref).max(axis=-1, keepdims=True)
    for g, o in zip(SPLIT_GRIDS[1:], outs[1:]):
        steps = np.abs(_ordered_bf16(o) - base)
        tiny = np.abs(to_f64(o) - ref) <= 1e-5 * row_max
        bad = (steps > 1) & ~tiny
        assert not bad.any(), (f"grid {g}: {int(bad.sum())} elements more than one bf16 step "
                               f"from the one-CTA result; worst {int(steps.max())}")


def _bf16_step(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    _, e = np.frexp(np.maximum(np.abs(x), 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


@pytest.mark.parametrize("H,Hk,D", [(32, 8, 128), (64, 8, 128), (16, 8, 64)])
def test_split_counts_tensor_core_within_p_rounding(H, Hk, D):
    """Tensor-core kernel: each probability p_t = 2^(s_t - m) is rounded to bf16 (relative
    error <= 2^-9) before the P V product, and the offset m is the running maximum of the
    keys seen so far, which depends on where the splits fall. Two split counts therefore
    differ by at most 2 * 2^-9 * (sum_t p_t |v_t|) / (sum_t p_t) per element, plus one bf16
    step of output rounding and fp32 rounding. The weighted mean of |v| comes from the
    oracle run on |V|."""
    case, outs = _split_outputs(H, Hk, D, 611 + H + D)
    ok, ov = oracle_after_store(case)
    abs_v = from_bits(ov).abs()
    mean_abs_v = oracle.decode(case.q, from_bits(ok), abs_v, case.block_tables,
                               case.context_lens)
    ref = to_f64(outs[0])
    row_max = np.abs(ref).max(axis=-1, keepdims=True)
    for g, o in zip(SPLIT_GRIDS[1:], outs[1:]):
        got = to_f64(o)
        bound = (2.0 ** -8 * mean_abs_v + _bf16_step(np.maximum(np.abs(got), np.abs(ref)))
                 + 1e-5 * row_max)
        diff = np.abs(got - ref)
        bad = diff > bound
        assert not bad.any(), (f"grid {g}: {int(bad.sum())} elements beyond the rounding bound; "
                               f"worst ratio {float((diff / bound).max()):.3f}")
        # the bound is a worst case; the typical difference sits far below it
        assert float(np.median(diff / bound)) < 0.25


def test_sharp_softmax_cases():
    """Near one-hot attention (one key aligned with q, scaled up) and constant values:
    cases where the output is far from the near-uniform average of N(0,1) data."""
    case = workloads.decode_case([50, 700, 1], 8, 4, 128, 16, seed=603)
    q = case.q.float()
    # make key 17 of sequence 1 equal to 3*q/|q| for every KV head's first query head
    b, t = 1, 17
    blk = int(case.block_tables[b, t // 16])
    for j in range(4):
        qv = q[b, 2 * j]
        case.k_cache[blk, t % 16, j] = (4.0 * qv / qv.norm() * np.sqrt(128) / 2).to(torch.bfloat16)
    # sequence 0: constant values per KV head (from the cache rows and the new token)
    for tt in range(49):
        blk0 = int(case.block_tables[0, tt // 16])
        for j in range(4):
            case.v_cache[blk0, tt % 16, j] = float(j + 1)
    for j in range(4):
        case.v_new[0, j] = float(j + 1)
    dc, out = run_case(case)
    o = to_f64(out)
    for h in range(8):
        np.testing.assert_allclose(o[0, h], np.full(128, h // 2 + 1.0), atol=1e-2)


def test_zero_query_gives_mean_of_values():
    case = workloads.decode_case([77, 300], 16, 8, 128, 32, seed=604)
    case.q.zero_()
    run_case(case)


def test_bad_block_id_is_flagged_not_read():
    """A corrupt block-table entry inside the context is never dereferenced: the device
    sets PA_DEV_ERR_BLOCK_ID and the kernel skips the copy."""
    case = workloads.decode_case([40, 40], 8, 8, 128, 16, seed=605)
    case.block_tables[1, 1] = case.num_blocks + 1000
    dc = DeviceCase(case)
    dc.decode()
    assert dc.dev_err() & pk.PA_DEV_ERR["block_id"]


def test_context_beyond_table_is_flagged_and_zeroed():
    case = workloads.decode_case([20, 20], 8, 8, 128, 16, seed=606, max_blocks=2)
    case.context_lens[1] = 2 * 16 + 5  # longer than the table can map
    dc = DeviceCase(case)
    out = dc.decode()
    assert dc.dev_err() & pk.PA_DEV_ERR["context"]
    assert np.all(to_f64(out)[1] == 0.0)


def test_host_validation_launches_nothing():
    dev = torch.device("cuda")
    q = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((4, 16, 8, 128), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((2, 1), dtype=torch.int32, device=dev)
    ctx = torch.ones(2, dtype=torch.int32, device=dev)
    out = torch.zeros_like(q)
    small = pk.DecodeWorkspace(2, 16, 8)
    small.nbytes = 16
    with pytest.raises(pk.PagedAttentionError, match="WORKSPACE"):
        pk.pa_decode(out, q, kc, kc, bt, ctx, workspace=small)
    with pytest.raises(pk.PagedAttentionError, match="SHAPE"):
        pk.pa_decode(out, q, kc, kc, bt, ctx, grid_ctas=100000)
    q96 = torch.zeros((2, 16, 96), dtype=torch.bfloat16, device=dev)
    kc96 = torch.zeros((4, 16, 8, 96), dtype=torch.bfloat16, device=dev)
    ws = pk.DecodeWorkspace(2, 16, 8)
    with pytest.raises(pk.PagedAttentionError, match="UNSUPPORTED"):  # head_dim 96
        pk.pa_decode(torch.zeros_like(q96), q96, kc96, kc96, bt, ctx, workspace=ws)


@pytest.mark.parametrize("num", [2, 3])
def test_full_size_workload(num):
    """Workload 2 (B=256, context U{100..2048}, pool 4096) and workload 3 (B=8, context
    U{32768..131072}, H=32): the whole output against the oracle."""
    case = workloads.workload(num)
    run_case(case, check_store=False)


@pytest.mark.parametrize("bs", [16, 256])
def test_full_size_prefix_sharing(bs):
    """Workload 4: B=512, lognormal lengths, groups of 64 sequences share their first 4
    physical blocks."""
    case = workloads.workload(4, block_size=bs)
    assert case.shared_blocks > 0
    run_case(case, check_store=False)


def test_workspace_reused_across_batch_sizes():
    """One workspace sized for 512 sequences serves calls with 4, 300, 64 and 512
    sequences in turn (same heads): partial results of a small call never land where a
    larger call keeps its arrival counters."""
    ws = pk.DecodeWorkspace(512, 16, 8, 128)
    rng = np.random.default_rng(611)
    for i, B in enumerate((4, 300, 64, 512)):
        lens = rng.integers(1, 700, size=B)
        case = workloads.decode_case(lens, 16, 8, 128, 64, seed=612 + i)
        dc = DeviceCase(case)
        dc.store()
        out = dc.decode(grid_ctas=0, workspace=ws)
        assert dc.dev_err() == 0
        ok, ov = oracle_after_store(case)
        got = to_f64(out)
        assert np.all(np.isfinite(got)), f"batch {B}: a row was never written"
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens)
        assert_close(got, ref, f"batch {B}")
