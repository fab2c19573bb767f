"""GPU parity of the head_dim 64 and IEEE fp16 variants (store, decode, fused decode step,
prefill) against the fp64 oracle. The nano-vllm overview page's block class ("PagedAttention：
KV Cache") takes head_dim and dtype as parameters and makes the block size configurable.
Tolerance as for bf16 / head_dim 128: |o - ref| <= 1e-2 + 1e-2*|ref|."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import DeviceCase, assert_close, bits, from_bits, to_f64

pytestmark = pytest.mark.gpu

VARIANTS = [(64, torch.bfloat16), (64, torch.float16), (128, torch.float16)]
IDS = ["d64-bf16", "d64-fp16", "d128-fp16"]


def stored(case):
    ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    dt = case.k_cache.dtype
    return ok, ov, from_bits(ok, dt), from_bits(ov, dt)


@pytest.mark.parametrize("D,dt", VARIANTS, ids=IDS)
@pytest.mark.parametrize("H,Hk,lens,bs", [
    (16, 8, [1, 17, 256, 300, 0], 256), (8, 8, [5, 40, 129], 16), (32, 8, [1000, 3, 77], 32),
    (8, 2, [64, 65, 1], 8), (4, 1, [300, 2], 64), (32, 16, [9, 500], 16), (64, 8, [130, 33], 16)])
def test_store_and_decode(D, dt, H, Hk, lens, bs):
    """Store (bit exact) then decode, over GQA groups 1..8 and head slabs 8, 4, 2, 1."""
    case = workloads.decode_case(lens, H, Hk, D, bs, seed=2000 + D + H + Hk + bs, dtype=dt)
    dc = DeviceCase(case)
    dc.store()
    for grid in (0, 3):
        out = dc.decode(grid_ctas=grid)
        assert dc.dev_err() == 0
        ok, ov, kt, vt = stored(case)
        assert np.array_equal(bits(dc.k_cache), ok) and np.array_equal(bits(dc.v_cache), ov)
        got = to_f64(out)
        assert np.all(np.isfinite(got))
        assert_close(got, oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens),
                     f"decode D={D} {dt}")


@pytest.mark.parametrize("D,dt", VARIANTS, ids=IDS)
def test_fused_step_equals_two_launches(D, dt):
    case = workloads.decode_case([1, 17, 33, 300, 0, 1000], 16, 4, D, 16, seed=2100 + D,
                                 dtype=dt)
    two = DeviceCase(case)
    two.store()
    ref = two.decode()
    one = DeviceCase(case)
    out = torch.full_like(one.q, float("nan"))
    pk.pa_decode_step(out, one.q, one.k_new, one.v_new, one.k_cache, one.v_cache, one.slots,
                      one.bt, one.ctx, dev_err=one.err)
    assert one.dev_err() == 0 and two.dev_err() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(one.k_cache.view(torch.int16), two.k_cache.view(torch.int16))
    ok, ov, kt, vt = stored(case)
    assert_close(to_f64(out), oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens),
                 "fused step")


@pytest.mark.parametrize("D,dt", VARIANTS, ids=IDS)
@pytest.mark.parametrize("cached,new,H,Hk,bs,causal", [
    ([0, 17, 256, 1000], [70, 300, 1, 257], 16, 8, 256, True),
    ([40, 0, 300], [100, 33, 130], 32, 8, 16, True),
    ([0, 150, 700], [200, 77, 129], 8, 8, 128, True),
    ([0, 37, 256], [50, 91, 300], 16, 4, 64, False),
    ([5, 0], [129, 64], 4, 1, 32, True)])
def test_prefill(D, dt, cached, new, H, Hk, bs, causal):
    case = workloads.prefill_case(cached, new, H, Hk, D, bs, seed=2200 + D + H + bs,
                                  causal=causal, dtype=dt)
    dc = DeviceCase(case)
    dc.store()
    out = dc.prefill()
    assert dc.dev_err() == 0
    ok, ov, kt, vt = stored(case)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.prefill(case.q, kt, vt, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, causal=causal)
    assert_close(got, ref, f"prefill D={D} {dt}")


@pytest.mark.parametrize("D,dt", VARIANTS, ids=IDS)
def test_single_token_prefill_equals_decode(D, dt):
    case = workloads.prefill_case([0, 99, 256, 511], [1, 1, 1, 1], 16, 8, D, 256, seed=2300 + D,
                                  dtype=dt)
    dc = DeviceCase(case)
    dc.store()
    pre = dc.prefill()
    dec = torch.empty_like(dc.q)
    ctx = torch.from_numpy(np.diff(case.cu_seqlens_k).astype(np.int32)).cuda()
    pk.pa_decode(dec, dc.q, dc.k_cache, dc.v_cache, dc.bt, ctx)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to_f64(pre), to_f64(dec), atol=2e-2, rtol=2e-2)


def test_fp16_large_values_round_as_fp16():
    """Values near fp16's range end (|v| up to 2^14) survive: the output is rounded to fp16,
    not through bf16."""
    case = workloads.decode_case([7, 40], 8, 4, 64, 16, seed=2400, dtype=torch.float16,
                                 poison=False)
    case.v_cache.mul_(4096.0)
    case.v_new.mul_(4096.0)
    dc = DeviceCase(case)
    dc.store()
    out = dc.decode()
    assert dc.dev_err() == 0
    ok, ov, kt, vt = stored(case)
    ref = oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens)
    got = to_f64(out)
    assert np.all(np.abs(got - ref) <= 2 * np.abs(ref) * 2.0 ** -11 + 4096 * 1e-3)


@pytest.mark.parametrize("D,dt", [(128, torch.bfloat16)] + VARIANTS, ids=["d128-bf16"] + IDS)
@pytest.mark.parametrize("H,Hk", [(24, 8), (40, 8), (48, 8), (56, 8), (64, 8), (32, 8), (20, 4),
                                  (10, 2), (7, 1)])
def test_tensor_core_groups(D, dt, H, Hk):
    """Query-head groups of 3..8 per KV head (the tensor-core path; 5 is the 40/8 layout of
    the 14B-class models): decode and the fused step, long and short contexts, split
    across CTAs (grid 5) and whole."""
    case = workloads.decode_case([1, 17, 300, 1500, 0, 64], H, Hk, D, 64,
                                 seed=2500 + H + 3 * Hk + D, dtype=dt)
    ok, ov, kt, vt = stored(case)
    ref = oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens)
    for grid in (0, 5):
        dc = DeviceCase(case)
        dc.store()
        out = dc.decode(grid_ctas=grid)
        assert dc.dev_err() == 0
        got = to_f64(out)
        assert np.all(np.isfinite(got))
        assert_close(got, ref, f"decode G={H // Hk} D={D} {dt} grid={grid}")
        one = DeviceCase(case)
        o2 = torch.full_like(one.q, float("nan"))
        pk.pa_decode_step(o2, one.q, one.k_new, one.v_new, one.k_cache, one.v_cache, one.slots,
                          one.bt, one.ctx, grid_ctas=grid, dev_err=one.err)
        assert one.dev_err() == 0
        assert torch.equal(o2.view(torch.int16), out.view(torch.int16))
        assert torch.equal(one.k_cache.view(torch.int16), dc.k_cache.view(torch.int16))


@pytest.mark.parametrize("bs", [5, 8, 12, 16, 24, 48, 256])
@pytest.mark.parametrize("H,Hk,D", [(32, 8, 128), (64, 8, 64), (16, 2, 128), (8, 1, 128),
                                    (12, 4, 64)])
def test_tensor_core_block_sizes(bs, H, Hk, D):
    """The tensor-core path's stage fill for every kind of block size: TMA boxes of a whole
    stage (256), of 8 to 48 tokens (several boxes per stage: 8, 16, 24 -> boxes of 8, 48 ->
    boxes of 16), and 16-byte copies where no box of 8 or more tokens fits a block (5, 12).
    Cache tails past each context hold NaN; decode and the fused step, split and whole."""
    case = workloads.decode_case([1, 9, 130, 700, 0, 33, 2049], H, Hk, D, bs,
                                 seed=2600 + bs + H + Hk + D)
    ok, ov, kt, vt = stored(case)
    ref = oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens)
    for grid in (0, 7):
        dc = DeviceCase(case)
        dc.store()
        out = dc.decode(grid_ctas=grid)
        assert dc.dev_err() == 0
        got = to_f64(out)
        assert np.all(np.isfinite(got))
        assert_close(got, ref, f"decode H={H} Hk={Hk} D={D} bs={bs} grid={grid}")
        one = DeviceCase(case)
        o2 = torch.full_like(one.q, float("nan"))
        pk.pa_decode_step(o2, one.q, one.k_new, one.v_new, one.k_cache, one.v_cache, one.slots,
                          one.bt, one.ctx, grid_ctas=grid, dev_err=one.err)
        assert one.dev_err() == 0
        assert torch.equal(o2.view(torch.int16), out.view(torch.int16))
        assert torch.equal(one.k_cache.view(torch.int16), dc.k_cache.view(torch.int16))
        assert torch.equal(one.v_cache.view(torch.int16), dc.v_cache.view(torch.int16))


@pytest.mark.parametrize("grid", [3, 20, 152])
def test_tensor_core_segment_switches(grid):
    """256 sequences, four in five of them a single tile (G=8, head_dim 128, block_size 16):
    every CTA switches sequence, and so reloads its Q slot, on almost every tile. Repeated
    launches must all match the oracle (a Q slot released before its loads complete shows
    up here as a few wrong rows)."""
    rng = np.random.default_rng(31)
    lens = np.where(rng.random(256) < 0.8, rng.integers(1, 17, 256), rng.integers(17, 80, 256))
    case = workloads.decode_case(lens.tolist(), 64, 8, 128, 16, seed=77)
    ok, ov, kt, vt = stored(case)
    ref = oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens)
    dc = DeviceCase(case)
    dc.store()
    for rep in range(12):
        out = dc.decode(grid_ctas=grid)
        assert dc.dev_err() == 0
        assert_close(to_f64(out), ref, f"segment switches grid={grid} launch {rep}")
