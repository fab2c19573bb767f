"""Seeded sweeps of random shapes through the store, the fused decode step and the
prefill, each compared with the fp64 oracle: batch sizes, length mixes (empty sequences
and block edges included), GQA group sizes 1-8, head slabs, head_dim 64/128, bf16 and
IEEE fp16, block sizes 16-256 and, for the decode, automatic and explicit CTA counts.
The pages fix the operations (the nano-vllm overview page: "KVCache的写入",
"PageAttention原理", "如何适配不同请求不同序列长度"); the sweeps only vary shapes. Cache
bytes bit exact, attention within |o - ref| <= 1e-2 + 1e-2*|ref|."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import DeviceCase, assert_close, bits, from_bits, to_f64

pytestmark = pytest.mark.gpu

GROUPS = [(8, 8), (16, 8), (32, 8), (64, 8), (8, 4), (16, 2), (4, 1), (12, 4), (16, 16)]
PREFILL_GROUPS = [(8, 8), (16, 8), (32, 8), (64, 8), (8, 4), (16, 2), (4, 1), (16, 16)]
DTYPES = [torch.bfloat16, torch.float16]


def _stored(case):
    ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    dt = case.k_cache.dtype
    return ok, ov, from_bits(ok, dt), from_bits(ov, dt)


@pytest.mark.parametrize("seed", range(24))
def test_random_fused_decode_step(seed):
    rng = np.random.default_rng(31000 + seed)
    H, Hk = GROUPS[rng.integers(len(GROUPS))]
    D = int(rng.choice([64, 128]))
    dt = DTYPES[rng.integers(2)]
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    B = int(rng.integers(1, 40))
    lens = rng.integers(1, 1500, size=B)
    # a few exact block edges
    for i in range(B):
        if rng.random() < 0.2:
            lens[i] = bs * int(rng.integers(1, 6)) + int(rng.choice([-1, 0, 1]))
    lens = np.maximum(lens, 1)
    case = workloads.decode_case(lens.tolist(), H, Hk, D, bs, seed=31100 + seed, dtype=dt)
    dc = DeviceCase(case)
    grid = int(rng.choice([0, 0, 1, 7, 200]))
    out = torch.full_like(dc.q, float("nan"))
    pk.pa_decode_step(out, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.slots, dc.bt,
                      dc.ctx, grid_ctas=grid, dev_err=dc.err)
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov, kt, vt = _stored(case)
    assert np.array_equal(bits(dc.k_cache), ok) and np.array_equal(bits(dc.v_cache), ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.decode(case.q, kt, vt, case.block_tables, case.context_lens)
    assert_close(got, ref, f"decode step H={H} Hk={Hk} D={D} {dt} bs={bs} B={B} grid={grid}")


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill(seed):
    rng = np.random.default_rng(32000 + seed)
    H, Hk = PREFILL_GROUPS[rng.integers(len(PREFILL_GROUPS))]
    D = int(rng.choice([64, 128]))
    dt = DTYPES[rng.integers(2)]
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    S = int(rng.integers(1, 24))
    cached = rng.integers(0, 700, size=S)
    new = rng.integers(1, 300, size=S)
    for i in range(S):
        if rng.random() < 0.3:
            cached[i] = 0
        if rng.random() < 0.2:
            new[i] = int(rng.choice([1, 63, 64, 65, 128, 129]))
    causal = bool(rng.random() < 0.75)
    case = workloads.prefill_case(cached.tolist(), new.tolist(), H, Hk, D, bs,
                                  seed=32100 + seed, causal=causal, dtype=dt)
    dc = DeviceCase(case)
    dc.store()
    out = dc.prefill()
    assert dc.dev_err() == 0, f"device error bits {dc.dev_err()}"
    ok, ov, kt, vt = _stored(case)
    assert np.array_equal(bits(dc.k_cache), ok) and np.array_equal(bits(dc.v_cache), ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.prefill(case.q, kt, vt, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, causal=causal)
    assert_close(got, ref, f"prefill H={H} Hk={Hk} D={D} {dt} bs={bs} S={S} causal={causal}")
