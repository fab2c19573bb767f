"""Pins of the oracle's IEEE binary16 (fp16) element type and of head_dim 64.

The fp16 widening is checked against numpy's float16 on every bit pattern (a library
routine); fp16 attention against scipy's softmax over a contiguous layout and against a
brute-force loop; fp16 and bf16 inputs holding the same exactly representable values
give the same result; head_dim 64 against the brute-force loop."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_107_gb300 import workloads
from tests.test_oracle_pins import brute_decode, brute_prefill


def test_f16_widening_matches_numpy_on_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _stored(case):
    kc, vc = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    dt = case.k_cache.dtype
    return (torch.from_numpy(kc.view(np.int16)).view(dt), torch.from_numpy(vc.view(np.int16)).view(dt))


@pytest.mark.parametrize("D,bs", [(64, 4), (64, 16), (128, 8)])
def test_fp16_decode_brute_force_tiny(D, bs):
    case = workloads.decode_case([1, 9, 40], 4, 2, D, bs, seed=300 + D + bs, dtype=torch.float16)
    kc, vc = _stored(case)
    got = oracle.decode(case.q, kc, vc, case.block_tables, case.context_lens)
    want = brute_decode(case.q, kc, vc, case.block_tables, case.context_lens, bs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("D", [64, 128])
def test_bf16_decode_head_dim_brute_force_tiny(D):
    case = workloads.decode_case([2, 17, 33], 8, 2, D, 16, seed=310 + D)
    kc, vc = _stored(case)
    got = oracle.decode(case.q, kc, vc, case.block_tables, case.context_lens)
    want = brute_decode(case.q, kc, vc, case.block_tables, case.context_lens, 16)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_fp16_decode_contiguous_matches_scipy_softmax():
    rng = np.random.default_rng(320)
    lens, H, Hk, D, bs = [1, 7, 16, 33], 8, 2, 64, 16
    B = len(lens)
    nblk = [-(-n // bs) for n in lens]
    kc = torch.zeros((sum(nblk), bs, Hk, D), dtype=torch.float16)
    vc = torch.zeros_like(kc)
    bt = np.full((B, max(nblk)), -1, np.int32)
    dk, dv = [], []
    nxt = 0
    for b, n in enumerate(lens):
        kk = torch.from_numpy(rng.standard_normal((n, Hk, D)).astype(np.float32)).half()
        vv = torch.from_numpy(rng.standard_normal((n, Hk, D)).astype(np.float32)).half()
        dk.append(kk.double().numpy())
        dv.append(vv.double().numpy())
        for j in range(nblk[b]):
            bt[b, j] = nxt
            lo, hi = j * bs, min(n, (j + 1) * bs)
            kc[nxt, :hi - lo] = kk[lo:hi]
            vc[nxt, :hi - lo] = vv[lo:hi]
            nxt += 1
    q = torch.from_numpy(rng.standard_normal((B, H, D)).astype(np.float32)).half()
    out = oracle.decode(q, kc, vc, bt, np.array(lens, np.int32))
    qd = q.double().numpy()
    for b, n in enumerate(lens):
        for h in range(H):
            j = h // (H // Hk)
            p = scipy.special.softmax(dk[b][:, j] @ qd[b, h] / math.sqrt(D))
            np.testing.assert_allclose(out[b, h], p @ dv[b][:, j], rtol=1e-12, atol=1e-13)


def test_fp16_and_bf16_agree_on_values_exact_in_both():
    """Multiples of 1/8 in [-4, 4] are exact in both formats: the two element types must
    give bit-identical fp64 results (pins that each type is widened by its own rule)."""
    rng = np.random.default_rng(330)
    case = workloads.decode_case([5, 40, 17], 8, 4, 64, 16, seed=331, poison=False)
    for t in (case.q, case.k_cache, case.v_cache):
        t.copy_(torch.from_numpy(rng.integers(-32, 33, size=t.shape).astype(np.float32) / 8))
    a = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens)
    b = oracle.decode(case.q.half(), case.k_cache.half(), case.v_cache.half(), case.block_tables,
                      case.context_lens)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("causal", [True, False])
def test_fp16_prefill_brute_force_tiny(causal):
    case = workloads.prefill_case([0, 7, 4], [3, 2, 6], 4, 2, 64, 4, seed=340, causal=causal,
                                  dtype=torch.float16)
    kc, vc = _stored(case)
    got = oracle.prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, causal=causal)
    want = brute_prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, 4, causal)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
