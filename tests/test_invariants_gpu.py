"""Bit-level invariants of the GPU path that follow from what paging is ("PagedAttention：KV
Cache", logical-to-physical block mapping; "nano-vllm解读", "PageAttention原理"): the block
table only relocates memory, so

* moving every block to another physical id (and the table and slots with it) changes
  no bit of any output: the kernels' split of the work depends on the context lengths
  only, never on where a block lives;
* a context of one key returns that key's value exactly (its probability is 1).

Both decode kernels, the fused step and the prefill are covered."""
import numpy as np
import pytest
import torch

import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import DeviceCase, bits

pytestmark = pytest.mark.gpu


def relabel(case, seed):
    """The same case with its blocks moved to physical ids perm[old] (data, tables, slots)."""
    rng = np.random.default_rng(seed)
    nb, bs = case.num_blocks, case.block_size
    perm = rng.permutation(nb)
    inv = np.argsort(perm)
    idx = torch.from_numpy(inv.astype(np.int64))
    moved = dict(case.__dict__)
    moved["k_cache"] = case.k_cache[idx].contiguous()  # new block perm[p] holds old block p
    moved["v_cache"] = case.v_cache[idx].contiguous()
    bt = case.block_tables.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    moved["block_tables"] = bt
    sl = case.slot_mapping.astype(np.int64).copy()
    ok = sl >= 0
    sl[ok] = perm[sl[ok] // bs] * bs + sl[ok] % bs
    moved["slot_mapping"] = sl.astype(np.int32)
    return type(case)(**moved)


@pytest.mark.parametrize("H,Hk,D", [(16, 8, 128), (32, 8, 128), (64, 8, 128), (16, 8, 64)])
@pytest.mark.parametrize("fused", [False, True])
def test_decode_bits_do_not_depend_on_physical_blocks(H, Hk, D, fused):
    lens = list(np.random.default_rng(11).integers(1, 3000, 40)) + [0, 1, 256]
    case = workloads.decode_case(lens, H, Hk, D, 256, seed=4400 + H + D, num_blocks=700)
    outs = []
    for c in (case, relabel(case, 1), relabel(case, 2)):
        dc = DeviceCase(c)
        if fused:
            out = torch.full_like(dc.q, float("nan"))
            pk.pa_decode_step(out, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.slots,
                              dc.bt, dc.ctx, dev_err=dc.err)
        else:
            dc.store()
            out = dc.decode()
        assert dc.dev_err() == 0
        outs.append(out)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_bits_do_not_depend_on_physical_blocks(D):
    case = workloads.prefill_case([0, 300, 1000, 77], [129, 77, 260, 500], 16, 8, D, 256,
                                  seed=4500 + D, num_blocks=64)
    outs = []
    for c in (case, relabel(case, 3), relabel(case, 4)):
        dc = DeviceCase(c)
        dc.store()
        out = dc.prefill()
        assert dc.dev_err() == 0
        outs.append(out)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("H,Hk,D", [(16, 8, 128), (32, 8, 128), (16, 8, 64)])
@pytest.mark.parametrize("fused", [False, True])
def test_one_key_returns_its_value_exactly(H, Hk, D, fused):
    """Every sequence has context 1: its only key is the new token, so each query head's
    output is that token's value row of its KV head, bit for bit."""
    B = 37
    case = workloads.decode_case([1] * B, H, Hk, D, 16, seed=4600 + H + D)
    dc = DeviceCase(case)
    if fused:
        out = torch.full_like(dc.q, float("nan"))
        pk.pa_decode_step(out, dc.q, dc.k_new, dc.v_new, dc.k_cache, dc.v_cache, dc.slots,
                          dc.bt, dc.ctx, dev_err=dc.err)
    else:
        dc.store()
        out = dc.decode()
    assert dc.dev_err() == 0
    G = H // Hk
    expect = bits(case.v_new).reshape(B, Hk, 1, D).repeat(G, axis=2).reshape(B, H, D)
    assert np.array_equal(bits(out), expect)
