"""pa_decode_noalloc: the decode entry point for callers that cannot allocate device
memory (a plugin inside a host program that owns all device memory, a runtime that forbids
allocation after start-up, a caller with a fixed memory budget). Its scratch is a fixed
array inside the library instead of a caller-allocated workspace.

Its output is checked element by element against the fp64 oracle applied after the
oracle's own store, at the parity tolerance, on two calls in a row (the second call finds
the array holding the first call's contents); it is also compared with pa_decode on the
same inputs.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process (the first call on the
device performs the one-time address lookup)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import (ATOL, RTOL, DeviceCase, assert_close, from_bits,
                               oracle_after_store, to_f64)

pytestmark = pytest.mark.gpu


def _close(got, ref):
    g, r = to_f64(got), to_f64(ref)
    assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r)), float(np.max(np.abs(g - r)))


def _oracle_decode(case):
    ok, ov = oracle_after_store(case)
    return oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                         case.context_lens)


def test_noalloc_matches_oracle_on_consecutive_calls():
    """48 random lengths up to 3000 plus 0, 1, 256 and 257 tokens; 4 query heads per KV
    head (the tensor-core decode), block size 256."""
    lens = list(np.random.default_rng(17).integers(1, 3000, 48)) + [0, 1, 256, 257]
    case = workloads.decode_case(lens, 32, 8, 128, 256, seed=107700, num_blocks=1024)
    dc = DeviceCase(case)
    dc.store()
    ref_lib = dc.decode()  # the workspace-taking entry point
    torch.cuda.synchronize()
    ref = _oracle_decode(case)
    for call in range(2):
        out = torch.full_like(dc.q, float("nan"))
        pk.pa_decode_noalloc(out, dc.q, dc.k_cache, dc.v_cache, dc.bt, dc.ctx, dev_err=dc.err)
        assert dc.dev_err() == 0, f"call {call}: device error bits"
        assert_close(to_f64(out), ref, f"noalloc call {call} vs oracle")
        _close(out, ref_lib)


def test_noalloc_cuda_core_shape_and_grids_after_first():
    """Two query heads per KV head (the CUDA-core decode), block size 16, a different batch
    and split counts right after the first test: the counters are cleared per call."""
    case = workloads.decode_case([5, 700, 33, 4097], 16, 8, 128, 16, seed=107701)
    dc = DeviceCase(case)
    dc.store()
    ref_lib = dc.decode(grid_ctas=7)
    torch.cuda.synchronize()
    ref = _oracle_decode(case)
    for grid in (7, 0):
        out = torch.full_like(dc.q, float("nan"))
        pk.pa_decode_noalloc(out, dc.q, dc.k_cache, dc.v_cache, dc.bt, dc.ctx, grid_ctas=grid,
                             dev_err=dc.err)
        assert dc.dev_err() == 0
        assert_close(to_f64(out), ref, f"noalloc grid {grid} vs oracle")
        _close(out, ref_lib)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """64 query heads and the largest grid (4 CTAs per SM) need 4*SMs*2*64*128*4 bytes of
    partial outputs, above the 16 MiB array: PA_ERR_WORKSPACE before any launch. The
    tensors themselves are a few KB."""
    dev = torch.device("cuda")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert 4 * sms * 2 * 64 * 128 * 4 > 16 << 20
    q = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((2, 16, 8, 128), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    ctx = torch.ones(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    with pytest.raises(pk.PagedAttentionError, match="WORKSPACE"):
        pk.pa_decode_noalloc(out, q, kc, kc, bt, ctx, grid_ctas=4 * sms)
    # the C entry point itself, with the same small buffers
    lib = pk.load_library()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.pa_decode_noalloc(P(out), P(q), P(kc), P(kc), P(bt), 1, P(ctx), 1, 64, 8, 128, 16,
                               ctypes.c_int64(2), ctypes.c_float(0.0), 4 * sms, None, None)
    assert rc == 4  # PA_ERR_WORKSPACE
