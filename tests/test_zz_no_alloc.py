"""pa_decode_noalloc: the decode entry point for callers that cannot allocate device
memory (its scratch is a fixed array inside the library). Its output must match
pa_decode's on the same inputs, call after call, within the parity tolerance.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process (the first call on the
device performs the one-time address lookup)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import ATOL, RTOL, DeviceCase, to_f64

pytestmark = pytest.mark.gpu


def _close(got, ref):
    g, r = to_f64(got), to_f64(ref)
    assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r)), float(np.max(np.abs(g - r)))


def test_noalloc_matches_pa_decode_on_consecutive_calls():
    lens = list(np.random.default_rng(17).integers(1, 3000, 48)) + [0, 1, 256, 257]
    case = workloads.decode_case(lens, 32, 8, 128, 256, seed=107700, num_blocks=1024)
    dc = DeviceCase(case)
    dc.store()
    ref = dc.decode()  # the workspace-taking entry point
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(dc.q, float("nan"))
        pk.pa_decode_noalloc(out, dc.q, dc.k_cache, dc.v_cache, dc.bt, dc.ctx, dev_err=dc.err)
        assert dc.dev_err() == 0, f"call {call}: device error bits"
        _close(out, ref)


def test_noalloc_second_shape_and_grid_after_first():
    """A different batch and split count right after: the counters are cleared per call."""
    case = workloads.decode_case([5, 700, 33, 4097], 16, 8, 128, 16, seed=107701)
    dc = DeviceCase(case)
    dc.store()
    ref = dc.decode(grid_ctas=7)
    for grid in (7, 0):
        out = torch.full_like(dc.q, float("nan"))
        pk.pa_decode_noalloc(out, dc.q, dc.k_cache, dc.v_cache, dc.bt, dc.ctx, grid_ctas=grid,
                             dev_err=dc.err)
        assert dc.dev_err() == 0
        _close(out, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    dev = torch.device("cuda")
    B = 1 << 20  # counters alone: 32 MiB > 16 MiB
    q = torch.zeros((B, 16, 128), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((2, 16, 8, 128), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    ctx = torch.zeros(B, dtype=torch.int32, device=dev)
    with pytest.raises(pk.PagedAttentionError, match="WORKSPACE"):
        pk.pa_decode_noalloc(torch.empty_like(q), q, kc, kc, bt, ctx)
