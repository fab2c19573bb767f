"""Bounded pipeline waits on the GPU: a wait that runs out ends the launch with
PA_DEV_ERR_TIMEOUT in the device error word instead of hanging, the CUDA context stays
usable, and the next call (on a zeroed workspace) is correct.

A wait cannot be made to run out in the product library without breaking the GPU's
memory system, so this test builds a second copy of the library into a temporary directory
with two preprocessor flags: PA_WAIT_CYCLES shortens every wait limit to 2^17 SM cycles
(about 65 us), and PA_TEST_DELAY_LAST_TILE_CYCLES makes the CUDA-core decode's producer
warp hold back the copies of its last key tile for 2^20 cycles (about 0.5 ms) before
issuing them. The consumer warps' wait on that tile therefore runs out; the producer still
issues the copies, late, and waits for them to land before the CTA exits, so nothing is
left in flight. One CTA (grid_ctas = 1) and one sequence keep every tile in that CTA, so
no partial result or arrival counter is involved. The tensor-core prefill is not driven
into a timeout."""
import ctypes
import os

import numpy as np
import pytest
import torch

import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import build as lib_build
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import DeviceCase, assert_close, from_bits, oracle_after_store, to_f64

import oracle

pytestmark = pytest.mark.gpu

WAIT_CYCLES = 1 << 17
DELAY_CYCLES = 1 << 20


@pytest.fixture(scope="module")
def timeout_lib(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("timeout_build") / "libpagedkv_timeout.so")
    lib_build.build(lib_path=path, extra_flags=(f"-DPA_WAIT_CYCLES={WAIT_CYCLES}ll",
                                                f"-DPA_TEST_DELAY_LAST_TILE_CYCLES={DELAY_CYCLES}ll"))
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64, f32,
                              i32, vp, sz, vp, vp]
    lib.pa_decode.restype = i32
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.pa_decode_workspace_size.restype = sz
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_wait_that_runs_out_sets_timeout_and_returns(timeout_lib):
    # one sequence of 300 tokens, 2 query heads per KV head at head_dim 128 (the CUDA-core
    # decode), block size 16: 19 key tiles, all in the single CTA
    case = workloads.decode_case([300], 16, 8, 128, 16, seed=107800)
    dc = DeviceCase(case)
    dc.store()
    torch.cuda.synchronize()
    B, H, D = dc.q.shape
    nb, bs, hk, _ = dc.k_cache.shape
    ws_bytes = timeout_lib.pa_decode_workspace_size(B, H, hk, D)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dc.dev)
    out = torch.full_like(dc.q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=dc.dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = timeout_lib.pa_decode(_ptr(out), _ptr(dc.q), _ptr(dc.k_cache), _ptr(dc.v_cache),
                               _ptr(dc.bt), dc.bt.shape[1], _ptr(dc.ctx), B, H, hk, D, 1, bs, nb,
                               0.0, 1, _ptr(ws), ws_bytes, _ptr(err), stream)
    assert rc == 0
    torch.cuda.synchronize()  # raises if the launch faulted
    assert int(err.item()) & pk.PA_DEV_ERR["timeout"], f"error word {int(err.item())}"

    # the context is still usable: the product library on a fresh workspace is correct
    dc.err.zero_()
    got = dc.decode(grid_ctas=1)
    assert dc.dev_err() == 0
    ok, ov = oracle_after_store(case)
    ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                        case.context_lens)
    assert_close(to_f64(got), ref, "decode after a timed-out launch")
