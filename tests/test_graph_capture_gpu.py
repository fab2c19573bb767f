"""The decode step as the engine runs it ("3.6 ModelRunner、CUDA Graph 与性能基准",
section 5): store + decode (two launches, or the fused pa_decode_step) captured once in a
CUDA graph for a batch-size bucket, then replayed with new inputs copied into static
buffers; rows past the real batch are padding (slot_mapping = -1, context_lens = 0).
Every replay must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import assert_close, bits, from_bits, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
def test_decode_step_graph_replay_with_padding_rows(fused):
    dev = torch.device("cuda")
    bucket, H, Hk, D, bs = 16, 16, 8, 128, 16
    maxb = 40
    nb = 2048
    base = workloads.decode_case([1] * bucket, H, Hk, D, bs, num_blocks=nb, seed=107900,
                                 max_blocks=maxb)
    kc = base.k_cache.to(dev)
    vc = base.v_cache.to(dev)
    # static graph inputs (the bucket's buffers)
    q = torch.zeros((bucket, H, D), dtype=torch.bfloat16, device=dev)
    k_new = torch.zeros((bucket, Hk, D), dtype=torch.bfloat16, device=dev)
    v_new = torch.zeros_like(k_new)
    slots = torch.full((bucket,), -1, dtype=torch.int32, device=dev)
    ctx = torch.zeros((bucket,), dtype=torch.int32, device=dev)
    bt = torch.full((bucket, maxb), -1, dtype=torch.int32, device=dev)
    out = torch.zeros((bucket, H, D), dtype=torch.bfloat16, device=dev)
    ws = pk.DecodeWorkspace(bucket, H, Hk, D, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        if fused:
            pk.pa_decode_step(out, q, k_new, v_new, kc, vc, slots, bt, ctx, workspace=ws,
                              dev_err=err)
        else:
            pk.pa_store_kvcache(k_new, v_new, kc, vc, slots, dev_err=err)
            pk.pa_decode(out, q, kc, vc, bt, ctx, workspace=ws, dev_err=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    rng = np.random.default_rng(107901)
    for real in (16, 11, 3, 1):
        # a fresh batch of `real` sequences over the same pool; the rest are padding rows
        lens = rng.integers(1, maxb * bs, size=real)
        case = workloads.decode_case(lens, H, Hk, D, bs, num_blocks=nb,
                                     seed=int(rng.integers(1 << 30)), max_blocks=maxb)
        kc.copy_(case.k_cache.to(dev))
        vc.copy_(case.v_cache.to(dev))
        q.zero_()
        q[:real] = case.q.to(dev)
        k_new[:real] = case.k_new.to(dev)
        v_new[:real] = case.v_new.to(dev)
        slots.fill_(-1)
        slots[:real] = torch.from_numpy(case.slot_mapping).to(dev)
        ctx.zero_()
        ctx[:real] = torch.from_numpy(case.context_lens).to(dev)
        bt.fill_(-1)
        bt[:real] = torch.from_numpy(case.block_tables).to(dev)
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                      case.slot_mapping)
        assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens)
        got = to_f64(out)
        assert_close(got[:real], ref, f"replay with {real} real rows")
        assert np.all(got[real:] == 0.0), "padding rows must be zero"


def test_prefill_step_graph_replay_with_padding_sequences():
    """Store + chunked prefill captured once for a bucket (4 sequences, 1024 new-token rows,
    at most 512 new tokens per sequence) and replayed on fresh batches over the same static
    buffers: unused sequences have no tokens (cu_seqlens repeat), unused token rows have
    slot -1. Every real output row must match the oracle; the tensor maps built at capture
    time stay valid because the cache buffers do not move."""
    dev = torch.device("cuda")
    S, N, maxq, maxk, H, Hk, D, bs = 4, 1024, 512, 2048, 16, 8, 128, 256
    maxb = maxk // bs
    nb = 64
    kc = torch.zeros((nb, bs, Hk, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    q = torch.zeros((N, H, D), dtype=torch.bfloat16, device=dev)
    k_new = torch.zeros((N, Hk, D), dtype=torch.bfloat16, device=dev)
    v_new = torch.zeros_like(k_new)
    slots = torch.full((N,), -1, dtype=torch.int32, device=dev)
    bt = torch.full((S, maxb), -1, dtype=torch.int32, device=dev)
    cu_q = torch.zeros((S + 1,), dtype=torch.int32, device=dev)
    cu_k = torch.zeros((S + 1,), dtype=torch.int32, device=dev)
    out = torch.zeros((N, H, D), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        pk.pa_store_kvcache(k_new, v_new, kc, vc, slots, dev_err=err)
        pk.pa_prefill_varlen(out, q, kc, vc, bt, cu_q, cu_k, maxq, maxk, causal=True,
                             dev_err=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture (no sequences yet)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    rng = np.random.default_rng(107902)
    for real in (4, 2, 1):
        new = rng.integers(1, maxq // 2 + 1, size=real)
        cached = rng.integers(0, maxk - maxq + 1, size=real)
        case = workloads.prefill_case(cached, new, H, Hk, D, bs, num_blocks=nb,
                                      seed=int(rng.integers(1 << 30)))
        T = int(case.cu_seqlens_q[-1])
        assert T <= N
        kc.copy_(case.k_cache.to(dev))
        vc.copy_(case.v_cache.to(dev))
        q.zero_()
        q[:T] = case.q.to(dev)
        k_new[:T] = case.k_new.to(dev)
        v_new[:T] = case.v_new.to(dev)
        slots.fill_(-1)
        slots[:T] = torch.from_numpy(case.slot_mapping).to(dev)
        bt.fill_(-1)
        bt[:real, :case.block_tables.shape[1]] = torch.from_numpy(case.block_tables).to(dev)
        cq = np.full(S + 1, T, np.int32)
        ck = np.full(S + 1, int(case.cu_seqlens_k[-1]), np.int32)
        cq[:real + 1] = case.cu_seqlens_q
        ck[:real + 1] = case.cu_seqlens_k
        cu_q.copy_(torch.from_numpy(cq))
        cu_k.copy_(torch.from_numpy(ck))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error bits {int(err.item())}"
        ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                      case.slot_mapping)
        assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)
        ref = oracle.prefill(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                             case.cu_seqlens_q, case.cu_seqlens_k, causal=True)
        got = to_f64(out)
        assert np.all(np.isfinite(got[:T]))
        assert_close(got[:T], ref, f"prefill replay with {real} sequences")
        assert np.all(np.isnan(got[T:])), "rows past the batch's tokens must not be written"


def test_decode_step_graphs_per_batch_bucket():
    """One graph per batch-size bucket (1, 2, 4, 8, 16, 32), as the engine captures them
    ("3.6 ModelRunner、CUDA Graph 与性能基准", section 5), all over slices of one set of
    static buffers and one workspace sized for the largest bucket. Each fresh batch replays
    the smallest bucket that holds it, its extra rows padding; the outputs must match the
    oracle."""
    dev = torch.device("cuda")
    buckets = (1, 2, 4, 8, 16, 32)
    top, H, Hk, D, bs = buckets[-1], 16, 8, 128, 32
    maxb, nb = 24, 1024
    kc = torch.zeros((nb, bs, Hk, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    q = torch.zeros((top, H, D), dtype=torch.bfloat16, device=dev)
    k_new = torch.zeros((top, Hk, D), dtype=torch.bfloat16, device=dev)
    v_new = torch.zeros_like(k_new)
    slots = torch.full((top,), -1, dtype=torch.int32, device=dev)
    ctx = torch.zeros((top,), dtype=torch.int32, device=dev)
    bt = torch.full((top, maxb), -1, dtype=torch.int32, device=dev)
    out = torch.zeros((top, H, D), dtype=torch.bfloat16, device=dev)
    ws = pk.DecodeWorkspace(top, H, Hk, D, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(n):
        pk.pa_decode_step(out[:n], q[:n], k_new[:n], v_new[:n], kc, vc, slots[:n], bt[:n],
                          ctx[:n], workspace=ws, dev_err=err)

    graphs = {}
    pool = None
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for n in buckets:
            step(n)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for n in reversed(buckets):  # largest first, sharing one memory pool
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, pool=pool):
            step(n)
        pool = g.pool()
        graphs[n] = g

    rng = np.random.default_rng(107903)
    for real in (1, 3, 7, 12, 32, 20, 2):
        n = min(b for b in buckets if b >= real)
        lens = rng.integers(1, maxb * bs, size=real)
        case = workloads.decode_case(lens, H, Hk, D, bs, num_blocks=nb,
                                     seed=int(rng.integers(1 << 30)), max_blocks=maxb)
        kc.copy_(case.k_cache.to(dev))
        vc.copy_(case.v_cache.to(dev))
        q.zero_()
        q[:real] = case.q.to(dev)
        k_new[:real] = case.k_new.to(dev)
        v_new[:real] = case.v_new.to(dev)
        slots.fill_(-1)
        slots[:real] = torch.from_numpy(case.slot_mapping).to(dev)
        ctx.zero_()
        ctx[:real] = torch.from_numpy(case.context_lens).to(dev)
        bt.fill_(-1)
        bt[:real] = torch.from_numpy(case.block_tables).to(dev)
        out.fill_(float("nan"))
        graphs[n].replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error bits {int(err.item())}"
        ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                      case.slot_mapping)
        assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens)
        got = to_f64(out)
        assert_close(got[:real], ref, f"{real} sequences in the bucket of {n}")
        assert np.all(got[real:n] == 0.0), "padding rows of the bucket must be zero"
        assert np.all(np.isnan(got[n:])), "rows past the bucket must not be written"
