"""GPU parity of pa_decode_step: the store of each sequence's new token and the decode over
the cache holding it, fused into one launch ("nano-vllm解读", sections "KVCache的写入" and
"CUDAGraph优化"; "3.6 ModelRunner、CUDA Graph 与性能基准", sections 2 and 5).

Each case checks two things. (1) The output and both caches equal, bit for bit, the two
separate launches pa_store_kvcache then pa_decode on a copy of the same inputs. (2) Both
equal the fp64 oracle applied after its own store: the caches bit for bit, the output
within |o - ref| <= 1e-2 + 1e-2*|ref|."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import workloads
from tests.gpu_helpers import (DeviceCase, assert_close, bits, from_bits, oracle_after_store,
                               to_f64)

pytestmark = pytest.mark.gpu


def fused(dc, grid_ctas=0, k_new=None, v_new=None, slots=None):
    out = torch.full_like(dc.q, float("nan"))
    pk.pa_decode_step(out, dc.q, dc.k_new if k_new is None else k_new,
                      dc.v_new if v_new is None else v_new, dc.k_cache, dc.v_cache,
                      dc.slots if slots is None else slots, dc.bt, dc.ctx,
                      grid_ctas=grid_ctas, dev_err=dc.err)
    return out


def run_step(case, grid_ctas=0, pairs=None, k_new=None, v_new=None):
    two = DeviceCase(case)
    two.store()
    ref_out = two.decode(grid_ctas=grid_ctas)
    assert two.dev_err() == 0
    one = DeviceCase(case)
    out = fused(one, grid_ctas, k_new=k_new, v_new=v_new)
    assert one.dev_err() == 0, f"device error bits {one.dev_err()}"
    # (1) the fused launch is the two launches, bit for bit
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), "output differs"
    assert torch.equal(one.k_cache.view(torch.int16), two.k_cache.view(torch.int16))
    assert torch.equal(one.v_cache.view(torch.int16), two.v_cache.view(torch.int16))
    # (2) against the oracle
    ok, ov = oracle_after_store(case)
    assert np.array_equal(bits(one.k_cache), ok) and np.array_equal(bits(one.v_cache), ov)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    if pairs is None:
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens)
        assert_close(got, ref, case.name)
    else:
        ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                            case.context_lens, pairs=pairs)
        assert_close(got.reshape(-1, case.head_dim)[pairs], ref, case.name)
    return one, out


def test_tiny_workload_with_skipped_slot():
    """B=4, context {1,17,256,300}; sequence 1 has slot -1, so its newest position keeps
    the value already in the cache and the decode reads that value."""
    run_step(workloads.workload(1))


@pytest.mark.parametrize("grid", [1, 2, 5, 600])
def test_tiny_any_split_count(grid):
    run_step(workloads.workload(1), grid_ctas=grid)


@pytest.mark.parametrize("lens,bs", [
    ([1], 256), ([1], 16), ([15, 16, 17], 16), ([255, 256, 257], 256), ([0, 3, 0], 16),
    ([31, 1, 64, 100, 2], 32), ([513, 7, 9], 8), ([17, 33], 8)])
def test_context_edges(lens, bs):
    """The new token alone in its tile (context 1, 17, 33), at a tile or block edge, tiles
    crossing blocks (block_size 8: one copy per row), padding rows."""
    run_step(workloads.decode_case(lens, 16, 8, 128, bs, seed=1400 + sum(lens) + bs))


@pytest.mark.parametrize("H,Hk", [(16, 16), (32, 16), (8, 4), (4, 2), (8, 1), (64, 8)])
def test_head_layouts(H, Hk):
    """KV head slabs of 8 (two slabs when Hk = 16), 4, 2 and 1 heads: each slab's CTA
    stores its own heads of the new row."""
    case = workloads.decode_case([1, 40, 300, 129, 16], H, Hk, 128, 16, seed=1500 + H + Hk)
    for grid in (0, 3):
        run_step(case, grid_ctas=grid)


def test_strided_new_rows():
    """k_new / v_new as views of a packed [B, 3*Hk*D] projection output (token stride
    3*Hk*D elements)."""
    case = workloads.decode_case([5, 260, 1, 999], 16, 8, 128, 256, seed=1600)
    B, Hk, D = 4, 8, 128
    packed = torch.zeros((B, 3, Hk, D), dtype=torch.bfloat16, device="cuda")
    packed[:, 1] = case.k_new.cuda()
    packed[:, 2] = case.v_new.cuda()
    run_step(case, k_new=packed[:, 1], v_new=packed[:, 2])


def test_workload_qwen3_decode_b256_sampled():
    """The 256-sequence decode step (contexts U{100..2048}, bs 256): every cache byte,
    and 4096 sampled (sequence, head) rows against the oracle."""
    case = workloads.workload(2, poison=False)
    rng = np.random.default_rng(2)
    pairs = np.sort(rng.choice(case.num_seqs * case.num_heads, 4096, replace=False))
    run_step(case, pairs=pairs)


@pytest.mark.parametrize("bs", [16, 256])
def test_workload_prefix_sharing(bs):
    """512 sequences, groups of 64 sharing their first <= 4 blocks: the shared blocks are
    full and never hold a newest position, so the fused store never races a reader."""
    case = workloads.workload(4, block_size=bs, poison=False)
    rng = np.random.default_rng(40 + bs)
    pairs = np.sort(rng.choice(case.num_seqs * case.num_heads, 4096, replace=False))
    run_step(case, pairs=pairs)


def test_long_context_split():
    """8 sequences of 32k..128k tokens: the last tile and its store sit in one CTA of a
    sequence split over many."""
    case = workloads.workload(3, poison=False)
    pairs = np.arange(0, case.num_seqs * case.num_heads, 7)
    run_step(case, pairs=pairs)


def test_slot_not_at_newest_position_is_flagged_and_not_stored():
    """A slot that is not the slot of position context_lens[b]-1, or a token of an empty
    sequence, sets PA_DEV_ERR_SLOT and writes nothing; the decode reads the cache as it
    was."""
    case = workloads.decode_case([40, 70, 0], 16, 8, 128, 16, seed=1700)
    dc = DeviceCase(case)
    before_k = dc.k_cache.clone()
    before_v = dc.v_cache.clone()
    slots = dc.slots.clone()
    slots[0] = int(case.block_tables[1, 0]) * 16 + 3   # a row of sequence 1's context
    slots[2] = 5                                      # token of an empty sequence
    out = fused(dc, slots=slots)
    assert dc.dev_err() & pk.PA_DEV_ERR["slot"]
    s1 = int(case.slot_mapping[1])
    k_rows = dc.k_cache.view(-1, 8 * 128)
    v_rows = dc.v_cache.view(-1, 8 * 128)
    # only sequence 1's token was stored
    exp_k = before_k.view(-1, 8 * 128).clone()
    exp_v = before_v.view(-1, 8 * 128).clone()
    exp_k[s1] = dc.k_new[1].reshape(-1)
    exp_v[s1] = dc.v_new[1].reshape(-1)
    assert torch.equal(k_rows.view(torch.int16), exp_k.view(torch.int16))
    assert torch.equal(v_rows.view(torch.int16), exp_v.view(torch.int16))
    # the output is the decode over that cache
    slot_np = case.slot_mapping.copy()
    slot_np[0] = -1
    ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache, slot_np)
    ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                        case.context_lens)
    assert_close(to_f64(out), ref, "flagged slots")


def test_rejects_bad_arguments():
    case = workloads.workload(1)
    dc = DeviceCase(case)
    out = torch.empty_like(dc.q)
    lib = pk.load_library()
    base = dict(out=out, q=dc.q, kn=dc.k_new, vn=dc.v_new, ks=8 * 128, vs=8 * 128)
    ws = pk.DecodeWorkspace(4, 16, 8, 128, device=dc.q.device)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return lib.pa_decode_step(
            a["out"].data_ptr(), a["q"].data_ptr(), a["kn"], a["vn"], a["ks"], a["vs"],
            dc.k_cache.data_ptr(), dc.v_cache.data_ptr(), dc.slots.data_ptr(),
            dc.bt.data_ptr(), 2, dc.ctx.data_ptr(), 4, 16, 8, 128, 1, 256, 16, 0.0, 0,
            ws.buffer.data_ptr(), ws.nbytes, None, None)

    kn, vn = dc.k_new.data_ptr(), dc.v_new.data_ptr()
    assert call(kn=kn, vn=vn) == 0
    assert call(kn=None, vn=vn) == 1                 # PA_ERR_NULL
    assert call(kn=kn + 2, vn=vn) == 6               # PA_ERR_ALIGN (start)
    assert call(kn=kn, vn=vn, ks=8 * 128 + 4) == 6   # PA_ERR_ALIGN (stride)
    assert call(kn=kn, vn=vn, vs=100) == 2           # PA_ERR_SHAPE (stride below a row)
    torch.cuda.synchronize()


def test_step_on_packed_buffers_equals_separate_tensors():
    """The step's inputs staged in one pinned buffer and moved with one copy
    (DecodeStepBuffers): the fused step on those device views gives the same bits."""
    from paged_kv_cache_107_gb300.step_io import DecodeStepBuffers
    case = workloads.decode_case([5, 260, 1, 999, 0, 77], 16, 8, 128, 256, seed=1800)
    ref_dc = DeviceCase(case)
    ref = fused(ref_dc)
    io = DecodeStepBuffers(6, 16, 8, 128, case.block_tables.shape[1])
    io.host["q"].copy_(case.q)
    io.host["k_new"].copy_(case.k_new)
    io.host["v_new"].copy_(case.v_new)
    io.host["slot_mapping"].copy_(torch.from_numpy(case.slot_mapping))
    io.host["block_tables"].copy_(torch.from_numpy(case.block_tables))
    io.host["context_lens"].copy_(torch.from_numpy(case.context_lens))
    io.upload()
    kc, vc = case.k_cache.cuda(), case.v_cache.cuda()
    out = torch.full_like(ref, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = io.dev
    pk.pa_decode_step(out, d["q"], d["k_new"], d["v_new"], kc, vc, d["slot_mapping"],
                      d["block_tables"], d["context_lens"], dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and ref_dc.dev_err() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), ref_dc.k_cache.view(torch.int16))


@pytest.mark.parametrize("group", [1, 2, 3])
def test_pipelined_steps_equal_sequential_steps(group):
    """Five decode steps (each sequence one token longer per step, fresh q / k_new / v_new)
    through DecodeStepPipeline, with uploads and downloads overlapping the neighbouring
    steps and the steps issued `group` at a time (a partial group at the end), give step by
    step the bits of the same five steps run one after another; the caches end equal."""
    from paged_kv_cache_107_gb300.step_io import DecodeStepPipeline
    lens0 = [5, 260, 1, 999, 0, 77, 300, 16]
    B, H, Hk, D, bs, n_steps = len(lens0), 16, 8, 128, 16, 5
    final = workloads.decode_case([n + n_steps - 1 if n > 0 else 0 for n in lens0], H, Hk, D,
                                  bs, seed=1900, poison=False)
    bt = final.block_tables
    g = torch.Generator().manual_seed(1901)
    steps = []
    for i in range(n_steps):
        lens = np.array([n + i if n > 0 else 0 for n in lens0], np.int32)
        slots = np.full(B, -1, np.int32)
        for b in range(B):
            if lens[b] > 0:
                pos = int(lens[b]) - 1
                slots[b] = int(bt[b, pos // bs]) * bs + pos % bs
        steps.append({"context_lens": torch.from_numpy(lens), "slot_mapping": torch.from_numpy(slots),
                      "block_tables": torch.from_numpy(bt),
                      "q": torch.randn((B, H, D), generator=g).to(torch.bfloat16),
                      "k_new": torch.randn((B, Hk, D), generator=g).to(torch.bfloat16),
                      "v_new": torch.randn((B, Hk, D), generator=g).to(torch.bfloat16)})
    kc_a, vc_a = final.k_cache.cuda(), final.v_cache.cuda()
    kc_b, vc_b = kc_a.clone(), vc_a.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = []
    for st in steps:
        o = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
        d = {k: v.cuda() for k, v in st.items()}
        pk.pa_decode_step(o, d["q"], d["k_new"], d["v_new"], kc_b, vc_b, d["slot_mapping"],
                          d["block_tables"], d["context_lens"], dev_err=err)
        ref.append(o.cpu())
    pipe = DecodeStepPipeline(B, H, Hk, D, bt.shape[1], depth=2 * group, group=group)

    def run(d, out):
        pk.pa_decode_step(out, d["q"], d["k_new"], d["v_new"], kc_a, vc_a, d["slot_mapping"],
                          d["block_tables"], d["context_lens"], dev_err=err)

    got = []
    for i, st in enumerate(steps):
        h = pipe.inputs(i)
        for name, v in st.items():
            h[name].copy_(v)
        pipe.submit(i, run)
        if i >= 1:
            got.append(pipe.output(i - 1).clone())
    got.append(pipe.output(n_steps - 1).clone())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for i, (a, r) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.int16), r.view(torch.int16)), f"step {i}"
    assert torch.equal(kc_a.view(torch.int16), kc_b.view(torch.int16))
    assert torch.equal(vc_a.view(torch.int16), vc_b.view(torch.int16))


def test_context_lens_written_by_the_kernel_just_before():
    """The step reads context_lens before it waits for the kernel launched ahead of it on
    the stream. An ordinary kernel lets its dependents start only when it completes, so
    context_lens written by such a kernel right before the step must be the ones used:
    the lengths start out wrong (all 1) and an elementwise kernel on the same stream writes
    the right ones just before each launch."""
    case = workloads.decode_case([300, 17, 1024, 65, 2000, 3], 16, 8, 128, 16, seed=1950,
                                 poison=False)
    ok, ov = oracle_after_store(case)
    ref = oracle.decode(case.q, from_bits(ok), from_bits(ov), case.block_tables,
                        case.context_lens)
    right = torch.from_numpy(case.context_lens).cuda()
    for rep in range(4):
        dc = DeviceCase(case)
        dc.ctx.fill_(1)
        torch.cuda.synchronize()
        torch.add(right, 0, out=dc.ctx)  # a kernel on the stream, immediately before
        out = fused(dc)
        assert dc.dev_err() == 0
        assert_close(to_f64(out), ref, f"lengths written just before, launch {rep}")


@pytest.mark.parametrize("H,Hk", [(16, 8), (64, 8), (28, 4)])
def test_many_short_sequences(H, Hk):
    """4096 sequences of 1..64 tokens (block_size 16): dozens of sequences per CTA, most of
    them whole, the rest cut at CTA boundaries; the fused step against the oracle on 4096
    sampled rows, and every cache byte."""
    rng = np.random.default_rng(1960 + H + Hk)
    lens = rng.integers(1, 65, size=4096)
    case = workloads.decode_case(lens.tolist(), H, Hk, 128, 16, seed=1961 + H, poison=True)
    pairs = np.sort(rng.choice(case.num_seqs * case.num_heads, 4096, replace=False))
    run_step(case, pairs=pairs)
