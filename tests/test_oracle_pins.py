"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these tests retypes the oracle's formula: each checks a closed form, an
invariant, a special case that reduces to a library routine (scipy's softmax over a
contiguous layout), a worked example printed on the pages, or a brute-force loop on tiny
inputs. A plausible slip in the oracle (dropped max subtraction, 1/D instead of
1/sqrt(D), h % Hk instead of h // (H/Hk), context_len - 1, an off-by-one block index, a
wrong causal offset, q and v swapped) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_kv_cache_107_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.float().double().numpy()


def contiguous_case(lens, H, Hk, D, bs, seed, q=None, k=None, v=None):
    """Caches laid out contiguously: sequence b owns physical blocks in order, so the
    block table row is a plain range. Returns (q, kc, vc, bt, lens, dense_k, dense_v)."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    nblk = [-(-n // bs) for n in lens]
    maxb = max(max(nblk), 1)
    nb = max(sum(nblk), 1)
    kc = np.full((nb, bs, Hk, D), np.nan, np.float32)
    vc = np.full((nb, bs, Hk, D), np.nan, np.float32)
    bt = np.full((B, maxb), -1, np.int32)
    dense_k, dense_v = [], []
    nxt = 0
    for b, n in enumerate(lens):
        kk = rng.standard_normal((n, Hk, D)).astype(np.float32) if k is None else k[b]
        vv = rng.standard_normal((n, Hk, D)).astype(np.float32) if v is None else v[b]
        kk = f64(bf16(kk)).astype(np.float32)
        vv = f64(bf16(vv)).astype(np.float32)
        dense_k.append(kk.astype(np.float64))
        dense_v.append(vv.astype(np.float64))
        for j in range(nblk[b]):
            bt[b, j] = nxt
            lo, hi = j * bs, min(n, (j + 1) * bs)
            kc[nxt, : hi - lo] = kk[lo:hi]
            vc[nxt, : hi - lo] = vv[lo:hi]
            nxt += 1
    if q is None:
        q = rng.standard_normal((B, H, D)).astype(np.float32)
    return bf16(q), bf16(kc), bf16(vc), bt, np.asarray(lens, np.int32), dense_k, dense_v


# ------------------------------------------------------------------------------ store


def test_store_equals_numpy_index_assignment():
    """Closed form of the store ("nano-vllm解读", KVCache的写入): row slot[i] of the
    flattened cache becomes token i's row; numpy fancy assignment is the reference."""
    rng = np.random.default_rng(1)
    nb, bs, hk, d = 6, 4, 2, 8
    kc = bf16(rng.standard_normal((nb, bs, hk, d)))
    vc = bf16(rng.standard_normal((nb, bs, hk, d)))
    k = bf16(rng.standard_normal((5, hk, d)))
    v = bf16(rng.standard_normal((5, hk, d)))
    slots = np.array([3, -1, 17, 0, 23], np.int32)
    ok, ov = oracle.store_kvcache(k, v, kc, vc, slots)
    ek = kc.view(torch.int16).numpy().view(np.uint16).reshape(nb * bs, hk * d).copy()
    ev = vc.view(torch.int16).numpy().view(np.uint16).reshape(nb * bs, hk * d).copy()
    keep = slots != -1
    ek[slots[keep]] = k.view(torch.int16).numpy().view(np.uint16).reshape(5, -1)[keep]
    ev[slots[keep]] = v.view(torch.int16).numpy().view(np.uint16).reshape(5, -1)[keep]
    assert np.array_equal(ok.reshape(nb * bs, -1), ek)
    assert np.array_equal(ov.reshape(nb * bs, -1), ev)


def test_store_slot_minus_one_leaves_cache_byte_identical():
    """Slot -1 is a padding row and writes nothing ("3.6 ModelRunner…", section 5)."""
    rng = np.random.default_rng(2)
    kc = bf16(rng.standard_normal((3, 4, 1, 8)))
    vc = bf16(rng.standard_normal((3, 4, 1, 8)))
    k = bf16(rng.standard_normal((4, 1, 8)))
    ok, ov = oracle.store_kvcache(k, k, kc, vc, np.full(4, -1, np.int32))
    assert np.array_equal(ok, kc.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(ov, vc.view(torch.int16).numpy().view(np.uint16))


def test_store_rejects_out_of_range_slot():
    kc = bf16(np.zeros((2, 2, 1, 8)))
    k = bf16(np.ones((1, 1, 8)))
    with pytest.raises(ValueError):
        oracle.store_kvcache(k, k, kc, kc, np.array([4], np.int32))


# --------------------------------------------------------------- layout worked example


def test_page_layout_example_slots_and_rows():
    """Worked mapping printed on the nano-vllm overview page (内存布局可视化, 逻辑映射):
    with 256-token blocks, sequence A's tokens 0..255 live in Block0 and 256..511 in
    Block1, and sequence B's tokens 0..99 in Block2 (partly used)."""
    ex = json.load(open(os.path.join(GOLDEN, "layout_example.json")))
    bs = ex["block_size"]
    for seq in ex["sequences"]:
        table = np.array(seq["block_table"], np.int32)
        for pos, slot in seq["slots"]:
            assert oracle.slot_of(table, pos, bs) == slot
    # The attention oracle must read exactly those rows: put 1 in every row the example
    # maps and NaN everywhere else; with q = 0 the output is the mean of the rows read,
    # i.e. 1 up to the rounding of 1/n, and any stray row turns it into NaN.
    nb, hk, d = 4, 1, 8
    kc = np.full((nb, bs, hk, d), np.nan, np.float32)
    vc = np.full((nb, bs, hk, d), np.nan, np.float32)
    seqs = ex["sequences"]
    B = len(seqs)
    bt = np.full((B, 2), -1, np.int32)
    lens = np.zeros(B, np.int32)
    for b, seq in enumerate(seqs):
        lens[b] = seq["num_tokens"]
        for j, blk in enumerate(seq["block_table"]):
            bt[b, j] = blk
        for pos in range(seq["num_tokens"]):
            blk = seq["block_table"][pos // bs]
            kc[blk, pos % bs] = 0.0
            vc[blk, pos % bs] = 1.0
    out = oracle.decode(bf16(np.zeros((B, 1, d))), bf16(kc), bf16(vc), bt, lens)
    np.testing.assert_allclose(out, np.ones((B, 1, d)), rtol=0, atol=1e-14)


def test_workload_slot_mapping_matches_page_formula():
    """The generator's slot_mapping (host prepare step) against the oracle's own slot of
    position len-1 ("3.6 ModelRunner…", section 2, prepare_decode)."""
    case = workloads.decode_case([1, 5, 16, 17, 40], 4, 2, 8, 16, seed=7)
    for b in range(case.num_seqs):
        n = int(case.context_lens[b])
        assert case.slot_mapping[b] == oracle.slot_of(case.block_tables[b], n - 1, 16)
    pc = workloads.prefill_case([0, 3, 16], [2, 5, 1], 4, 2, 8, 8, seed=8)
    r = 0
    for s in range(3):
        c, n = int(pc.cu_seqlens_k[s + 1] - pc.cu_seqlens_k[s]) - int(
            pc.cu_seqlens_q[s + 1] - pc.cu_seqlens_q[s]), int(
            pc.cu_seqlens_q[s + 1] - pc.cu_seqlens_q[s])
        for pos in range(c, c + n):
            assert pc.slot_mapping[r] == oracle.slot_of(pc.block_tables[s], pos, 8)
            r += 1


# ------------------------------------------------------------------- decode closed forms


@pytest.mark.parametrize("H,Hk", [(4, 4), (4, 2), (8, 2)])
def test_decode_single_key_returns_its_value(H, Hk):
    """Softmax over one key is 1, so o = v exactly (context_len == 1)."""
    q, kc, vc, bt, lens, dk, dv = contiguous_case([1, 1], H, Hk, 16, 4, seed=3)
    out = oracle.decode(q, kc, vc, bt, lens)
    g = H // Hk
    for b in range(2):
        for h in range(H):
            assert np.array_equal(out[b, h], dv[b][0, h // g])


def test_decode_zero_query_is_mean_of_values():
    """q = 0 gives equal scores, so o is the plain mean of the context's values."""
    lens = [1, 7, 33]
    q0 = np.zeros((3, 4, 16), np.float32)
    q, kc, vc, bt, lens, dk, dv = contiguous_case(lens, 4, 2, 16, 8, seed=4, q=q0)
    out = oracle.decode(q, kc, vc, bt, lens)
    for b in range(3):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], dv[b][:, h // 2].mean(axis=0), rtol=0,
                                       atol=1e-13)


def test_decode_gqa_head_mapping_with_constant_values():
    """Every KV head j carries its own constant value c_j; query head h must return
    c_{h // (H/Hk)} whatever q and k are (GQA contiguous groups)."""
    H, Hk, D = 8, 4, 8
    n = 10
    v = [np.broadcast_to(np.arange(1, Hk + 1, dtype=np.float32)[None, :, None],
                         (n, Hk, D)).copy()]
    q, kc, vc, bt, lens, dk, dv = contiguous_case([n], H, Hk, D, 4, seed=5, v=v)
    out = oracle.decode(q, kc, vc, bt, lens)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], np.full(D, 1 + h // (H // Hk)), atol=1e-13)


def test_decode_two_keys_closed_form_scale():
    """Two keys, q = a*e0, k1 = e0, k2 = 0, v1 = e1, v2 = e2. The weights are the
    logistic function of a*scale with scale = 1/sqrt(D) ("nano-vllm解读", Nano-vllm中的使用:
    softmax_scale = 1/sqrt(HEAD_DIM))."""
    D = 64
    a = 3.0
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = a
    k = np.zeros((2, 1, D), np.float32)
    k[0, 0, 0] = 1.0
    v = np.zeros((2, 1, D), np.float32)
    v[0, 0, 1] = 1.0
    v[1, 0, 2] = 1.0
    qq, kc, vc, bt, lens, _, _ = contiguous_case([2], 1, 1, D, 4, seed=0, q=q, k=[k], v=[v])
    out = oracle.decode(qq, kc, vc, bt, lens)
    s = a / math.sqrt(D)
    w1 = 1.0 / (1.0 + math.exp(-s))
    assert abs(out[0, 0, 1] - w1) < 1e-14
    assert abs(out[0, 0, 2] - (1.0 - w1)) < 1e-14
    assert out[0, 0, 0] == 0.0


def test_decode_dominant_key_and_no_overflow():
    """One key with a score ~1000 above the rest: o equals its value to machine precision.
    Without the max subtraction exp() would overflow to inf/NaN."""
    D = 32
    n = 9
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, :] = 16.0
    k = np.zeros((n, 1, D), np.float32)
    k[4, 0, :] = 16.0  # score = 16*16*32/sqrt(32) ~ 1448
    rng = np.random.default_rng(6)
    v = rng.standard_normal((n, 1, D)).astype(np.float32)
    qq, kc, vc, bt, lens, _, dv = contiguous_case([n], 1, 1, D, 4, seed=0, q=q, k=[k], v=[v])
    out = oracle.decode(qq, kc, vc, bt, lens)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], dv[0][4, 0], rtol=0, atol=1e-300)


def test_decode_contiguous_matches_scipy_softmax():
    """Special case that reduces to a library routine: with the cache laid out
    contiguously (block table = a plain range), the oracle equals
    scipy.special.softmax(scale * K q) @ V over the dense K/V of each sequence."""
    lens = [1, 5, 16, 17, 64]
    H, Hk, D = 8, 2, 32
    q, kc, vc, bt, lens_a, dk, dv = contiguous_case(lens, H, Hk, D, 16, seed=9)
    out = oracle.decode(q, kc, vc, bt, lens_a)
    qd = f64(q)
    for b, n in enumerate(lens):
        for h in range(H):
            j = h // (H // Hk)
            p = scipy.special.softmax(dk[b][:, j] @ qd[b, h] / math.sqrt(D))
            np.testing.assert_allclose(out[b, h], p @ dv[b][:, j], rtol=1e-12, atol=1e-13)


def test_decode_lse_closed_forms():
    """LSE (natural log): q = 0 gives log(n); a single key gives scale*q.k."""
    lens = [1, 12]
    q, kc, vc, bt, lens_a, dk, dv = contiguous_case(lens, 2, 1, 16, 8, seed=10)
    _, lse = oracle.decode(q, kc, vc, bt, lens_a, return_lse=True)
    qd = f64(q)
    np.testing.assert_allclose(lse[0], dk[0][0, 0] @ qd[0].T / 4.0, rtol=1e-13)
    q0 = bf16(np.zeros((2, 2, 16)))
    _, lse0 = oracle.decode(q0, kc, vc, bt, lens_a, return_lse=True)
    np.testing.assert_allclose(lse0[1], math.log(12), rtol=1e-14)


def test_decode_zero_context_gives_zero_row():
    """A CUDA-graph padding row (context_len 0) reads nothing and returns zeros."""
    q, kc, vc, bt, lens, _, _ = contiguous_case([0, 3], 2, 1, 8, 4, seed=11)
    out = oracle.decode(q, kc, vc, bt, lens)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    assert np.all(np.isfinite(out[1]))


# ---------------------------------------------------------------------- invariants


def _permute_blocks(case, rng):
    """Move every physical block to a new random id and rewrite the tables."""
    nb = case.num_blocks
    perm = rng.permutation(nb)  # old id -> new id
    kc = torch.empty_like(case.k_cache)
    vc = torch.empty_like(case.v_cache)
    kc[torch.from_numpy(perm)] = case.k_cache
    vc[torch.from_numpy(perm)] = case.v_cache
    bt = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    return kc, vc, bt.astype(np.int32)


def test_decode_invariant_under_physical_block_permutation():
    """Paging only relocates memory ("nano-vllm解读", PageAttention原理): permuting the
    physical block ids, with the data moved along, leaves the result bitwise unchanged."""
    case = workloads.decode_case([1, 17, 64, 100, 255], 8, 2, 32, 16, seed=12)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens)
    kc, vc, bt = _permute_blocks(case, np.random.default_rng(13))
    got = oracle.decode(case.q, kc, vc, bt, case.context_lens)
    assert np.array_equal(ref, got)


def test_decode_ignores_unreferenced_rows():
    """Rows past the context (tails of last blocks, unused blocks) never matter: the
    generator poisons them with NaN and the output must stay finite; overwriting them with
    +-1e30 changes nothing."""
    case = workloads.decode_case([3, 16, 17, 40], 4, 2, 16, 16, seed=14, num_blocks=12)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens)
    assert np.all(np.isfinite(ref))
    kc = case.k_cache.clone()
    vc = case.v_cache.clone()
    kc[torch.isnan(kc.float())] = 1e30
    vc[torch.isnan(vc.float())] = -1e30
    got = oracle.decode(case.q, kc, vc, case.block_tables, case.context_lens)
    assert np.array_equal(ref, got)


def test_decode_shared_prefix_blocks_read_identically():
    """Sequences that share physical prefix blocks ("nano-vllm解读", 前缀缓存) and have
    the same q and length give identical rows, equal to private copies of the blocks."""
    case = workloads.decode_case([40, 40, 40], 4, 2, 16, 8, seed=15, share_group=3,
                                 share_blocks=4)
    assert case.shared_blocks == 4
    q = case.q.clone()
    q[1] = q[0]
    q[2] = q[0]
    out = oracle.decode(q, case.k_cache, case.v_cache, case.block_tables, case.context_lens)
    # the three sequences differ only in their private tail blocks, so make those equal
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    for j in range(4, 5):
        for b in (1, 2):
            kc[int(case.block_tables[b, j])] = kc[int(case.block_tables[0, j])]
            vc[int(case.block_tables[b, j])] = vc[int(case.block_tables[0, j])]
    out = oracle.decode(q, kc, vc, case.block_tables, case.context_lens)
    assert np.array_equal(out[0], out[1]) and np.array_equal(out[0], out[2])
    # private copies of the shared blocks give the same rows
    bt2 = case.block_tables.copy()
    spare = [i for i in range(case.num_blocks) if i not in set(case.block_tables.ravel())]
    kc2, vc2 = kc.clone(), vc.clone()
    for j in range(4):
        kc2[spare[j]] = kc[int(bt2[1, j])]
        vc2[spare[j]] = vc[int(bt2[1, j])]
        bt2[1, j] = spare[j]
    out2 = oracle.decode(q, kc2, vc2, bt2, case.context_lens)
    assert np.array_equal(out2, out)


def test_decode_linearity_in_values():
    """o is linear in V: doubling V doubles o exactly; adding 1 to every value adds 1."""
    rng = np.random.default_rng(16)
    n = 13
    v = [rng.integers(-2, 3, size=(n, 1, 16)).astype(np.float32)]
    k = [rng.standard_normal((n, 1, 16)).astype(np.float32)]
    q = rng.standard_normal((1, 1, 16)).astype(np.float32)
    base = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 0, q=q, k=k, v=v)[:5])
    twice = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 0, q=q, k=k, v=[2 * v[0]])[:5])
    plus1 = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 0, q=q, k=k, v=[v[0] + 1])[:5])
    np.testing.assert_allclose(twice, 2 * base, rtol=0, atol=1e-14)
    np.testing.assert_allclose(plus1, base + 1, rtol=0, atol=1e-14)


def test_decode_key_shift_invariance():
    """Adding the same vector u to every key shifts every score by scale*q.u, which the
    softmax cancels."""
    rng = np.random.default_rng(17)
    n = 11
    k = [rng.integers(-3, 4, size=(n, 1, 16)).astype(np.float32)]
    q = rng.integers(-2, 3, size=(1, 1, 16)).astype(np.float32)
    u = np.zeros(16, np.float32)
    u[3] = 2.0
    a = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 18, q=q, k=k)[:5])
    b = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 18, q=q, k=[k[0] + u])[:5])
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_decode_output_is_convex_combination():
    """Each output component lies between the min and max of that component over the
    context's values."""
    q, kc, vc, bt, lens, dk, dv = contiguous_case([5, 30], 4, 2, 16, 8, seed=19)
    out = oracle.decode(q, kc, vc, bt, lens)
    for b in range(2):
        for h in range(4):
            vv = dv[b][:, h // 2]
            assert np.all(out[b, h] >= vv.min(axis=0) - 1e-14)
            assert np.all(out[b, h] <= vv.max(axis=0) + 1e-14)


def brute_decode(q, kc, vc, bt, lens, bs):
    """Pure-Python triple loop on tiny shapes."""
    qd, kd, vd = f64(q), f64(kc), f64(vc)
    B, H, D = qd.shape
    Hk = kd.shape[2]
    out = [[[0.0] * D for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            j = h // (H // Hk)
            scores = []
            for t in range(int(lens[b])):
                blk = int(bt[b][t // bs])
                s = 0.0
                for d in range(D):
                    s += qd[b][h][d] * kd[blk][t % bs][j][d]
                scores.append(s / math.sqrt(D))
            if not scores:
                continue
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            tot = sum(e)
            for t in range(len(e)):
                blk = int(bt[b][t // bs])
                for d in range(D):
                    out[b][h][d] += e[t] / tot * vd[blk][t % bs][j][d]
    return np.array(out)


@pytest.mark.parametrize("bs", [4, 16])
def test_decode_brute_force_tiny(bs):
    case = workloads.decode_case([1, 9, 40], 4, 2, 8, bs, seed=20 + bs)
    # the store first, as the step orders it
    kc, vc = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    kct = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vct = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    got = oracle.decode(case.q, kct, vct, case.block_tables, case.context_lens)
    want = brute_decode(case.q, kct, vct, case.block_tables, case.context_lens, bs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_decode_subset_rows_match_full():
    case = workloads.decode_case([5, 40, 7], 4, 2, 16, 8, seed=23)
    full = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                         case.context_lens)
    pairs = np.array([11, 0, 5], np.int64)
    sub = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                        case.context_lens, pairs=pairs)
    assert np.array_equal(sub, full.reshape(-1, 16)[pairs])


# --------------------------------------------------------------------------- prefill


def _stored(case):
    kc, vc = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    return (torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16),
            torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16))


def test_prefill_rows_equal_decode_at_their_position():
    """Causal: new token i of sequence s (absolute position c_s + i) sees keys
    0..c_s+i ("3.6 ModelRunner…", section 2), i.e. exactly a decode with context
    c_s + i + 1 over the same table."""
    case = workloads.prefill_case([0, 5, 16, 3], [4, 1, 9, 20], 4, 2, 16, 8, seed=24)
    kc, vc = _stored(case)
    out = oracle.prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, causal=True)
    for s in range(case.num_seqs):
        q0, q1 = int(case.cu_seqlens_q[s]), int(case.cu_seqlens_q[s + 1])
        c = int(case.cu_seqlens_k[s + 1] - case.cu_seqlens_k[s]) - (q1 - q0)
        for i in range(q1 - q0):
            dec = oracle.decode(case.q[q0 + i:q0 + i + 1], kc, vc,
                                case.block_tables[s:s + 1],
                                np.array([c + i + 1], np.int32))
            assert np.array_equal(out[q0 + i], dec[0])


def test_prefill_first_row_without_cache_is_its_own_value():
    """With no cached prefix the first new token sees only itself: o = v_0."""
    case = workloads.prefill_case([0], [6], 4, 2, 16, 4, seed=25)
    kc, vc = _stored(case)
    out = oracle.prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k)
    v0 = f64(case.v_new)[0]
    for h in range(4):
        assert np.array_equal(out[0, h], v0[h // 2])


def test_prefill_noncausal_rows_see_all_keys():
    case = workloads.prefill_case([3, 0], [5, 7], 4, 2, 16, 4, seed=26, causal=False)
    kc, vc = _stored(case)
    out = oracle.prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, causal=False)
    for s in range(2):
        q0, q1 = int(case.cu_seqlens_q[s]), int(case.cu_seqlens_q[s + 1])
        k_s = int(case.cu_seqlens_k[s + 1] - case.cu_seqlens_k[s])
        dec = oracle.decode(case.q[q0:q1], kc, vc,
                            np.repeat(case.block_tables[s:s + 1], q1 - q0, 0),
                            np.full(q1 - q0, k_s, np.int32))
        assert np.array_equal(out[q0:q1], dec)


def test_prefill_noncausal_key_permutation_invariance():
    """Without a mask, attention does not depend on the order of the keys: shuffling the
    logical positions of the K/V rows (same rows, new order) leaves o unchanged."""
    rng = np.random.default_rng(27)
    n = 12
    k = rng.standard_normal((n, 1, 16)).astype(np.float32)
    v = rng.standard_normal((n, 1, 16)).astype(np.float32)
    q = rng.standard_normal((1, 1, 16)).astype(np.float32)
    perm = rng.permutation(n)
    a = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 0, q=q, k=[k], v=[v])[:5])
    b = oracle.decode(*contiguous_case([n], 1, 1, 16, 4, 0, q=q, k=[k[perm]], v=[v[perm]])[:5])
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def brute_prefill(q, kc, vc, bt, cu_q, cu_k, bs, causal):
    qd, kd, vd = f64(q), f64(kc), f64(vc)
    T, H, D = qd.shape
    Hk = kd.shape[2]
    out = np.zeros((T, H, D))
    for s in range(len(cu_q) - 1):
        n = int(cu_q[s + 1] - cu_q[s])
        k_s = int(cu_k[s + 1] - cu_k[s])
        c = k_s - n
        for i in range(n):
            for h in range(H):
                j = h // (H // Hk)
                last = c + i if causal else k_s - 1
                sc = []
                for t in range(last + 1):
                    blk = int(bt[s][t // bs])
                    sc.append(sum(qd[cu_q[s] + i][h][d] * kd[blk][t % bs][j][d]
                                  for d in range(D)) / math.sqrt(D))
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                z = sum(e)
                for t in range(last + 1):
                    blk = int(bt[s][t // bs])
                    out[cu_q[s] + i][h] += e[t] / z * vd[blk][t % bs][j]
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_brute_force_tiny(causal):
    case = workloads.prefill_case([0, 7, 4], [3, 2, 6], 4, 2, 8, 4, seed=28, causal=causal)
    kc, vc = _stored(case)
    got = oracle.prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, causal=causal)
    want = brute_prefill(case.q, kc, vc, case.block_tables, case.cu_seqlens_q,
                         case.cu_seqlens_k, 4, causal)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------- golden regressions


@pytest.mark.parametrize("name", ["decode_small.json", "prefill_small.json"])
def test_golden_regression(name):
    """Stored values written by tests/golden/make_golden.py (oracle only). They anchor the
    oracle against silent change; the pins above are what tie it to the pages."""
    g = json.load(open(os.path.join(GOLDEN, name)))
    case = g["inputs"]
    q = torch.tensor(case["q_bits"], dtype=torch.int16).view(torch.bfloat16)
    kc = torch.tensor(case["k_cache_bits"], dtype=torch.int16).view(torch.bfloat16)
    vc = torch.tensor(case["v_cache_bits"], dtype=torch.int16).view(torch.bfloat16)
    bt = np.array(case["block_tables"], np.int32)
    if g["kind"] == "decode":
        out = oracle.decode(q, kc, vc, bt, np.array(case["context_lens"], np.int32))
    else:
        out = oracle.prefill(q, kc, vc, bt, np.array(case["cu_seqlens_q"], np.int32),
                             np.array(case["cu_seqlens_k"], np.int32), causal=case["causal"])
    np.testing.assert_allclose(out, np.array(g["expected"]), rtol=1e-13, atol=1e-14)
