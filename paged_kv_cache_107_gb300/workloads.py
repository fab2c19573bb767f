"""Seeded synthetic workloads for paged-KV attention.

This module only draws inputs. It holds none of the attention arithmetic and imports
neither the CUDA library nor the oracle, so the tests, the benchmark and the oracle can
all take their inputs from here. It mirrors the host-side preparation step of the engine
the pages describe ("3.6 ModelRunner、CUDA Graph 与性能基准", section 2, prepare_prefill /
prepare_decode): block tables right-padded with -1, context_lens = len(seq) including the
just-stored token, slot_mapping = physical block * block_size + offset for every new token,
cu_seqlens_q / cu_seqlens_k as cumulative lengths.

Values: fp32 N(0, 1) from numpy's default_rng, rounded to bf16 (round to nearest even) by
torch. Physical block ids: rng.permutation(num_blocks) taken in order, so logical blocks
land on random physical blocks. Cache rows that no sequence references (unused blocks and
the tail of each sequence's last block) are filled with NaN when ``poison`` is set, so any
read of them shows up in the output.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

SEED_BASE = 107000


@dataclasses.dataclass
class PagedCase:
    """One layer's worth of paged-attention inputs (host tensors)."""

    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    block_tables: np.ndarray          # int32 [B, max_blocks], -1 padded
    context_lens: np.ndarray          # int32 [B] total keys after the store
    q: torch.Tensor                   # bf16 [B, H, D] (decode) or [sum n, H, D] (prefill)
    k_new: torch.Tensor               # bf16 [N, Hk, D]
    v_new: torch.Tensor               # bf16 [N, Hk, D]
    slot_mapping: np.ndarray          # int32 [N], -1 = padding row
    k_cache: torch.Tensor             # bf16 [nb, bs, Hk, D], state BEFORE the store
    v_cache: torch.Tensor
    cu_seqlens_q: Optional[np.ndarray] = None  # int32 [S+1] (prefill)
    cu_seqlens_k: Optional[np.ndarray] = None  # int32 [S+1] (prefill)
    causal: bool = True
    seed: int = 0
    shared_blocks: int = 0            # physical blocks referenced by more than one sequence

    @property
    def num_seqs(self) -> int:
        return int(self.block_tables.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def is_prefill(self) -> bool:
        return self.cu_seqlens_q is not None

    @property
    def max_seqlen_q(self) -> int:
        if not self.is_prefill:
            return 1
        return int(np.max(np.diff(self.cu_seqlens_q))) if self.num_seqs else 0

    @property
    def max_seqlen_k(self) -> int:
        if not self.is_prefill:
            return int(self.context_lens.max()) if self.num_seqs else 0
        return int(np.max(np.diff(self.cu_seqlens_k))) if self.num_seqs else 0

    def total_context(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    def referenced_blocks(self) -> np.ndarray:
        """Distinct physical block ids read by the attention call."""
        ids = []
        for b in range(self.num_seqs):
            nblk = -(-int(self.context_lens[b]) // self.block_size)
            ids.append(self.block_tables[b, :nblk])
        if not ids:
            return np.zeros(0, np.int64)
        return np.unique(np.concatenate(ids).astype(np.int64))


def _bf16(x: np.ndarray, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """fp32 values rounded (nearest even) to the 16-bit element type (bf16 or fp16)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


def _fill_blocks(cache: torch.Tensor, ids: np.ndarray, rng: np.random.Generator,
                 chunk: int = 256) -> None:
    """Fill whole physical blocks `ids` (in that order) with N(0,1) values of the cache's
    element type."""
    _, bs, hk, d = cache.shape
    for s in range(0, len(ids), chunk):
        part = ids[s:s + chunk]
        vals = rng.standard_normal((len(part), bs, hk, d), dtype=np.float32)
        cache[torch.from_numpy(part.astype(np.int64))] = _bf16(vals, cache.dtype)


def _empty_cache(nb: int, bs: int, hk: int, d: int, poison: bool,
                 dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    fill = float("nan") if poison else 0.0
    return torch.full((nb, bs, hk, d), fill, dtype=dtype)


def _poison_tails(cache: torch.Tensor, tables: np.ndarray, lens: np.ndarray, bs: int,
                  value: float) -> None:
    """Overwrite positions len..end of each sequence's last block."""
    for b in range(tables.shape[0]):
        n = int(lens[b])
        if n % bs == 0:
            continue
        blk = int(tables[b, n // bs])
        cache[blk, n % bs:] = value


def _assign_blocks(lens: np.ndarray, bs: int, nb: int, rng: np.random.Generator,
                   max_blocks: Optional[int] = None, share_group: int = 0,
                   share_blocks: int = 0):
    """Block tables for sequences of the given lengths, ids drawn from a permutation.

    With share_group > 0, consecutive groups of `share_group` sequences share their first
    blocks: sequence b shares logical block j when j < min(share_blocks, (len_b - 1) // bs),
    i.e. only full blocks that do not hold the newest token (so a store never writes a
    shared block).
    """
    B = len(lens)
    nblk = [-(-int(n) // bs) for n in lens]
    maxb = max(nblk) if (max_blocks is None and B) else (max_blocks or 1)
    maxb = max(maxb, 1)
    tables = np.full((B, maxb), -1, np.int32)
    perm = rng.permutation(nb)
    nxt = 0
    shared_ids = {}
    for b in range(B):
        share_here = 0
        if share_group > 0:
            share_here = min(share_blocks, max(int(lens[b]) - 1, 0) // bs)
        for j in range(nblk[b]):
            if j < share_here:
                key = (b // share_group, j)
                if key not in shared_ids:
                    shared_ids[key] = int(perm[nxt])
                    nxt += 1
                tables[b, j] = shared_ids[key]
            else:
                tables[b, j] = int(perm[nxt])
                nxt += 1
        if nxt > nb:
            raise ValueError("block pool too small for the drawn lengths")
    return tables, len(shared_ids)


def decode_case(context_lens: Sequence[int], num_heads: int = 16, num_kv_heads: int = 8,
                head_dim: int = 128, block_size: int = 256, num_blocks: Optional[int] = None,
                seed: int = SEED_BASE, poison: bool = True, skip_slots: Sequence[int] = (),
                max_blocks: Optional[int] = None, share_group: int = 0,
                share_blocks: int = 0, name: str = "decode",
                dtype: torch.dtype = torch.bfloat16) -> PagedCase:
    """A decode step: each sequence b stores one new token at position len_b - 1 and then
    attends over positions 0..len_b-1. Sequences with len_b == 0 are CUDA-graph padding
    rows: slot -1 and no blocks. Sequences listed in skip_slots get slot -1 too (their
    position len_b - 1 keeps the value that was already in the cache)."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(context_lens, dtype=np.int32)
    B = len(lens)
    bs = block_size
    need = sum(-(-int(n) // bs) for n in lens)
    nb = num_blocks if num_blocks is not None else max(need + 4, 8)
    tables, nshared = _assign_blocks(lens, bs, nb, rng, max_blocks, share_group, share_blocks)
    k_cache = _empty_cache(nb, bs, num_kv_heads, head_dim, poison, dtype)
    v_cache = _empty_cache(nb, bs, num_kv_heads, head_dim, poison, dtype)
    used = np.unique(tables[tables >= 0]).astype(np.int64) if B else np.zeros(0, np.int64)
    _fill_blocks(k_cache, used, rng)
    _fill_blocks(v_cache, used, rng)
    if poison:
        _poison_tails(k_cache, tables, lens, bs, float("nan"))
        _poison_tails(v_cache, tables, lens, bs, float("nan"))
    q = _bf16(rng.standard_normal((B, num_heads, head_dim), dtype=np.float32), dtype)
    k_new = _bf16(rng.standard_normal((B, num_kv_heads, head_dim), dtype=np.float32), dtype)
    v_new = _bf16(rng.standard_normal((B, num_kv_heads, head_dim), dtype=np.float32), dtype)
    slots = np.full(B, -1, np.int32)
    skip = set(int(s) for s in skip_slots)
    for b in range(B):
        n = int(lens[b])
        if n == 0 or b in skip:
            continue
        pos = n - 1
        slots[b] = int(tables[b, pos // bs]) * bs + pos % bs
    return PagedCase(name=name, num_heads=num_heads, num_kv_heads=num_kv_heads,
                     head_dim=head_dim, block_size=bs, num_blocks=nb, block_tables=tables,
                     context_lens=lens, q=q, k_new=k_new, v_new=v_new, slot_mapping=slots,
                     k_cache=k_cache, v_cache=v_cache, seed=seed, shared_blocks=nshared)


def prefill_case(cached: Sequence[int], new: Sequence[int], num_heads: int = 16,
                 num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 256,
                 num_blocks: Optional[int] = None, seed: int = SEED_BASE, poison: bool = True,
                 causal: bool = True, name: str = "prefill",
                 dtype: torch.dtype = torch.bfloat16) -> PagedCase:
    """A chunked-prefill step: sequence s has cached[s] tokens already in the cache (a
    prefix hit or an earlier chunk) and new[s] new tokens that are stored and then attend
    causally over positions 0..cached[s]+i."""
    rng = np.random.default_rng(seed)
    c = np.asarray(cached, dtype=np.int64)
    n = np.asarray(new, dtype=np.int64)
    S = len(c)
    bs = block_size
    total = (c + n).astype(np.int32)
    need = sum(-(-int(t) // bs) for t in total)
    nb = num_blocks if num_blocks is not None else max(need + 4, 8)
    tables, _ = _assign_blocks(total, bs, nb, rng)
    k_cache = _empty_cache(nb, bs, num_kv_heads, head_dim, poison, dtype)
    v_cache = _empty_cache(nb, bs, num_kv_heads, head_dim, poison, dtype)
    used = np.unique(tables[tables >= 0]).astype(np.int64) if S else np.zeros(0, np.int64)
    _fill_blocks(k_cache, used, rng)
    _fill_blocks(v_cache, used, rng)
    if poison:
        # the new tokens' rows are not in the cache yet: poison them, the store fills them
        for s in range(S):
            for pos in range(int(c[s]), int(total[s])):
                k_cache[int(tables[s, pos // bs]), pos % bs] = float("nan")
                v_cache[int(tables[s, pos // bs]), pos % bs] = float("nan")
        _poison_tails(k_cache, tables, total, bs, float("nan"))
        _poison_tails(v_cache, tables, total, bs, float("nan"))
    nq = int(n.sum())
    q = _bf16(rng.standard_normal((nq, num_heads, head_dim), dtype=np.float32), dtype)
    k_new = _bf16(rng.standard_normal((nq, num_kv_heads, head_dim), dtype=np.float32), dtype)
    v_new = _bf16(rng.standard_normal((nq, num_kv_heads, head_dim), dtype=np.float32), dtype)
    slots = np.empty(nq, np.int32)
    cu_q = np.zeros(S + 1, np.int32)
    cu_k = np.zeros(S + 1, np.int32)
    r = 0
    for s in range(S):
        for pos in range(int(c[s]), int(total[s])):
            slots[r] = int(tables[s, pos // bs]) * bs + pos % bs
            r += 1
        cu_q[s + 1] = cu_q[s] + int(n[s])
        cu_k[s + 1] = cu_k[s] + int(total[s])
    return PagedCase(name=name, num_heads=num_heads, num_kv_heads=num_kv_heads,
                     head_dim=head_dim, block_size=bs, num_blocks=nb, block_tables=tables,
                     context_lens=total, q=q, k_new=k_new, v_new=v_new, slot_mapping=slots,
                     k_cache=k_cache, v_cache=v_cache, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                     causal=causal, seed=seed)


# ---------------------------------------------------------------------------------------
# The five named workloads. Seeds are SEED_BASE + workload number.
# ---------------------------------------------------------------------------------------

WORKLOADS = {
    1: "tiny paged decode: B=4, ctx {1,17,256,300}, H=16, Hk=8, D=128, bs=256, nb=16, "
       "store of 4 tokens with one slot=-1",
    2: "Qwen3-0.6B-shaped decode step: B=256, ctx U{100..2048}, H=16, Hk=8, D=128, bs=256, "
       "pool 4096 blocks, store of 256 tokens",
    3: "long-context split-KV decode: B=8, ctx U{32768..131072}, H=32, Hk=8, D=128, bs=256, "
       "pool 4096 blocks",
    4: "prefix-cache + block-size stress: B=512, ctx lognormal(6,1) clipped 1..4096, "
       "64-seq groups share their first 4 blocks, H=16, Hk=8, D=128, bs 16 or 256",
    5: "chunked prefill: 32 seqs, cached U{0..2048}, new U{100..1024}, causal, H=16, Hk=8, "
       "D=128, bs=256, store of all new tokens",
}


def workload(num: int, block_size: Optional[int] = None, poison: bool = True,
             num_blocks: Optional[int] = None, head_dim: int = 128,
             dtype: torch.dtype = torch.bfloat16) -> PagedCase:
    """Build named workload `num` (1..5). Workload 4 takes block_size 16 or 256.
    num_blocks overrides the pool size of workloads 2, 3 and 5 (the drawn lengths and the
    values do not change; only the physical ids do). head_dim (64 or 128) and the element
    type (bf16 or fp16) apply to workloads 2 and 5: the same lengths and block tables with
    other head sizes or element types."""
    if (head_dim != 128 or dtype != torch.bfloat16) and num not in (2, 5):
        raise ValueError("head_dim / dtype variants exist for workloads 2 and 5")
    sfx = "" if (head_dim == 128 and dtype == torch.bfloat16) else \
        f"_d{head_dim}_{'fp16' if dtype == torch.float16 else 'bf16'}"
    seed = SEED_BASE + num
    if num == 1:
        return decode_case([1, 17, 256, 300], 16, 8, 128, 256, num_blocks=16, seed=seed,
                           poison=poison, skip_slots=[1], max_blocks=2, name="w1_tiny_decode")
    rng = np.random.default_rng(seed)
    if num == 2:
        lens = rng.integers(100, 2048 + 1, size=256)
        return decode_case(lens, 16, 8, head_dim, 256, num_blocks=num_blocks or 4096,
                           seed=seed + 1000, poison=poison, max_blocks=8,
                           name="w2_qwen3_decode_b256" + sfx, dtype=dtype)
    if num == 3:
        lens = rng.integers(32768, 131072 + 1, size=8)
        return decode_case(lens, 32, 8, 128, 256, num_blocks=num_blocks or 4096,
                           seed=seed + 1000, poison=poison, max_blocks=512,
                           name="w3_long_context_b8")
    if num == 4:
        bs = block_size or 256
        lens = np.clip(np.round(rng.lognormal(6.0, 1.0, size=512)), 1, 4096).astype(np.int64)
        need = sum(-(-int(n) // bs) for n in lens)
        return decode_case(lens, 16, 8, 128, bs, num_blocks=need + need // 4 + 8,
                           seed=seed + 1000 + bs, poison=poison, share_group=64,
                           share_blocks=4, name=f"w4_prefix_share_bs{bs}")
    if num == 5:
        cached = rng.integers(0, 2048 + 1, size=32)
        new = rng.integers(100, 1024 + 1, size=32)
        return prefill_case(cached, new, 16, 8, head_dim, 256, num_blocks=num_blocks or 4096,
                            seed=seed + 1000, poison=poison, causal=True,
                            name="w5_chunked_prefill" + sfx, dtype=dtype)
    raise ValueError(f"no workload {num}")
