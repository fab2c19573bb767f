"""Write the small golden regression fixtures from the oracle alone.

Run from the repository root: python tests/golden/make_golden.py
Inputs are drawn with numpy's default_rng (seeds below) and rounded to bf16; the
expected values come from oracle.decode / oracle.prefill and nothing else.
"""
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def bits(t):
    return t.contiguous().view(torch.int16).tolist()


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def decode_small():
    rng = np.random.default_rng(107100)
    nb, bs, hk, d, H = 4, 4, 2, 8, 4
    kc = bf16(rng.standard_normal((nb, bs, hk, d)))
    vc = bf16(rng.standard_normal((nb, bs, hk, d)))
    bt = np.array([[2, 0], [3, -1]], np.int32)
    lens = np.array([6, 3], np.int32)
    q = bf16(rng.standard_normal((2, H, d)))
    out = oracle.decode(q, kc, vc, bt, lens)
    return {"kind": "decode",
            "source": "decode over a paged cache, block_size 4, two sequences; written by make_golden.py",
            "inputs": {"q_bits": bits(q), "k_cache_bits": bits(kc), "v_cache_bits": bits(vc),
                       "block_tables": bt.tolist(), "context_lens": lens.tolist()},
            "expected": out.tolist()}


def prefill_small():
    rng = np.random.default_rng(107101)
    nb, bs, hk, d, H = 4, 4, 1, 8, 2
    kc = bf16(rng.standard_normal((nb, bs, hk, d)))
    vc = bf16(rng.standard_normal((nb, bs, hk, d)))
    bt = np.array([[1, 3], [0, 2]], np.int32)
    cu_q = np.array([0, 3, 5], np.int32)
    cu_k = np.array([0, 7, 12], np.int32)
    q = bf16(rng.standard_normal((5, H, d)))
    out = oracle.prefill(q, kc, vc, bt, cu_q, cu_k, causal=True)
    return {"kind": "prefill",
            "source": "causal prefill with cached prefixes 4 and 3, block_size 4; written by make_golden.py",
            "inputs": {"q_bits": bits(q), "k_cache_bits": bits(kc), "v_cache_bits": bits(vc),
                       "block_tables": bt.tolist(), "cu_seqlens_q": cu_q.tolist(),
                       "cu_seqlens_k": cu_k.tolist(), "causal": True},
            "expected": out.tolist()}


if __name__ == "__main__":
    for name, fn in [("decode_small.json", decode_small), ("prefill_small.json", prefill_small)]:
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f)
        print("wrote", name)
