"""CPU fp64 oracle for paged-KV attention — TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library's product path never does, and this
package imports nothing from the library: the two share no code. The arithmetic lives in
``oracle.c`` (plain C, one loop per definition on the pages); this module only builds it
with gcc and marshals numpy arrays into it.

Definitions followed (page title, section): see the header of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "lib")
_LIB_PATH = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_STATUS = {0: "ok", 1: "bad slot", 2: "bad block id", 3: "bad context length",
                 4: "bad shape", 5: "bad cu_seqlens"}


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/lib/liboracle.so with gcc (-O2, OpenMP)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load(path=None):
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib = ctypes.CDLL(path or build())
        p = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_store_kvcache.argtypes = [p, p, i64, i64, p, p, p, i64, i32, i32, i64]
        lib.oracle_store_kvcache.restype = i32
        lib.oracle_decode.argtypes = [p, p, p, p, p, p, i32, p, i32, i32, i32, i32, i32, i64,
                                      dbl, p, i64, i32, i32]
        lib.oracle_decode.restype = i32
        lib.oracle_prefill.argtypes = [p, p, p, p, p, p, i32, p, p, i32, i32, i32, i32, i32,
                                       i64, i32, dbl, p, i64, i32, i32]
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = dbl
        lib.oracle_prefill.restype = i32
        lib.oracle_slot_of.argtypes = [p, i32, i64, i32]
        lib.oracle_slot_of.restype = i64
        lib.oracle_staged_apply.argtypes = [p, i64, i64, i32, i32, p, p, p, p]
        lib.oracle_staged_apply.restype = i32
        u32, u64 = ctypes.c_uint32, ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [p, p, p]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_philox_bits.argtypes = [u64, u64, u64]
        lib.oracle_philox_bits.restype = u32
        lib.oracle_uniform.argtypes = [u32]
        lib.oracle_uniform.restype = dbl
        lib.oracle_gumbel_sample.argtypes = [p, p, p, p, i64, i32, i32, i64, p, p, p, i32]
        lib.oracle_gumbel_sample.restype = i32
        lib.oracle_gumbel_scores.argtypes = [p, p, i32, i64, ctypes.c_float, u64, u64]
        lib.oracle_gumbel_scores.restype = i32
        lib.oracle_max_threads.argtypes = [i32]
        lib.oracle_max_threads.restype = i32
        _lib = lib
        return lib


def use_library(path):
    """Point the wrappers at another build of oracle.c (the mutation tests compile
    deliberately broken copies to check that the pins catch them). Returns the previous
    handle; pass it to restore_library."""
    global _lib
    prev = _lib
    _lib = None
    _load(path)
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def _u16(a) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array of its raw bits (torch or numpy input)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and "bfloat16" in str(a.dtype):
        import torch  # only reached when a torch tensor is passed
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits as uint16, got {a.dtype}")
    return a


def _bits(a):
    """16-bit float data (torch bf16 / fp16, numpy float16, or raw uint16 bf16 bits) as a
    C-contiguous uint16 array of its bits, and 1 if it is IEEE binary16, else 0."""
    if hasattr(a, "view") and hasattr(a, "dtype") and "float16" in str(a.dtype) \
            and "bfloat16" not in str(a.dtype):
        if hasattr(a, "detach"):  # torch
            import torch
            a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            a = np.ascontiguousarray(a).view(np.uint16)
        return np.ascontiguousarray(a), 1
    return _u16(a), 0


def f16_to_double(bits: int) -> float:
    """Exact value of an IEEE binary16 bit pattern."""
    return float(_load().oracle_f16_to_double(bits))


def _i32(a) -> np.ndarray:
    if hasattr(a, "cpu"):
        a = a.detach().cpu().numpy()
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: {ORACLE_STATUS.get(rc, rc)}")


def max_threads(nthreads: int = 0) -> int:
    """Number of OpenMP threads the oracle will use (after setting it when > 0)."""
    return int(_load().oracle_max_threads(int(nthreads)))


def store_kvcache(k, v, k_cache, v_cache, slot_mapping):
    """Return (k_cache', v_cache') as uint16 arrays (the raw 16-bit elements) after the
    store of the new rows: a bit copy, so bf16 and fp16 alike.

    k, v: [N, Hk, D]; caches [nb, bs, Hk, D]; slot_mapping int32 [N].
    The inputs are not modified.
    """
    lib = _load()
    k, v = _bits(k)[0], _bits(v)[0]
    kc, vc = _bits(k_cache)[0].copy(), _bits(v_cache)[0].copy()
    slots = _i32(slot_mapping)
    n, hk, d = k.shape
    num_slots = kc.shape[0] * kc.shape[1]
    rc = lib.oracle_store_kvcache(_ptr(k), _ptr(v), hk * d, hk * d, _ptr(kc), _ptr(vc),
                                  _ptr(slots), n, hk, d, num_slots)
    _check(rc, "store")
    return kc, vc


def decode(q, k_cache, v_cache, block_tables, context_lens, scale=None, pairs=None,
           nthreads=0, return_lse=False):
    """fp64 decode attention. q bf16 [B, H, D]; caches bf16 [nb, bs, Hk, D].

    Returns out [B, H, D] float64 (or [len(pairs), D] when pairs, a list of b*H+h
    indices, is given) and, if return_lse, the natural-log LSE per row.
    """
    lib = _load()
    q, f16 = _bits(q)
    (kc, fk), (vc, fv) = _bits(k_cache), _bits(v_cache)
    assert f16 == fk == fv, "q, k_cache and v_cache must share one element type"
    bt, ctx = _i32(block_tables), _i32(context_lens)
    B, H, D = q.shape
    nb, bs, hk, d2 = kc.shape
    assert d2 == D and vc.shape == kc.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if pairs is not None:
        pairs = np.ascontiguousarray(pairs, dtype=np.int64)
        out = np.zeros((len(pairs), D), np.float64)
        lse = np.zeros(len(pairs), np.float64)
        pp, npairs = _ptr(pairs), len(pairs)
    else:
        out = np.zeros((B, H, D), np.float64)
        lse = np.zeros((B, H), np.float64)
        pp, npairs = None, 0
    maxb = bt.shape[1] if bt.ndim == 2 else 0
    rc = lib.oracle_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), maxb,
                           _ptr(ctx), B, H, hk, D, bs, nb, float(scale), pp, npairs,
                           int(nthreads), f16)
    _check(rc, "decode")
    return (out, lse) if return_lse else out


def prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, causal=True,
            scale=None, rows=None, nthreads=0, return_lse=False):
    """fp64 varlen prefill attention. q bf16 or fp16 [sum n, H, D] (caches of the same type).
    rows: optional list of token_row*H + h indices (compact output)."""
    lib = _load()
    q, f16 = _bits(q)
    (kc, fk), (vc, fv) = _bits(k_cache), _bits(v_cache)
    assert f16 == fk == fv, "q, k_cache and v_cache must share one element type"
    bt = _i32(block_tables)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    T, H, D = q.shape
    nb, bs, hk, _ = kc.shape
    S = len(cq) - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((len(rows), D), np.float64)
        lse = np.zeros(len(rows), np.float64)
        rp, nrows = _ptr(rows), len(rows)
    else:
        out = np.zeros((T, H, D), np.float64)
        lse = np.zeros((T, H), np.float64)
        rp, nrows = None, 0
    maxb = bt.shape[1] if bt.ndim == 2 else 0
    rc = lib.oracle_prefill(_ptr(out), _ptr(lse), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), maxb,
                            _ptr(cq), _ptr(ck), S, H, hk, D, bs, nb, 1 if causal else 0,
                            float(scale), rp, nrows, int(nthreads), f16)
    _check(rc, "prefill")
    return (out, lse) if return_lse else out


def staged_write_apply(base, writes):
    """Return a copy of the 2-D array `base` after the staged writes, applied in staging
    order: each write is (row, start, values) and puts the values at row `row`, columns
    start .. start+len(values)-1 ("Model Runner V2 设计文档", "4. StagedWriteTensor")."""
    out = np.ascontiguousarray(np.array(base, copy=True))
    if out.ndim != 2:
        raise ValueError("base must be 2-D")
    rows = np.array([int(w[0]) for w in writes], dtype=np.int64)
    starts = np.array([int(w[1]) for w in writes], dtype=np.int64)
    vals = [np.asarray(w[2], dtype=out.dtype).reshape(-1) for w in writes]
    lens = np.array([len(v) for v in vals], dtype=np.int64)
    flat = (np.ascontiguousarray(np.concatenate(vals)) if vals
            else np.zeros(1, dtype=out.dtype))
    rc = _load().oracle_staged_apply(_ptr(out), out.shape[0], out.shape[1], out.itemsize,
                                     len(writes), _ptr(rows), _ptr(starts), _ptr(lens),
                                     _ptr(flat))
    _check(rc, "staged write")
    return out


def philox4x32_10(counter, key):
    """Philox4x32-10 (Salmon et al., SC 2011): four 32-bit counter words and two key words
    -> four 32-bit outputs."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox_bits(seed: int, offset: int, i: int) -> int:
    """The 32 random bits of vocabulary element i for a row's (seed, offset)."""
    return int(_load().oracle_philox_bits(seed, offset, i))


def uniform(bits: int) -> float:
    """u = (2*(bits >> 9) + 1) / 2^24."""
    return float(_load().oracle_uniform(bits))


def _logits_arg(logits):
    import torch
    if isinstance(logits, torch.Tensor):
        if logits.dtype == torch.bfloat16:
            return _u16(logits), 1
        logits = logits.numpy()
    a = np.ascontiguousarray(logits, dtype=np.float32)
    return a, 0


def gumbel_sample(logits, temperatures, seeds, offsets, nthreads=0):
    """Gumbel-max sample of each row of logits [B, V] (binary32, or a bf16 torch tensor):
    returns (index int64 [B], best score [B], runner-up score [B]) in fp64."""
    a, is_bf16 = _logits_arg(logits)
    B, V = a.shape
    t = np.ascontiguousarray(temperatures, dtype=np.float32)
    sd = np.ascontiguousarray(seeds, dtype=np.uint64)
    of = np.ascontiguousarray(offsets, dtype=np.uint64)
    out = np.zeros(B, np.int64)
    best = np.zeros(B, np.float64)
    second = np.zeros(B, np.float64)
    rc = _load().oracle_gumbel_sample(_ptr(out), _ptr(best), _ptr(second), _ptr(a), V, is_bf16,
                                      B, V, _ptr(t), _ptr(sd), _ptr(of), int(nthreads))
    _check(rc, "gumbel sample")
    return out, best, second


def gumbel_scores(row_logits, temperature: float, seed: int, offset: int):
    """All fp64 scores logits/T - ln(-ln u) of one row (the logit alone when T <= 0)."""
    a, is_bf16 = _logits_arg(row_logits)
    a = a.reshape(-1)
    out = np.zeros(a.shape[0], np.float64)
    _load().oracle_gumbel_scores(_ptr(out), _ptr(a), is_bf16, a.shape[0], float(temperature),
                                 int(seed), int(offset))
    return out


def slot_of(block_table_row, pos: int, block_size: int) -> int:
    """Slot of logical position pos for one sequence's block-table row (-1 if unmapped)."""
    lib = _load()
    row = _i32(block_table_row)
    return int(lib.oracle_slot_of(_ptr(row), len(row), int(pos), int(block_size)))
