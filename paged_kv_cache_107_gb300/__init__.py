"""paged_kv_cache_107_gb300 — paged-KV attention for GB300 (sm_103a).

A thin Python binding over the C ABI of ``lib/libpagedkv.so`` (declared in
``include/pa.h``). Every function marshals torch tensors into pointers and sizes and
calls the library with the same name; all arithmetic runs in the library's CUDA
kernels. There is no CPU or PyTorch fallback: if the library is missing or a CUDA device
is absent the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = ["pa_store_kvcache", "pa_decode", "pa_decode_step", "pa_decode_workspace_size",
           "pa_prefill_varlen", "pa_decode_noalloc", "pa_staged_write_apply",
           "pa_staged_pack", "pa_staged_pack_bound", "pa_staged_upload_apply",
           "PaStagedLayout", "pa_sample_workspace_size", "pa_gumbel_sample",
           "SampleWorkspace",
           "pa_status_str", "pa_version", "DecodeWorkspace", "library_path", "load_library",
           "PA_DEV_ERR"]

PA_DEV_ERR = {"block_id": 1, "slot": 2, "context": 4, "timeout": 8, "seqlens": 16,
              "staged": 32}

PA_ERR_WORKSPACE_CODE = 4

_lock = threading.Lock()
_lib = None


class PagedAttentionError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: Optional[str] = None):
    """Load (once) the CUDA library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise PagedAttentionError(
                f"CUDA library not found at {p}; build it first "
                "(python -m paged_kv_cache_107_gb300.build or __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        lib.pa_status_str.argtypes = [i32]
        lib.pa_status_str.restype = ctypes.c_char_p
        lib.pa_version.argtypes = []
        lib.pa_version.restype = i32
        lib.pa_store_kvcache.argtypes = [vp, vp, i64, i64, vp, vp, vp, i32, i32, i32, i32, i64,
                                         vp, vp]
        lib.pa_store_kvcache.restype = i32
        lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.pa_decode_workspace_size.restype = sz
        lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i64,
                                  f32, i32, vp, sz, vp, vp]
        lib.pa_decode.restype = i32
        lib.pa_decode_step.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, i32, vp, i32,
                                       i32, i32, i32, i32, i32, i64, f32, i32, vp, sz, vp, vp]
        lib.pa_decode_step.restype = i32
        lib.pa_sample_workspace_size.argtypes = [i32]
        lib.pa_sample_workspace_size.restype = sz
        lib.pa_gumbel_sample.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, vp, vp, sz, vp, vp]
        lib.pa_gumbel_sample.restype = i32
        lib.pa_staged_write_apply.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, vp, i32, i64,
                                              vp, vp]
        lib.pa_staged_write_apply.restype = i32
        lib.pa_prefill_varlen.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                          i32, i32, i32, i64, i32, f32, vp, vp]
        lib.pa_prefill_varlen.restype = i32
        _lib = lib
        return lib


def pa_status_str(status: int) -> str:
    return load_library().pa_status_str(int(status)).decode()


def pa_version() -> int:
    return int(load_library().pa_version())


def _check(rc: int, what: str):
    if rc != 0:
        raise PagedAttentionError(f"{what}: {pa_status_str(rc)}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _one_device(*tensors, stream=None) -> None:
    """Every tensor lies on one CUDA device, that device is the current one (the library
    launches there, on its current or the given stream), and a given stream belongs to it.
    Checked before any launch: a kernel handed another device's pointers would fault."""
    devs = {t.device for t in tensors if t is not None}
    if any(d.type != "cuda" for d in devs):
        raise PagedAttentionError("every tensor must be a CUDA tensor")
    idx = {torch.cuda.current_device() if d.index is None else d.index for d in devs}
    if len(idx) > 1:
        raise PagedAttentionError(f"tensors on several devices: cuda:{sorted(idx)}")
    cur = torch.cuda.current_device()
    if idx and idx != {cur}:
        raise PagedAttentionError(
            f"tensors are on cuda:{next(iter(idx))} but the current device is cuda:{cur}; "
            "call under torch.cuda.device(...) of the tensors' device")
    if stream is not None and stream.device.index is not None and stream.device.index != cur:
        raise PagedAttentionError(f"stream belongs to {stream.device}, tensors to cuda:{cur}")


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: Optional[int] = None):
    if not t.is_cuda:
        raise PagedAttentionError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise PagedAttentionError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise PagedAttentionError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def pa_store_kvcache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                     dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v [N, Hk, D] bf16 or fp16 (token stride may exceed Hk*D); caches [nb, bs, Hk, D]
    of the same type (the store is a bit copy)."""
    _need16(k_cache, "k_cache", 4)
    _need16(v_cache, "v_cache", 4, k_cache.dtype)
    _need16(k, "k", 3, k_cache.dtype)
    _need16(v, "v", 3, k_cache.dtype)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    nb, bs, hk, d = k_cache.shape
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and v_cache.shape == k_cache.shape):
        raise PagedAttentionError("caches must be contiguous and of equal shape")
    for name, t in (("k", k), ("v", v)):
        if t.shape[1:] != (hk, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise PagedAttentionError(f"{name} rows must be [Hk, D] contiguous")
    if slot_mapping.shape[0] != k.shape[0] or v.shape[0] != k.shape[0]:
        raise PagedAttentionError("slot_mapping / k / v token counts differ")
    _one_device(k, v, k_cache, v_cache, slot_mapping, dev_err, stream=stream)
    rc = load_library().pa_store_kvcache(
        _ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(k_cache), _ptr(v_cache),
        _ptr(slot_mapping), k.shape[0], hk, d, bs, nb, _ptr(dev_err), _stream(stream))
    _check(rc, "pa_store_kvcache")


def pa_staged_write_apply(base: torch.Tensor, rows: torch.Tensor, starts: torch.Tensor,
                          offsets: torch.Tensor, values: torch.Tensor,
                          dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """base [R, C] device tensor (rows may be strided, columns contiguous); rows, starts
    int32 [W]; offsets int32 [W+1]; values [offsets[W]] of base's element size. Run w
    writes values[offsets[w]:offsets[w+1]] to base[rows[w], starts[w]:...]."""
    if base.dim() != 2 or base.stride(1) != 1:
        raise PagedAttentionError("base must be 2-D with contiguous columns")
    for name, t in (("rows", rows), ("starts", starts), ("offsets", offsets)):
        _need(t, name, torch.int32, 1)
    if values.element_size() != base.element_size() or values.dim() != 1:
        raise PagedAttentionError("values must be 1-D with base's element size")
    W = rows.shape[0]
    if starts.shape[0] != W or offsets.shape[0] != W + 1:
        raise PagedAttentionError("rows / starts / offsets sizes disagree")
    _one_device(base, rows, starts, offsets, values, dev_err, stream=stream)
    rc = load_library().pa_staged_write_apply(
        _ptr(base), base.shape[0], base.shape[1], base.stride(0), base.element_size(),
        _ptr(rows), _ptr(starts), _ptr(offsets), _ptr(values), W, values.shape[0],
        _ptr(dev_err), _stream(stream))
    _check(rc, "pa_staged_write_apply")


class PaStagedLayout(ctypes.Structure):
    """pa_staged_layout: byte offsets of the packed arrays, run and value counts."""
    _fields_ = [("rows_offset", ctypes.c_int64), ("starts_offset", ctypes.c_int64),
                ("offsets_offset", ctypes.c_int64), ("values_offset", ctypes.c_int64),
                ("num_writes", ctypes.c_int32), ("num_values", ctypes.c_int64),
                ("bytes", ctypes.c_int64)]


def _staged_lib():
    lib = load_library()
    if not getattr(lib.pa_staged_pack, "_pa_typed", False):
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.pa_staged_pack_bound.argtypes = [i32, i64, i32]
        lib.pa_staged_pack_bound.restype = sz
        lib.pa_staged_pack.argtypes = [vp, vp, vp, vp, i32, i32, vp, sz,
                                       ctypes.POINTER(PaStagedLayout)]
        lib.pa_staged_pack.restype = i32
        lib.pa_staged_pack._pa_typed = True
    return lib


def pa_staged_pack_bound(num_writes: int, num_values: int, elem_bytes: int) -> int:
    return int(_staged_lib().pa_staged_pack_bound(num_writes, num_values, elem_bytes))


def pa_staged_pack(rows, starts, lens, values, elem_bytes: int, packed) -> PaStagedLayout:
    """Native merge + pack (host code, no GPU): rows, starts, lens int32 numpy arrays and
    values a numpy array of elem_bytes-byte elements, in staging order; `packed` a writable
    host byte array (numpy, or the numpy view of a pinned tensor). Returns the layout;
    raises with the needed size when `packed` is too small."""
    import numpy as np
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    starts = np.ascontiguousarray(starts, dtype=np.int32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    values = np.ascontiguousarray(values)
    lay = PaStagedLayout()
    rc = _staged_lib().pa_staged_pack(
        rows.ctypes.data, starts.ctypes.data, lens.ctypes.data,
        values.ctypes.data if values.size else None, len(rows), elem_bytes,
        packed.ctypes.data, packed.nbytes, ctypes.byref(lay))
    if rc == PA_ERR_WORKSPACE_CODE:
        raise PagedAttentionError(f"pa_staged_pack: buffer too small, {lay.bytes} bytes needed")
    _check(rc, "pa_staged_pack")
    return lay


def pa_staged_upload_apply(base: torch.Tensor, packed_host: torch.Tensor,
                           packed_dev: torch.Tensor, layout: PaStagedLayout,
                           dev_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """One H2D copy of a packed buffer (pinned host uint8 tensor -> device uint8 tensor)
    and the apply of its runs to `base` [R, C] (contiguous columns), on `stream`."""
    lib = _staged_lib()
    fn = lib.pa_staged_upload_apply
    if not getattr(fn, "_pa_typed", False):
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        fn.argtypes = [vp, i64, i64, i64, i32, vp, vp, ctypes.POINTER(PaStagedLayout), vp, vp]
        fn.restype = i32
        fn._pa_typed = True
    if base.dim() != 2 or base.stride(1) != 1:
        raise PagedAttentionError("base must be 2-D with contiguous columns")
    if packed_dev.numel() < layout.bytes or packed_host.numel() < layout.bytes:
        raise PagedAttentionError("packed buffers smaller than layout.bytes")
    _one_device(base, packed_dev, dev_err, stream=stream)
    rc = fn(base.data_ptr(), base.shape[0], base.shape[1], base.stride(0), base.element_size(),
            packed_host.data_ptr(), packed_dev.data_ptr(), ctypes.byref(layout),
            _ptr(dev_err), _stream(stream))
    _check(rc, "pa_staged_upload_apply")


PA_DTYPE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
_ATTN_TYPES = (torch.bfloat16, torch.float16)


def _need16(t: torch.Tensor, name: str, ndim: int, dtype: Optional[torch.dtype] = None):
    """A CUDA tensor of 16-bit floats (bf16 or fp16; `dtype` when given)."""
    if not t.is_cuda:
        raise PagedAttentionError(f"{name} must be a CUDA tensor")
    if t.dtype not in _ATTN_TYPES or (dtype is not None and t.dtype != dtype):
        raise PagedAttentionError(f"{name} must be {dtype or 'bf16 or fp16'}, got {t.dtype}")
    if t.dim() != ndim:
        raise PagedAttentionError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def pa_sample_workspace_size(num_seqs: int) -> int:
    return int(load_library().pa_sample_workspace_size(num_seqs))


class SampleWorkspace:
    """Zero-initialised sampler scratch (per-row keys and arrival counters; every call
    leaves it zero). One workspace per stream of concurrent calls."""

    def __init__(self, num_seqs: int, device=None):
        self.nbytes = pa_sample_workspace_size(max(num_seqs, 1))
        self.num_seqs = num_seqs
        self.buffer = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")


_sample_ws = {}


def pa_gumbel_sample(out: torch.Tensor, logits: torch.Tensor, temperatures: torch.Tensor,
                     seeds: torch.Tensor, offsets: torch.Tensor,
                     workspace: Optional[SampleWorkspace] = None,
                     dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out int64 [B]; logits [B, V] fp32 or bf16 with contiguous columns (any row stride);
    temperatures fp32 [B] (<= 0: greedy); seeds, offsets int64 [B] read as uint64."""
    if logits.dim() != 2 or logits.stride(1) != 1 or logits.dtype not in PA_DTYPE:
        raise PagedAttentionError("logits must be 2-D fp32/bf16 with contiguous columns")
    if not logits.is_cuda:
        raise PagedAttentionError("logits must be a CUDA tensor")
    B, V = logits.shape
    _need(out, "out", torch.int64, 1)
    _need(temperatures, "temperatures", torch.float32, 1)
    _need(seeds, "seeds", torch.int64, 1)
    _need(offsets, "offsets", torch.int64, 1)
    if not (out.shape[0] == temperatures.shape[0] == seeds.shape[0] == offsets.shape[0] == B):
        raise PagedAttentionError("out / temperatures / seeds / offsets must have B entries")
    if workspace is None:
        key = (logits.device.index, B)
        workspace = _sample_ws.get(key)
        if workspace is None:
            workspace = _sample_ws[key] = SampleWorkspace(B, device=logits.device)
    _one_device(out, logits, temperatures, seeds, offsets, workspace.buffer, dev_err,
                stream=stream)
    rc = load_library().pa_gumbel_sample(
        _ptr(out), _ptr(logits), logits.stride(0) if B > 1 else V, PA_DTYPE[logits.dtype], B, V,
        _ptr(temperatures), _ptr(seeds), _ptr(offsets), _ptr(workspace.buffer),
        workspace.nbytes, _ptr(dev_err), _stream(stream))
    _check(rc, "pa_gumbel_sample")
    return out


def pa_decode_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int,
                             head_dim: int = 128) -> int:
    return int(load_library().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads,
                                                       head_dim))


class DecodeWorkspace:
    """Zero-initialised decode scratch (its arrival counters must start at zero; every
    successful call leaves them zero). One workspace per stream of concurrent calls."""

    def __init__(self, num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int = 128,
                 device=None):
        n = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim)
        if n == 0:
            raise PagedAttentionError("invalid decode workspace sizes")
        self.nbytes = n
        self.buffer = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
        self.key = (num_seqs, num_heads, num_kv_heads, head_dim)

    def fits(self, num_seqs, num_heads, num_kv_heads, head_dim=128) -> bool:
        return pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim) <= self.nbytes

    def reset(self):
        self.buffer.zero_()


_ws_cache = {}


def _default_workspace(B, H, Hk, D, device) -> DecodeWorkspace:
    key = (device.index if device.index is not None else torch.cuda.current_device(), H, Hk, D)
    ws = _ws_cache.get(key)
    if ws is None or not ws.fits(B, H, Hk, D):
        ws = DecodeWorkspace(max(B, 1), H, Hk, D, device=device)
        _ws_cache[key] = ws
    return ws


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor,
              scale: Optional[float] = None, grid_ctas: int = 0,
              workspace: Optional[DecodeWorkspace] = None,
              dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out, q [B, H, D] bf16 or fp16 (D = 64 or 128); caches [nb, bs, Hk, D] of the same
    type; block_tables [B, maxb] int32 (-1 padded); context_lens [B] int32."""
    _need16(q, "q", 3)
    for name, t, dt, nd in (("out", out, q.dtype, 3),
                            ("k_cache", k_cache, q.dtype, 4),
                            ("v_cache", v_cache, q.dtype, 4),
                            ("block_tables", block_tables, torch.int32, 2),
                            ("context_lens", context_lens, torch.int32, 1)):
        _need(t, name, dt, nd)
        if not t.is_contiguous():
            raise PagedAttentionError(f"{name} must be contiguous")
    if not q.is_contiguous():
        raise PagedAttentionError("q must be contiguous")
    B, H, D = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if out.shape != q.shape or d2 != D or v_cache.shape != k_cache.shape:
        raise PagedAttentionError("shape mismatch")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise PagedAttentionError("block_tables / context_lens batch mismatch")
    if workspace is None:
        workspace = _default_workspace(B, H, hk, D, q.device)
    _one_device(out, q, k_cache, v_cache, block_tables, context_lens, workspace.buffer, dev_err,
                stream=stream)
    rc = load_library().pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, H, hk, D, PA_DTYPE[q.dtype], bs, nb,
        float(scale) if scale is not None else 0.0, int(grid_ctas), _ptr(workspace.buffer),
        workspace.nbytes, _ptr(dev_err), _stream(stream))
    _check(rc, "pa_decode")
    return out


def pa_decode_step(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                   block_tables: torch.Tensor, context_lens: torch.Tensor,
                   scale: Optional[float] = None, grid_ctas: int = 0,
                   workspace: Optional[DecodeWorkspace] = None,
                   dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Store of each sequence's new token plus decode, in one launch: the same result as
    pa_store_kvcache(k_new, v_new, ..., slot_mapping) then pa_decode(...). k_new, v_new
    [B, Hk, D] of q's type (token stride a multiple of 8 elements); slot_mapping [B]
    int32, -1 or the slot of position context_lens[b]-1 of sequence b."""
    _need16(q, "q", 3)
    for name, t, dt, nd in (("out", out, q.dtype, 3), ("q", q, q.dtype, 3),
                            ("k_cache", k_cache, q.dtype, 4),
                            ("v_cache", v_cache, q.dtype, 4),
                            ("block_tables", block_tables, torch.int32, 2),
                            ("context_lens", context_lens, torch.int32, 1),
                            ("slot_mapping", slot_mapping, torch.int32, 1)):
        _need(t, name, dt, nd)
        if not t.is_contiguous():
            raise PagedAttentionError(f"{name} must be contiguous")
    _need16(k_new, "k_new", 3, q.dtype)
    _need16(v_new, "v_new", 3, q.dtype)
    B, H, D = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if out.shape != q.shape or d2 != D or v_cache.shape != k_cache.shape:
        raise PagedAttentionError("shape mismatch")
    if block_tables.shape[0] != B or context_lens.shape[0] != B or slot_mapping.shape[0] != B:
        raise PagedAttentionError("block_tables / context_lens / slot_mapping batch mismatch")
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t.shape != (B, hk, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise PagedAttentionError(f"{name} must be [B, Hk, D] with contiguous rows")
    if workspace is None:
        workspace = _default_workspace(B, H, hk, D, q.device)
    _one_device(out, q, k_new, v_new, k_cache, v_cache, slot_mapping, block_tables,
                context_lens, workspace.buffer, dev_err, stream=stream)
    rc = load_library().pa_decode_step(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), k_new.stride(0), v_new.stride(0),
        _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, H, hk, D, PA_DTYPE[q.dtype], bs, nb,
        float(scale) if scale is not None else 0.0, int(grid_ctas), _ptr(workspace.buffer),
        workspace.nbytes, _ptr(dev_err), _stream(stream))
    _check(rc, "pa_decode_step")
    return out


def pa_prefill_varlen(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                      cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int,
                      max_seqlen_k: int, causal: bool = True, scale: Optional[float] = None,
                      dev_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out, q [sum n, H, D] bf16 or fp16 (D = 64 or 128); caches of the same type hold every
    key/value row already (store first)."""
    _need16(q, "q", 3)
    for name, t, dt, nd in (("out", out, q.dtype, 3), ("q", q, q.dtype, 3),
                            ("k_cache", k_cache, q.dtype, 4),
                            ("v_cache", v_cache, q.dtype, 4),
                            ("block_tables", block_tables, torch.int32, 2),
                            ("cu_seqlens_q", cu_seqlens_q, torch.int32, 1),
                            ("cu_seqlens_k", cu_seqlens_k, torch.int32, 1)):
        _need(t, name, dt, nd)
        if not t.is_contiguous():
            raise PagedAttentionError(f"{name} must be contiguous")
    T, H, D = q.shape
    nb, bs, hk, d2 = k_cache.shape
    S = cu_seqlens_q.shape[0] - 1
    if out.shape != q.shape or d2 != D or v_cache.shape != k_cache.shape:
        raise PagedAttentionError("shape mismatch")
    if cu_seqlens_k.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise PagedAttentionError("cu_seqlens / block_tables batch mismatch")
    _one_device(out, q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, dev_err,
                stream=stream)
    rc = load_library().pa_prefill_varlen(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), S, int(max_seqlen_q),
        int(max_seqlen_k), H, hk, D, PA_DTYPE[q.dtype], bs, nb, 1 if causal else 0,
        float(scale) if scale is not None else 0.0, _ptr(dev_err), _stream(stream))
    _check(rc, "pa_prefill_varlen")
    return out


def pa_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: Optional[float] = None,
                      grid_ctas: int = 0, dev_err: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """pa_decode for callers that cannot allocate device memory: same arguments without a
    workspace; the library's fixed 16 MiB device scratch is used instead (see pa.h for the
    size limit and for why overlapping calls must be serialised)."""
    lib = load_library()
    fn = lib.pa_decode_noalloc
    if not getattr(fn, "_pa_typed", False):
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        fn.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, i32, vp,
                       vp]
        fn.restype = ctypes.c_int
        fn._pa_typed = True
    for name, t, dt, nd in (("out", out, torch.bfloat16, 3), ("q", q, torch.bfloat16, 3),
                            ("k_cache", k_cache, torch.bfloat16, 4),
                            ("v_cache", v_cache, torch.bfloat16, 4),
                            ("block_tables", block_tables, torch.int32, 2),
                            ("context_lens", context_lens, torch.int32, 1)):
        _need(t, name, dt, nd)
        if not t.is_contiguous():
            raise PagedAttentionError(f"{name} must be contiguous")
    B, H, D = q.shape
    nb, bs, hk, d2 = k_cache.shape
    if out.shape != q.shape or d2 != D or v_cache.shape != k_cache.shape:
        raise PagedAttentionError("shape mismatch")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise PagedAttentionError("block_tables / context_lens batch mismatch")
    _one_device(out, q, k_cache, v_cache, block_tables, context_lens, dev_err, stream=stream)
    rc = fn(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), B, H, hk, D, bs, nb,
            float(scale) if scale is not None else 0.0, int(grid_ctas), _ptr(dev_err),
            _stream(stream))
    _check(rc, "pa_decode_noalloc")
    return out
