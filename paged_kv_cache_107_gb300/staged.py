"""StagedWriteTensor: a device-resident 2-D tensor updated by staged runs of writes.

"Model Runner V2 设计文档", section "4. StagedWriteTensor": the tensor (block tables,
for instance) stays on the GPU; the host stages only the changed runs, packs them into
one contiguous buffer, copies that buffer in one host-to-device copy and launches one
kernel (pa_staged_write_apply) that applies them. No full copy of the tensor and no
host-device synchronisation on the way.

Host side only: staging, merging overlapping runs of the same row (later writes win, so
the packed runs never overlap) and packing. Every element of the tensor is written by
the CUDA kernel."""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import PagedAttentionError, _ptr, _stream, load_library

_NP = {torch.int32: np.int32, torch.float32: np.float32, torch.int64: np.int64,
       torch.int16: np.int16, torch.uint8: np.uint8, torch.float64: np.float64}


def merge_runs(staged: Sequence[Tuple[int, int, np.ndarray]]) -> List[Tuple[int, int, np.ndarray]]:
    """Staged (row, start, values) writes, in staging order -> non-overlapping runs with
    the same effect: within a row, a later write overrides an earlier one where they
    overlap; runs that overlap or touch are joined. Output sorted by (row, start)."""
    by_row: Dict[int, List[Tuple[int, np.ndarray]]] = {}
    for row, start, vals in staged:
        if len(vals):
            by_row.setdefault(row, []).append((start, vals))
    out = []
    for row in sorted(by_row):
        writes = by_row[row]
        if len(writes) == 1:
            out.append((row, writes[0][0], writes[0][1]))
            continue
        lo = min(s for s, _ in writes)
        hi = max(s + len(v) for s, v in writes)
        buf = np.zeros(hi - lo, dtype=writes[0][1].dtype)
        mask = np.zeros(hi - lo, dtype=bool)
        for s, v in writes:  # staging order: later writes land last
            buf[s - lo:s - lo + len(v)] = v
            mask[s - lo:s - lo + len(v)] = True
        # maximal runs of covered columns
        edges = np.flatnonzero(np.diff(np.concatenate(([0], mask.view(np.int8), [0]))))
        for a, b in zip(edges[0::2], edges[1::2]):
            out.append((row, lo + int(a), buf[a:b].copy()))
    return out


def pack_runs(runs: Sequence[Tuple[int, int, np.ndarray]], elem_bytes: int) -> Tuple[np.ndarray, dict]:
    """One contiguous byte buffer: int32 rows[W], starts[W], offsets[W+1], then the values
    (aligned to max(elem_bytes, 4)). Returns the buffer and the byte offsets of each part."""
    W = len(runs)
    lens = np.array([len(v) for _, _, v in runs], dtype=np.int64)
    offsets = np.zeros(W + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    if offsets[-1] > np.iinfo(np.int32).max:
        raise PagedAttentionError("too many staged values for int32 offsets")
    head = 4 * (3 * W + 1)
    align = max(elem_bytes, 16)
    val_off = (head + align - 1) // align * align
    total = val_off + int(offsets[-1]) * elem_bytes
    buf = np.zeros(total, dtype=np.uint8)
    meta = buf[:head].view(np.int32)
    meta[:W] = [r for r, _, _ in runs]
    meta[W:2 * W] = [s for _, s, _ in runs]
    meta[2 * W:3 * W + 1] = offsets
    if W:
        buf[val_off:] = np.concatenate([v for _, _, v in runs]).view(np.uint8)
    return buf, {"rows": 0, "starts": 4 * W, "offsets": 8 * W, "values": val_off,
                 "num_writes": W, "num_values": int(offsets[-1])}


class StagedWriteTensor:
    """A [rows, cols] tensor on the GPU with host-staged run writes.

    stage_write(row, start, values) records a run on the host; apply_write() merges the
    staged runs, packs them into one pinned buffer, copies it to the device in one copy and
    applies it with one kernel launch on `stream`. Both calls return without waiting for
    the GPU; the pinned buffer of a previous apply is reused only after its copy ended."""

    def __init__(self, size: Tuple[int, int], dtype: torch.dtype = torch.int32,
                 device="cuda", init: Optional[torch.Tensor] = None):
        if dtype not in _NP:
            raise PagedAttentionError(f"unsupported dtype {dtype}")
        self.gpu = (init.to(device=device, dtype=dtype).contiguous().clone() if init is not None
                    else torch.zeros(size, dtype=dtype, device=device))
        if self.gpu.dim() != 2:
            raise PagedAttentionError("StagedWriteTensor is 2-D")
        self.dtype = dtype
        self._np = _NP[dtype]
        self._staged: List[Tuple[int, int, np.ndarray]] = []
        self._pinned: Optional[torch.Tensor] = None
        self._dev: Optional[torch.Tensor] = None
        self._copied: Optional[torch.cuda.Event] = None
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=self.gpu.device)
        self.last_h2d_bytes = 0

    def stage_write(self, row: int, start: int, value) -> None:
        self._staged.append((int(row), int(start), np.array(value, dtype=self._np).reshape(-1)))

    def apply_write(self, stream=None) -> None:
        if not self._staged:
            return
        runs = merge_runs(self._staged)
        self._staged = []
        buf, lay = pack_runs(runs, self.gpu.element_size())
        n = buf.nbytes
        if self._pinned is None or self._pinned.numel() < n:
            cap = max(n, 4096)
            self._pinned = torch.empty(cap, dtype=torch.uint8).pin_memory()
            self._dev = torch.empty(cap, dtype=torch.uint8, device=self.gpu.device)
            self._copied = None
        if self._copied is not None:
            self._copied.synchronize()  # the previous copy must have read the pinned buffer
        self._pinned[:n].numpy()[:] = buf
        s = stream if stream is not None else torch.cuda.current_stream(self.gpu.device)
        with torch.cuda.stream(s):
            self._dev[:n].copy_(self._pinned[:n], non_blocking=True)
            self._copied = torch.cuda.Event()
            self._copied.record(s)
        self.last_h2d_bytes = n
        base = self._dev.data_ptr()
        rc = load_library().pa_staged_write_apply(
            _ptr(self.gpu), self.gpu.shape[0], self.gpu.shape[1], self.gpu.stride(0),
            self.gpu.element_size(), base + lay["rows"], base + lay["starts"],
            base + lay["offsets"], base + lay["values"], lay["num_writes"], lay["num_values"],
            _ptr(self.dev_err), _stream(s))
        if rc != 0:
            raise PagedAttentionError(f"pa_staged_write_apply: {load_library().pa_status_str(rc).decode()}")
