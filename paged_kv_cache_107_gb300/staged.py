"""StagedWriteTensor: a device-resident 2-D tensor updated by staged runs of writes.

"Model Runner V2 设计文档", section "4. StagedWriteTensor": the tensor (block tables,
for instance) stays on the GPU; the host stages only the changed runs, packs them into
one contiguous buffer, copies that buffer in one host-to-device copy and launches one
kernel that applies them. No full copy of the tensor and no host-device synchronisation.

Merging and packing run in the library's native host code (pa_staged_pack), straight
into a pinned buffer; the apply is the CUDA kernel behind pa_staged_write_apply. This
module only collects the staged writes and passes pointers."""
from __future__ import annotations

from typing import List, Optional, Tuple

import numpy as np
import torch

from . import (PaStagedLayout, PagedAttentionError, pa_staged_pack, pa_staged_pack_bound,
               pa_staged_upload_apply)

_NP = {torch.int32: np.int32, torch.float32: np.float32, torch.int64: np.int64,
       torch.int16: np.int16, torch.uint8: np.uint8, torch.float64: np.float64}


Layout = PaStagedLayout


def pack(rows, starts, lens, values, elem_bytes: int, out: Optional[np.ndarray] = None):
    """Native merge + pack of staged writes (numpy arrays, staging order). Returns the
    packed bytes (a view of `out` when given) and the layout."""
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    need = pa_staged_pack_bound(len(lens), int(lens.sum()) if len(lens) else 0, elem_bytes)
    if out is None or out.nbytes < need:
        out = np.empty(max(need, 16), dtype=np.uint8)
    lay = pa_staged_pack(rows, starts, lens, values, elem_bytes, out)
    return out[:lay.bytes], lay


def unpack(buf: np.ndarray, lay: Layout, dtype) -> List[Tuple[int, int, np.ndarray]]:
    """The runs of a packed buffer as (row, start, values) (for tests and inspection)."""
    W = lay.num_writes
    rows = buf[lay.rows_offset:lay.rows_offset + 4 * W].view(np.int32)
    starts = buf[lay.starts_offset:lay.starts_offset + 4 * W].view(np.int32)
    offs = buf[lay.offsets_offset:lay.offsets_offset + 4 * (W + 1)].view(np.int32)
    vals = buf[lay.values_offset:].view(dtype)
    return [(int(rows[k]), int(starts[k]), vals[offs[k]:offs[k + 1]]) for k in range(W)]


class _Slot:
    """One pinned host buffer, its device copy target, and the event of its last copy."""

    def __init__(self, nbytes: int, device):
        self.host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        self.host_np = self.host.numpy()
        self.dev = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.copied: Optional[torch.cuda.Event] = None


class StagedWriteTensor:
    """A [rows, cols] tensor on the GPU with host-staged run writes.

    stage_write(row, start, values) records one run; stage_writes(rows, starts, values,
    lens) records many from arrays. apply_write() merges and packs them natively into a
    pinned buffer, copies it to the device in one copy and applies it with one kernel
    launch on `stream` (one native call for both). Neither call waits for the GPU: the
    packed buffers form a ring of RING slots, and a slot is reused only once the copy it
    last fed has ended (a wait that happens only when the ring wraps faster than the
    GPU consumes it)."""

    RING = 3

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
        self._clear()
        self._slots: List[Optional[_Slot]] = [None] * self.RING
        self._next = 0
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=self.gpu.device)
        self.last_h2d_bytes = 0

    def _clear(self):
        self._rows, self._starts, self._lens, self._vals = [], [], [], []

    def stage_write(self, row: int, start: int, value) -> None:
        v = np.array(value, dtype=self._np).reshape(-1)
        self._rows.append(np.array([row], np.int32))
        self._starts.append(np.array([start], np.int32))
        self._lens.append(np.array([v.size], np.int32))
        self._vals.append(v)

    def stage_writes(self, rows, starts, values, lens=None) -> None:
        """Many runs at once, in order: run k writes lens[k] values (default 1 each) taken
        in turn from `values`."""
        rows = np.asarray(rows, np.int32).reshape(-1)
        lens = (np.ones(rows.size, np.int32) if lens is None
                else np.asarray(lens, np.int32).reshape(-1))
        self._rows.append(rows)
        self._starts.append(np.asarray(starts, np.int32).reshape(-1))
        self._lens.append(lens)
        self._vals.append(np.asarray(values, dtype=self._np).reshape(-1))

    def apply_write(self, stream=None) -> None:
        if not self._rows:
            return
        one = len(self._rows) == 1
        rows = self._rows[0] if one else np.concatenate(self._rows)
        starts = self._starts[0] if one else np.concatenate(self._starts)
        lens = self._lens[0] if one else np.concatenate(self._lens)
        vals = self._vals[0] if one else np.concatenate(self._vals)
        self._clear()
        eb = self.gpu.element_size()
        need = pa_staged_pack_bound(len(rows), int(lens.sum()), eb)
        k = self._next
        self._next = (k + 1) % self.RING
        slot = self._slots[k]
        if slot is None or slot.host.numel() < need:
            slot = self._slots[k] = _Slot(max(need, 4096), self.gpu.device)
        elif slot.copied is not None:
            slot.copied.synchronize()  # its last copy must have read the pinned buffer
        lay = pa_staged_pack(rows, starts, lens, vals, eb, slot.host_np)
        s = stream if stream is not None else torch.cuda.current_stream(self.gpu.device)
        pa_staged_upload_apply(self.gpu, slot.host, slot.dev, lay, dev_err=self.dev_err,
                               stream=s)
        if slot.copied is None:
            slot.copied = torch.cuda.Event()
        slot.copied.record(s)
        self.last_h2d_bytes = lay.bytes
