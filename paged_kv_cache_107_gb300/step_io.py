"""Decode-step inputs staged in one pinned host buffer and moved with one copy.

The decode step ("3.6 ModelRunner、CUDA Graph 与性能基准", section 5: the step's inputs are
copied into static device buffers, then the captured graph replays) needs q, the new
tokens' K and V, slot_mapping, block_tables and context_lens on the device. Staging them
in one pinned host buffer whose layout matches one device buffer turns the step's six
host-to-device copies into one; the device tensors are views into that buffer, so they
can be handed to pa_decode_step (and captured in a CUDA graph) as they are."""
from __future__ import annotations

from typing import Dict, Tuple

import torch

_ALIGN = 256


class DecodeStepBuffers:
    """Pinned host views (`host[name]`) and device views (`dev[name]`) of one packed buffer
    holding q [B, H, D], k_new / v_new [B, Hk, D], slots [B], block_tables [B, maxb] and
    context_lens [B]. Fill the host views, call upload(stream), run the step on the device
    views."""

    def __init__(self, num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                 max_blocks: int, dtype: torch.dtype = torch.bfloat16, device="cuda"):
        B, H, Hk, D = num_seqs, num_heads, num_kv_heads, head_dim
        self.spec: Dict[str, Tuple[Tuple[int, ...], torch.dtype]] = {
            "q": ((B, H, D), dtype), "k_new": ((B, Hk, D), dtype), "v_new": ((B, Hk, D), dtype),
            "slot_mapping": ((B,), torch.int32), "block_tables": ((B, max_blocks), torch.int32),
            "context_lens": ((B,), torch.int32)}
        self.offsets = {}
        off = 0
        for name, (shape, dt) in self.spec.items():
            off = (off + _ALIGN - 1) // _ALIGN * _ALIGN
            self.offsets[name] = off
            n = 1
            for s in shape:
                n *= s
            off += n * torch.tensor([], dtype=dt).element_size()
        self.nbytes = off
        self.host_buf = torch.empty(self.nbytes, dtype=torch.uint8).pin_memory()
        self.dev_buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.host = {n: self._view(self.host_buf, n) for n in self.spec}
        self.dev = {n: self._view(self.dev_buf, n) for n in self.spec}

    def _view(self, buf: torch.Tensor, name: str) -> torch.Tensor:
        shape, dt = self.spec[name]
        n = 1
        for s in shape:
            n *= s
        size = n * torch.tensor([], dtype=dt).element_size()
        off = self.offsets[name]
        return buf[off:off + size].view(dt).view(shape)

    def upload(self, stream=None) -> None:
        """One asynchronous host-to-device copy of every input of the step."""
        s = stream if stream is not None else torch.cuda.current_stream(self.dev_buf.device)
        with torch.cuda.stream(s):
            self.dev_buf.copy_(self.host_buf, non_blocking=True)
