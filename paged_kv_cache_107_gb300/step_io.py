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


class DecodeStepPipeline:
    """Decode steps whose host<->device copies overlap the neighbouring steps' compute.

    `depth` sets of DecodeStepBuffers and output buffers are used in turn. Step i's inputs
    move in on an upload stream while step i-1 computes, and its output moves out on a
    download stream while step i+1 computes; CUDA events keep each buffer's uses in order
    (a slot's device inputs are overwritten only after the step that read them finished,
    its device output only after the copy that read it out finished, its pinned host
    inputs only after their upload finished).

        pipe = DecodeStepPipeline(B, H, Hk, D, max_blocks)
        for i in range(n):
            views = pipe.inputs(i)       # pinned host views of step i's inputs
            ...fill views...
            pipe.submit(i, run)          # run(dev_views, out) launches step i
            ...
            host_out = pipe.output(i)    # step i's output on the host (waits for it)
    """

    def __init__(self, num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                 max_blocks: int, dtype: torch.dtype = torch.bfloat16, device="cuda",
                 depth: int = 2, compute_stream=None):
        if depth < 2:
            raise ValueError("a pipeline needs at least two buffer sets")
        self.depth = depth
        self.device = torch.device(device)
        self.bufs = [DecodeStepBuffers(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks,
                                       dtype=dtype, device=device) for _ in range(depth)]
        shape = (num_seqs, num_heads, head_dim)
        self.out_dev = [torch.empty(shape, dtype=dtype, device=device) for _ in range(depth)]
        self.out_host = [torch.empty(shape, dtype=dtype).pin_memory() for _ in range(depth)]
        self.compute = (compute_stream if compute_stream is not None
                        else torch.cuda.current_stream(self.device))
        self.up = torch.cuda.Stream(self.device)
        self.down = torch.cuda.Stream(self.device)
        self.uploaded = [torch.cuda.Event() for _ in range(depth)]
        self.computed = [torch.cuda.Event() for _ in range(depth)]
        self.downloaded = [torch.cuda.Event() for _ in range(depth)]
        self.used = [False] * depth
        self.h2d_bytes = self.bufs[0].nbytes
        self.d2h_bytes = self.out_host[0].numel() * self.out_host[0].element_size()

    def inputs(self, i: int) -> Dict[str, torch.Tensor]:
        """Pinned host views of step i's inputs, free to be written."""
        k = i % self.depth
        if self.used[k]:
            self.uploaded[k].synchronize()
        return self.bufs[k].host

    def start_after(self, event) -> None:
        """Make the copy streams wait for `event` (e.g. the start of a timed region)."""
        self.up.wait_event(event)
        self.down.wait_event(event)

    def submit(self, i: int, run) -> None:
        """Upload step i's inputs, run it, and copy its output back, all asynchronously."""
        k = i % self.depth
        b = self.bufs[k]
        if self.used[k]:
            self.up.wait_event(self.computed[k])         # the last step that read these inputs
        with torch.cuda.stream(self.up):
            b.dev_buf.copy_(b.host_buf, non_blocking=True)
        self.uploaded[k].record(self.up)
        self.compute.wait_event(self.uploaded[k])
        if self.used[k]:
            self.compute.wait_event(self.downloaded[k])  # the last copy out of this output
        with torch.cuda.stream(self.compute):
            run(b.dev, self.out_dev[k])
        self.computed[k].record(self.compute)
        self.down.wait_event(self.computed[k])
        with torch.cuda.stream(self.down):
            self.out_host[k].copy_(self.out_dev[k], non_blocking=True)
        self.downloaded[k].record(self.down)
        self.used[k] = True

    def output(self, i: int) -> torch.Tensor:
        """Step i's output in pinned host memory (valid until step i + depth is submitted)."""
        k = i % self.depth
        self.downloaded[k].synchronize()
        return self.out_host[k]

    def join(self, stream=None) -> None:
        """Make `stream` (default: the compute stream) wait for every submitted copy."""
        s = stream if stream is not None else self.compute
        for k in range(self.depth):
            if self.used[k]:
                s.wait_event(self.uploaded[k])
                s.wait_event(self.downloaded[k])
