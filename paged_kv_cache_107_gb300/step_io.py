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
    move in on an upload stream while earlier steps compute, and its output moves out on a
    download stream while later steps compute; CUDA events keep each buffer's uses in order
    (a slot's device inputs are overwritten only after the step that read them finished,
    its device output only after the copy that read it out finished, its pinned host
    inputs only after their upload finished).

    With group = g > 1 the steps are issued g at a time: the g uploads, then the g steps
    back to back on the compute stream behind one event wait, then the g downloads. Inside
    a group the steps follow each other directly, so each decode launch starts as the one
    before it drains (dependent launches); an event wait between every two steps would
    stop that. depth must hold two groups.

        pipe = DecodeStepPipeline(B, H, Hk, D, max_blocks)
        for i in range(n):
            views = pipe.inputs(i)       # pinned host views of step i's inputs
            ...fill views...
            pipe.submit(i, run)          # run(dev_views, out) launches step i
            ...
        pipe.flush()                     # issue a last, partial group
        host_out = pipe.output(i)        # step i's output on the host (waits for it)
    """

    def __init__(self, num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                 max_blocks: int, dtype: torch.dtype = torch.bfloat16, device="cuda",
                 depth: int = 2, compute_stream=None, group: int = 1):
        if group < 1 or depth < 2 * group:
            raise ValueError("a pipeline needs room for two groups of steps")
        self.depth = depth
        self.group = group
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
        # per slot: the events of the last group that used it
        self.uploaded = [None] * depth
        self.computed = [None] * depth
        self.downloaded = [None] * depth
        self.pending = []  # (step, run) submitted but not yet issued
        self.h2d_bytes = self.bufs[0].nbytes
        self.d2h_bytes = self.out_host[0].numel() * self.out_host[0].element_size()

    def inputs(self, i: int) -> Dict[str, torch.Tensor]:
        """Pinned host views of step i's inputs, free to be written."""
        k = i % self.depth
        if self.uploaded[k] is not None:
            self.uploaded[k].synchronize()
        return self.bufs[k].host

    def start_after(self, event) -> None:
        """Make the copy streams wait for `event` (e.g. the start of a timed region)."""
        self.up.wait_event(event)
        self.down.wait_event(event)

    def submit(self, i: int, run) -> None:
        """Queue step i (its upload, its launch by run(dev_views, out), its download); a
        full group is issued at once, asynchronously."""
        self.pending.append((i, run))
        if len(self.pending) == self.group:
            self.flush()

    def flush(self) -> None:
        """Issue the queued steps (a group, or fewer at the end)."""
        if not self.pending:
            return
        slots = [i % self.depth for i, _ in self.pending]
        # uploads: each slot's device inputs are free once the step that last read them ran
        for e in {id(self.computed[k]): self.computed[k] for k in slots
                  if self.computed[k] is not None}.values():
            self.up.wait_event(e)
        with torch.cuda.stream(self.up):
            for k in slots:
                self.bufs[k].dev_buf.copy_(self.bufs[k].host_buf, non_blocking=True)
        up_ev = torch.cuda.Event()
        up_ev.record(self.up)
        # the steps, back to back behind one wait (and the last copies out of their outputs)
        self.compute.wait_event(up_ev)
        for e in {id(self.downloaded[k]): self.downloaded[k] for k in slots
                  if self.downloaded[k] is not None}.values():
            self.compute.wait_event(e)
        with torch.cuda.stream(self.compute):
            for i, run in self.pending:
                k = i % self.depth
                run(self.bufs[k].dev, self.out_dev[k])
        comp_ev = torch.cuda.Event()
        comp_ev.record(self.compute)
        # downloads
        self.down.wait_event(comp_ev)
        with torch.cuda.stream(self.down):
            for k in slots:
                self.out_host[k].copy_(self.out_dev[k], non_blocking=True)
        down_ev = torch.cuda.Event()
        down_ev.record(self.down)
        for k in slots:
            self.uploaded[k], self.computed[k], self.downloaded[k] = up_ev, comp_ev, down_ev
        self.pending = []

    def output(self, i: int) -> torch.Tensor:
        """Step i's output in pinned host memory (valid until step i + depth is submitted);
        issues the queued steps first if step i is among them."""
        if any(j == i for j, _ in self.pending):
            self.flush()
        k = i % self.depth
        self.downloaded[k].synchronize()
        return self.out_host[k]

    def join(self, stream=None) -> None:
        """Issue the queued steps and make `stream` (default: the compute stream) wait for
        every submitted copy."""
        self.flush()
        s = stream if stream is not None else self.compute
        for e in {id(x): x for x in self.uploaded + self.downloaded if x is not None}.values():
            s.wait_event(e)
