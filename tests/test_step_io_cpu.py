"""Layout of DecodeStepBuffers (host side; the pinned buffer needs no GPU to be described):
every input is a view at a 256-byte aligned offset, the views do not overlap and they hold
exactly the tensors' bytes."""
import pytest
import torch

from paged_kv_cache_107_gb300.step_io import DecodeStepBuffers


def test_offsets_aligned_and_disjoint(monkeypatch):
    # avoid pinning and device allocation on a machine without a GPU
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)
    real_empty = torch.empty

    def cpu_empty(*a, **kw):
        kw.pop("device", None)
        return real_empty(*a, **kw)
    monkeypatch.setattr(torch, "empty", cpu_empty)
    io = DecodeStepBuffers(256, 16, 8, 128, 8)
    spans = []
    for name, (shape, dt) in io.spec.items():
        off = io.offsets[name]
        assert off % 256 == 0
        n = 1
        for s in shape:
            n *= s
        size = n * torch.tensor([], dtype=dt).element_size()
        spans.append((off, off + size))
        assert tuple(io.host[name].shape) == shape and io.host[name].dtype == dt
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] == io.nbytes
    io.host["context_lens"].fill_(7)
    assert int(io.host_buf[io.offsets["context_lens"]:io.offsets["context_lens"] + 4].view(torch.int32)[0]) == 7
