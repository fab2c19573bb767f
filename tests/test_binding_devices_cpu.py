"""The binding refuses, before any launch, tensors that are not on one CUDA device equal
to the current one, and a stream of another device (a kernel handed another device's
pointers would fault). Checked with stand-in tensors and streams: no GPU is needed."""
from types import SimpleNamespace

import pytest
import torch

import paged_kv_cache_107_gb300 as pk


def fake(dev):
    return SimpleNamespace(device=torch.device(dev))


@pytest.fixture
def current_is_0(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)


def test_one_device_accepts_the_current_device(current_is_0):
    pk._one_device(fake("cuda:0"), fake("cuda:0"), None, fake("cuda"))
    pk._one_device(fake("cuda:0"), stream=fake("cuda:0"))


@pytest.mark.parametrize("devs", [("cuda:0", "cuda:1"), ("cuda:0", "cpu"), ("cpu",)])
def test_one_device_rejects_mixed_or_host_tensors(current_is_0, devs):
    with pytest.raises(pk.PagedAttentionError):
        pk._one_device(*[fake(d) for d in devs])


def test_one_device_rejects_another_current_device(current_is_0):
    with pytest.raises(pk.PagedAttentionError, match="current device"):
        pk._one_device(fake("cuda:1"), fake("cuda:1"))


def test_one_device_rejects_a_stream_of_another_device(current_is_0):
    with pytest.raises(pk.PagedAttentionError, match="stream"):
        pk._one_device(fake("cuda:0"), stream=fake("cuda:3"))


def test_entry_points_refuse_host_tensors_before_loading_anything():
    """The public calls check their tensors before touching the library or CUDA."""
    x = torch.zeros(4, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(2, 16, 8, 128, dtype=torch.bfloat16)
    i32 = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(pk.PagedAttentionError):
        pk.pa_store_kvcache(x, x, kc, kc, i32)
    with pytest.raises(pk.PagedAttentionError):
        pk.pa_decode(torch.zeros(4, 16, 128, dtype=torch.bfloat16),
                     torch.zeros(4, 16, 128, dtype=torch.bfloat16), kc, kc,
                     torch.zeros(4, 1, dtype=torch.int32), i32)
