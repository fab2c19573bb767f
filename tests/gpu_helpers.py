"""Shared plumbing for the GPU parity tests: move a workload to the device, run the
library through its C ABI, compute the oracle on the same inputs, compare."""
import numpy as np
import torch

import oracle
import paged_kv_cache_107_gb300 as pk

# |o - ref| <= ATOL + RTOL * |ref| for bf16 attention with fp32 accumulation
ATOL = 1e-2
RTOL = 1e-2


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a, dtype=torch.bfloat16):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


class DeviceCase:
    def __init__(self, case, device="cuda"):
        self.case = case
        self.dev = torch.device(device)
        self.k_cache = case.k_cache.to(self.dev)
        self.v_cache = case.v_cache.to(self.dev)
        self.q = case.q.to(self.dev)
        self.k_new = case.k_new.to(self.dev)
        self.v_new = case.v_new.to(self.dev)
        self.slots = torch.from_numpy(case.slot_mapping).to(self.dev)
        self.bt = torch.from_numpy(case.block_tables).to(self.dev)
        self.ctx = torch.from_numpy(case.context_lens).to(self.dev)
        if case.is_prefill:
            self.cu_q = torch.from_numpy(case.cu_seqlens_q).to(self.dev)
            self.cu_k = torch.from_numpy(case.cu_seqlens_k).to(self.dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)

    def store(self):
        pk.pa_store_kvcache(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slots,
                            dev_err=self.err)

    def decode(self, grid_ctas=0, workspace=None):
        out = torch.full_like(self.q, float("nan"))
        pk.pa_decode(out, self.q, self.k_cache, self.v_cache, self.bt, self.ctx,
                     grid_ctas=grid_ctas, workspace=workspace, dev_err=self.err)
        return out

    def prefill(self):
        out = torch.full_like(self.q, float("nan"))
        c = self.case
        pk.pa_prefill_varlen(out, self.q, self.k_cache, self.v_cache, self.bt, self.cu_q,
                             self.cu_k, c.max_seqlen_q, c.max_seqlen_k, causal=c.causal,
                             dev_err=self.err)
        return out

    def dev_err(self):
        torch.cuda.synchronize()
        return int(self.err.item())


def oracle_after_store(case):
    """The oracle's own store of the new tokens into a host copy of the cache."""
    ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    return ok, ov


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bad = ~(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} outside {ATOL}+{RTOL}|ref|; first {idx.tolist()}: "
            f"got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}; max abs err "
            f"{np.nanmax(np.abs(got - ref))}")


def to_f64(t):
    return t.float().cpu().double().numpy()
