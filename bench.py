#!/usr/bin/env python3
"""Benchmark of the paged-KV decode step on GB300.

One step = one pass of the hot path over one batch: the store of every sequence's new
token into the paged cache, then paged GQA decode attention over context_lens that
include it (split across CTAs, partials combined in-kernel). The timed step is the fused
call pa_decode_step (store and attention in one launch); the same step as two launches
(pa_store_kvcache, then pa_decode) is timed beside it. The default workload is the
Qwen3-0.6B-shaped decode step: B=256, context U{100..2048}, H=16, H_kv=8, D=128,
block_size=256, a 4096-block pool, bf16.

Metric: effective KV-read GB/s of the step (sum over sequences of context*H_kv*D*2*2
bytes, divided by the step time), with seqs/s beside it. Inputs are larger than L2
(about 1.1 GB of K/V per step), so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torch.distributed.run: every rank runs its own replica of the
workload (weak scaling); there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn: effective KV-read GB/s (% of GB300 HBM peak), seqs/s"
NOMINAL_HBM_GBS = 8000.0
E2E_GROUP = 5  # end-to-end leg: decode steps issued together (their copies batched)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def burst_bf16_peak():
    """The measured burst bf16 dense rate (a kernel timed alone), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def source_sha256(*names) -> str:
    """sha256 over the named csrc/ files, in order (the kernel and the headers it uses)."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_107_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


DECODE_SOURCES = ("decode_kernel.cuh", "pa_device.cuh")
DECODE_TC_SOURCES = ("decode_tc.cuh", "decode_kernel.cuh", "pa_device.cuh")
PREFILL_SOURCES = ("prefill_kernel.cuh", "prefill.cu", "umma.cuh", "pa_device.cuh", "tensor_map.cu",
                   "tensor_map.h")
STORE_SOURCES = ("store.cu", "pa_device.cuh")


def profile_value(sources, summary: str, key: str):
    """A number recorded as `key: value` in a committed ncu summary, if the summary was
    taken on the current kernel sources (sha256 recorded in it); otherwise None."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_v = re.search(re.escape(key) + r":\s*([0-9.eE+]+)", text)
        if m_sha and m_v and m_sha.group(1) == source_sha256(*sources):
            return float(m_v.group(1))
    except OSError:
        pass
    return None


SAMPLER_SOURCES = ("sample.cu", "pa_device.cuh")
# ncu summaries of the fused decode step, by workload
STEP_PROFILES = {"w2_qwen3_decode_b256": "decode_step_w2_qwen3_b256.md",
                 "w3_long_context_b8": "decode_tc_w3_long_context_b8.md"}


def kernel_traffic(sources, summary: str, workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if that summary was taken on the
    current kernel sources (sha256 recorded in it), on this workload and of this kernel
    (its `workload:` and `kernel:` lines); otherwise None."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
        sha = source_sha256(*sources)
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
        m_w = re.search(r"^workload:\s*(\S+)\s*$", text, re.M)
        m_k = re.search(r"^kernel:\s*(\S+)\s*$", text, re.M)
        if (m_sha and m_b and m_w and m_k and m_sha.group(1) == sha
                and m_w.group(1) == workload and m_k.group(1) == kernel):
            return float(m_b.group(1))
    except OSError:
        pass
    return None


def decode_step_kernel(num_heads: int, num_kv_heads: int, head_dim: int) -> str:
    """Which kernel runs the fused decode step for this shape (the routing rule of the
    library's launcher: the CUDA-core kernel for 1-2 query heads per KV head at head_dim
    128 when one head slab holds every KV head, the tensor-core kernel otherwise)."""
    g = num_heads // num_kv_heads
    one_slab = num_kv_heads in (1, 2, 4, 8)
    if g >= 3 or not (head_dim == 128 and one_slab):
        return "paged_decode_tc_kernel/fused"
    return "paged_decode_kernel/fused"


def decode_step_sources(kernel: str):
    return DECODE_TC_SOURCES if kernel.startswith("paged_decode_tc_kernel") else DECODE_SOURCES


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed region.

    Polls NVML (read-only queries through the driver's libnvidia-ml) from a thread about
    every millisecond, so even a timed region of a few milliseconds gets samples; falls
    back to `nvidia-smi -lms 200` when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []
        self.reason_bits = 0
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self.source = "none"

    def _nvml_handle(self):
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        handle = ctypes.c_void_p()
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
        except Exception:
            uuid = None
        ok = False
        if uuid:
            for cand in (uuid, "GPU-" + uuid):
                if nv.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(handle)) == 0:
                    ok = True
                    break
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle)) != 0:
            raise OSError("no NVML handle")
        return nv, handle

    def __enter__(self):
        import ctypes
        import threading
        try:
            nv, h = self._nvml_handle()
        except OSError:
            return self._start_smi()
        self.source = "nvml"
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or getattr(
            nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._stop = threading.Event()

        def poll():
            clk = ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            while not self._stop.is_set():
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    self.samples.append(float(clk.value))
                if get_reasons(h, ctypes.byref(rs)) == 0:
                    self.reason_bits |= int(rs.value)
                self._stop.wait(0.001)

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        return self

    def _start_smi(self):
        self.source = "nvidia-smi"
        self.out_path = f"/tmp/pa_clocks_{os.getpid()}.csv"
        try:
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.source = "none"
        return self

    def __exit__(self, *exc):
        if self.source == "nvml":
            self._stop.set()
            self._thread.join(timeout=2)
        elif self.source == "nvidia-smi":
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40,
                    "sw_thermal_slowdown": 0x20, "sw_power_cap": 0x4}
            for line in open(self.out_path):
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    continue
                for n, v in zip(names, parts[2:6]):
                    if v.lower().startswith("active"):
                        self.reason_bits |= bits[n]
            os.unlink(self.out_path)

    def summary(self):
        reasons = sorted(n for b, n in self.REASONS.items() if self.reason_bits & b)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
                "source": self.source}


def dist_setup(n_gpus: int):
    import torch
    if n_gpus <= 1 and "WORLD_SIZE" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_summary(case):
    tot_ctx = case.total_context()
    kv_bytes = tot_ctx * case.num_kv_heads * case.head_dim * 2 * 2
    qo_bytes = case.num_seqs * case.num_heads * case.head_dim * 2 * 2
    meta_bytes = case.block_tables.nbytes + case.context_lens.nbytes
    store_bytes = int((case.slot_mapping >= 0).sum()) * case.num_kv_heads * case.head_dim * 2 * 2 * 2
    return tot_ctx, kv_bytes, qo_bytes + meta_bytes, store_bytes


def oracle_store(case):
    import oracle
    t0 = time.perf_counter()
    ok, ov = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                  case.slot_mapping)
    return ok, ov, time.perf_counter() - t0


def cpu_baseline(case, seconds: float = 10.0, threads: int = 0, stored=None):
    """Time the fp64 oracle (as it stands) on a bounded sample of the workload: whole
    sequences, all heads, until about `seconds` of CPU time has passed."""
    import numpy as np
    import oracle
    cores = oracle.max_threads(threads)
    # the store of the step (once), then decode over consecutive sequences of the batch
    ok, ov, t_store = stored if stored is not None else oracle_store(case)
    done_seqs, done_ctx, t_dec = 0, 0, 0.0
    H = case.num_heads
    chunk = 8
    b = 0
    while t_dec < seconds:
        if b >= case.num_seqs:
            b = 0  # whole batch done: go round again until the time budget is used
        sel = list(range(b, min(b + chunk, case.num_seqs)))
        pairs = np.array([s * H + h for s in sel for h in range(H)], np.int64)
        t0 = time.perf_counter()
        oracle.decode(case.q, ok, ov, case.block_tables, case.context_lens, pairs=pairs,
                      nthreads=threads)
        t_dec += time.perf_counter() - t0
        done_seqs += len(sel)
        done_ctx += int(case.context_lens[sel].astype(np.int64).sum())
        b += chunk
    kv = done_ctx * case.num_kv_heads * case.head_dim * 4
    return {"seqs_per_s": done_seqs / t_dec, "gbs": kv / t_dec / 1e9, "cores": cores,
            "sample": f"{done_seqs} sequence-passes over the {case.num_seqs}-sequence batch (all {H} heads), "
                      f"{done_ctx} context tokens, fp64 oracle, {t_dec:.1f} s decode + "
                      f"{t_store:.1f} s store of the step on the host"}


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores (no reference implementation
    exists to install). Only rank 0 works."""
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    from paged_kv_cache_107_gb300 import workloads
    case = workloads.workload(args.workload, poison=False)
    tot_ctx, kv_bytes, _, _ = workload_summary(case)
    vals = []
    base = None
    stored = oracle_store(case)
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(case, seconds=args.ref_seconds, stored=stored)
        if i >= args.warmup:
            vals.append(r["gbs"])
            base = r
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": kv_bytes / (v * 1e9) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "num_seqs": case.num_seqs,
                   "total_context_tokens": tot_ctx},
        "seqs_per_s": base["seqs_per_s"],
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": base["cores"], "kind": "oracle",
                         "sample": base["sample"]},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


def prefill_flops(case) -> float:
    """4*H*D per unmasked (query, key) pair: sum over sequences of sum_i (c_s + i + 1)."""
    import numpy as np
    n = np.diff(case.cu_seqlens_q).astype(np.float64)
    k = np.diff(case.cu_seqlens_k).astype(np.float64)
    c = k - n
    if case.causal:
        pairs = float(np.sum(n * c + n * (n + 1) / 2))
    else:
        pairs = float(np.sum(n * k))
    return 4.0 * case.num_heads * case.head_dim * pairs


def prefill_cpu_baseline(case, seconds: float, threads: int = 0, stored=None):
    """Time the fp64 oracle's prefill (as it stands) on a bounded sample of the chunked
    prefill: (query token, head) rows in a seeded random order, in chunks, until about
    `seconds` of wall time has passed. FLOPs count 4*D per unmasked (row, key) pair, as
    the GPU figure does."""
    import numpy as np
    import oracle
    cores = oracle.max_threads(threads)
    ok, ov = stored if stored is not None else oracle.store_kvcache(
        case.k_new, case.v_new, case.k_cache, case.v_cache, case.slot_mapping)
    H, D = case.num_heads, case.head_dim
    n = np.diff(case.cu_seqlens_q).astype(np.int64)
    c = np.diff(case.cu_seqlens_k).astype(np.int64) - n
    seq_of_tok = np.repeat(np.arange(len(n)), n)
    keys_of_tok = c[seq_of_tok] + (np.arange(int(n.sum())) - np.repeat(case.cu_seqlens_q[:-1], n)) + 1
    if not case.causal:
        keys_of_tok = (c + n)[seq_of_tok]
    order = np.random.default_rng(107005).permutation(int(n.sum()) * H)
    chunk = 1024 if threads != 1 else 64
    done_rows, done_pairs, t = 0, 0, 0.0
    kb = ok.view(np.uint16)
    vb = ov.view(np.uint16)
    while t < seconds and done_rows < len(order):
        rows = np.sort(order[done_rows:done_rows + chunk])
        t0 = time.perf_counter()
        oracle.prefill(case.q, kb, vb, case.block_tables, case.cu_seqlens_q, case.cu_seqlens_k,
                       causal=case.causal, rows=rows, nthreads=threads)
        t += time.perf_counter() - t0
        done_rows += len(rows)
        done_pairs += int(keys_of_tok[rows // H].sum())
    flops = 4.0 * D * done_pairs
    return {"tokens_per_s": done_rows / H / t, "gflops": flops / t / 1e9, "cores": cores,
            "sample": f"{done_rows} (query token, head) rows of the {int(n.sum())}-token "
                      f"chunk in a seeded random order ({done_pairs} unmasked row-key pairs), "
                      f"fp64 oracle, {t:.1f} s"}


def measure_prefill(dev, steps: int, warmup: int, pool_blocks=None, head_dim=128, dtype=None,
                    cpu_seconds: float = 0.0):
    """Chunked-prefill step of workload 5: store of every new token, then causal prefill.
    Returns timings (CUDA events on the stream), TFLOP/s and the fraction of the measured
    bf16 tensor peak, burst (the prefill is timed alone, launch by launch) and sustained
    (fp16 has the same dense tensor rate). With cpu_seconds > 0 the fp64 oracle's prefill is
    timed beside it on the host cores (all of them, then one thread)."""
    import torch
    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300 import workloads
    case = workloads.workload(5, poison=True, num_blocks=pool_blocks, head_dim=head_dim,
                              dtype=dtype or torch.bfloat16)
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    q, kn, vn = case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev)
    slots = torch.from_numpy(case.slot_mapping).to(dev)
    bt = torch.from_numpy(case.block_tables).to(dev)
    cu_q = torch.from_numpy(case.cu_seqlens_q).to(dev)
    cu_k = torch.from_numpy(case.cu_seqlens_k).to(dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def store():
        pk.pa_store_kvcache(kn, vn, kc, vc, slots, dev_err=err, stream=stream)

    def prefill():
        pk.pa_prefill_varlen(out, q, kc, vc, bt, cu_q, cu_k, case.max_seqlen_q, case.max_seqlen_k,
                             causal=True, dev_err=err, stream=stream)

    for _ in range(max(warmup, 3)):
        store()
        prefill()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for e0, e1, e2 in ev:
        e0.record(stream)
        store()
        e1.record(stream)
        prefill()
        e2.record(stream)
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in prefill")
    st_ms = statistics.median(a.elapsed_time(b) for a, b, _ in ev)
    pf_ms = statistics.median(b.elapsed_time(c) for _, b, c in ev)
    flops = prefill_flops(case)
    _, tflops_peak, src = measured_peaks()
    tflops_burst, bsrc = burst_bf16_peak()
    nq = int(case.cu_seqlens_q[-1])
    store_bytes = nq * case.num_kv_heads * case.head_dim * 2 * 2 * 2
    res = {"workload": case.name, "new_tokens": nq, "flops": flops,
           "prefill_ms": pf_ms, "store_ms": st_ms,
           "tflops": flops / (pf_ms * 1e-3) / 1e12,
           "tflops_frac": flops / (pf_ms * 1e-3) / 1e12 / tflops_burst,
           "peak_tflops": tflops_burst, "peak_source": f"{bsrc} bf16 dense (burst: the prefill "
                                                       "is timed alone, launch by launch)",
           "tflops_frac_sustained": flops / (pf_ms * 1e-3) / 1e12 / tflops_peak,
           "peak_tflops_sustained": tflops_peak,
           "tokens_per_s": nq / (pf_ms * 1e-3),
           "store_gbs": store_bytes / (st_ms * 1e-3) / 1e9}
    if head_dim == 128 and (dtype is None or dtype == torch.bfloat16):
        hbm_peak, _, hsrc = measured_peaks()
        # the store of the chunk's new tokens: K and V rows read and written once
        res["store_roofline"] = {
            "kernel": "store_kvcache_kernel", "bound": "hbm", "unit": "GB/s",
            "achieved": res["store_gbs"], "peak": hbm_peak, "frac": res["store_gbs"] / hbm_peak,
            "peak_source": f"{hsrc} HBM copy GB/s", "alg_bytes_per_launch": store_bytes,
            "traffic": kernel_traffic(STORE_SOURCES, "store_kvcache_w5_prefill.md", case.name,
                                      "store_kvcache_kernel")}
    if head_dim == 128 and (dtype is None or dtype == torch.bfloat16):
        res["roofline"] = {
            "kernel": "paged_prefill_kernel", "bound": "tensor", "unit": "TFLOP/s",
            "achieved": res["tflops"], "peak": tflops_burst, "frac": res["tflops_frac"],
            "peak_source": f"{bsrc} cuBLAS bf16 dense, burst (kernel timed alone)",
            "frac_of_sustained": res["tflops_frac_sustained"],
            "traffic": kernel_traffic(PREFILL_SOURCES, "prefill_w5_chunked.md", case.name,
                                      "paged_prefill_kernel")}
    if cpu_seconds > 0:
        import oracle
        stored = oracle.store_kvcache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                      case.slot_mapping)
        cb = prefill_cpu_baseline(case, cpu_seconds, stored=stored)
        c1 = prefill_cpu_baseline(case, max(cpu_seconds / 3, 1.0), threads=1, stored=stored)
        res["cpu_baseline"] = {"value": cb["tokens_per_s"], "unit": "tokens/s",
                               "gflops": cb["gflops"], "cores": cb["cores"], "kind": "oracle",
                               "sample": cb["sample"],
                               "single_thread": {"value": c1["tokens_per_s"], "unit": "tokens/s",
                                                 "gflops": c1["gflops"], "cores": c1["cores"],
                                                 "sample": c1["sample"]}}
    return res


def measure_variants(dev, steps: int, warmup: int, only=None, pool_blocks=None):
    """head_dim 64 / IEEE fp16 variants on the shapes of the decode step (workload 2: the
    fused store + decode, one launch) and of the chunked prefill (workload 5); and the
    decode step with 4 and 8 query heads per KV head (the tensor-core path). `only` keeps
    one variant (its tag); `pool_blocks` sizes the decode steps' block pools (at least the
    1229 blocks their tables use) for profiler captures."""
    import torch
    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300 import workloads
    hbm_peak, _, peak_src = measured_peaks()
    res = {"peak_gbs": hbm_peak, "peak_source": f"{peak_src} HBM copy GB/s"}
    for D, dt, tag, heads in ((64, torch.bfloat16, "d64_bf16", 16), (64, torch.float16, "d64_fp16", 16),
                              (128, torch.float16, "d128_fp16", 16), (128, torch.bfloat16, "g4", 32),
                              (128, torch.bfloat16, "g8", 64)):
        if only is not None and tag != only:
            continue
        if heads == 16:
            case = workloads.workload(2, poison=True, num_blocks=pool_blocks, head_dim=D,
                                      dtype=dt)
        else:  # the same lengths and tables with 4 or 8 query heads per KV head
            base = workloads.workload(2, poison=False)
            case = workloads.decode_case(base.context_lens, heads, 8, D, 256,
                                         num_blocks=pool_blocks or 4096,
                                         seed=107002 + 1000, poison=True, max_blocks=8,
                                         name=f"w2_decode_b256_h{heads}_hk8", dtype=dt)
        tot_ctx, kv_bytes, small_bytes, store_bytes = workload_summary(case)
        kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
        q, kn, vn = case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev)
        slots = torch.from_numpy(case.slot_mapping).to(dev)
        bt = torch.from_numpy(case.block_tables).to(dev)
        ctx = torch.from_numpy(case.context_lens).to(dev)
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = pk.DecodeWorkspace(case.num_seqs, case.num_heads, case.num_kv_heads, D, device=dev)
        stream = torch.cuda.current_stream(dev)

        def step():
            pk.pa_decode_step(out, q, kn, vn, kc, vc, slots, bt, ctx, workspace=ws, dev_err=err,
                              stream=stream)

        for _ in range(max(warmup, 3)):
            step()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        # the same steps back to back, no events between them (each launch a dependent of
        # the one before, as in a decode loop)
        lo, hi = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lo.record(stream)
        for _ in range(steps):
            step()
        hi.record(stream)
        torch.cuda.synchronize(dev)
        loop_ms = lo.elapsed_time(hi) / steps
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item())} in the {tag} step")
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        alg = kv_bytes + small_bytes + case.slot_mapping.nbytes + store_bytes // 2
        res["decode_step_" + tag] = {
            "workload": case.name, "step_us": ms * 1e3,
            "kv_gbs": kv_bytes / (ms * 1e-3) / 1e9,
            "achieved_gbs": alg / (ms * 1e-3) / 1e9,
            "frac_of_hbm": alg / (ms * 1e-3) / 1e9 / hbm_peak,
            "alg_bytes_per_launch": alg,
            "loop_step_us": loop_ms * 1e3,
            "loop_kv_gbs": kv_bytes / (loop_ms * 1e-3) / 1e9,
            # back to back, as the headline step loop runs: the same bytes over the loop's
            # time per step (each launch a dependent of the one before)
            "loop_frac_of_hbm": alg / (loop_ms * 1e-3) / 1e9 / hbm_peak}
        summary = {"g8": "decode_tc_g8_w2_b256.md", "d64_bf16": "decode_tc_d64_w2_b256.md"}
        if tag in summary:
            res["decode_step_" + tag]["traffic"] = kernel_traffic(
                DECODE_TC_SOURCES, summary[tag], case.name, "paged_decode_tc_kernel/fused")
        del kc, vc, case
        if heads == 16 and only is None:
            res["prefill_" + tag] = measure_prefill(dev, steps=min(steps, 20), warmup=warmup,
                                                    head_dim=D, dtype=dt)
    if only is None:
        res["decode_step_block_sizes"] = measure_block_sizes(dev, min(steps, 30), warmup)
        res["decode_step_batch_sizes"] = measure_batch_sizes(dev, min(steps, 30), warmup)
    return res


def measure_long_context(dev, steps: int, warmup: int, pool_blocks=None):
    """The long-context split-KV decode step (B=8, context U{32768..131072}, H=32, H_kv=8,
    so 4 query heads per KV head, D=128, block size 256, the 4096-block pool): the fused
    store + decode, one launch at a time (CUDA events per launch, for the roofline) and
    back to back. Only 64 (sequence, KV head) pairs exist, so every sequence is split
    across CTAs and combined in-kernel. K/V bytes (about 2.4 GB) exceed L2: no flush."""
    import torch
    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300 import workloads
    case = workloads.workload(3, poison=True, num_blocks=pool_blocks)
    tot_ctx, kv_bytes, small_bytes, store_bytes = workload_summary(case)
    H, Hk, D = case.num_heads, case.num_kv_heads, case.head_dim
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    q, kn, vn = case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev)
    slots = torch.from_numpy(case.slot_mapping).to(dev)
    bt = torch.from_numpy(case.block_tables).to(dev)
    ctx = torch.from_numpy(case.context_lens).to(dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pk.DecodeWorkspace(case.num_seqs, H, Hk, D, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        pk.pa_decode_step(out, q, kn, vn, kc, vc, slots, bt, ctx, workspace=ws, dev_err=err,
                          stream=stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    lo, hi = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lo.record(stream)
    for _ in range(steps):
        step()
    hi.record(stream)
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the long-context step")
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    loop_ms = lo.elapsed_time(hi) / steps
    hbm_peak, _, peak_src = measured_peaks()
    alg = kv_bytes + small_bytes + case.slot_mapping.nbytes + store_bytes // 2
    kname = decode_step_kernel(H, Hk, D)
    return {
        "workload": case.name, "num_seqs": case.num_seqs, "total_context_tokens": tot_ctx,
        "kv_bytes_per_step": kv_bytes, "step_us": ms * 1e3,
        "kv_gbs": kv_bytes / (ms * 1e-3) / 1e9, "seqs_per_s": case.num_seqs / (ms * 1e-3),
        "loop_step_us": loop_ms * 1e3, "loop_kv_gbs": kv_bytes / (loop_ms * 1e-3) / 1e9,
        "loop_frac_of_hbm": alg / (loop_ms * 1e-3) / 1e9 / hbm_peak,
        "pct_of_nominal_hbm": 100.0 * kv_bytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "roofline": {"kernel": kname, "bound": "hbm", "unit": "GB/s",
                     "achieved": alg / (ms * 1e-3) / 1e9, "peak": hbm_peak,
                     "peak_source": f"{peak_src} HBM copy GB/s",
                     "frac": alg / (ms * 1e-3) / 1e9 / hbm_peak, "alg_bytes_per_launch": alg,
                     "traffic": kernel_traffic(decode_step_sources(kname),
                                               STEP_PROFILES.get(case.name, ""), case.name,
                                               kname)},
        "l2": "K/V read per step (~2.4 GB) >> 129 MB L2; no flush"}


def measure_block_sizes(dev, steps: int, warmup: int):
    """The fused decode step on the decode-step lengths (B=256, ctx U{100..2048}, H=16,
    H_kv=8, D=128) for block sizes 16..256: one launch at a time and back to back. Cache
    contents are made on the device (the parity tests cover these block sizes)."""
    import numpy as np
    import torch
    import paged_kv_cache_107_gb300 as pk
    B, H, Hk, D = 256, 16, 8, 128
    res = {}
    for bs in (16, 32, 64, 128, 256):
        rng = np.random.default_rng(107002)
        lens = rng.integers(100, 2048 + 1, size=B).astype(np.int32)
        nblk = (lens + bs - 1) // bs
        nb = int(nblk.sum())
        perm = rng.permutation(nb).astype(np.int32)
        bt = np.full((B, int(nblk.max())), -1, np.int32)
        o = 0
        for b in range(B):
            bt[b, :nblk[b]] = perm[o:o + nblk[b]]
            o += nblk[b]
        pos = lens - 1
        slots = (bt[np.arange(B), pos // bs].astype(np.int64) * bs + pos % bs).astype(np.int32)
        g = torch.Generator(device=dev)
        g.manual_seed(107002 + bs)
        kc = torch.randn((nb, bs, Hk, D), generator=g, device=dev).to(torch.bfloat16)
        vc = torch.randn((nb, bs, Hk, D), generator=g, device=dev).to(torch.bfloat16)
        q = torch.randn((B, H, D), generator=g, device=dev).to(torch.bfloat16)
        kn = torch.randn((B, Hk, D), generator=g, device=dev).to(torch.bfloat16)
        vn = torch.randn((B, Hk, D), generator=g, device=dev).to(torch.bfloat16)
        sd = torch.from_numpy(slots).to(dev)
        btd = torch.from_numpy(bt).to(dev)
        ctx = torch.from_numpy(lens).to(dev)
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = pk.DecodeWorkspace(B, H, Hk, D, device=dev)
        stream = torch.cuda.current_stream(dev)

        def step():
            pk.pa_decode_step(out, q, kn, vn, kc, vc, sd, btd, ctx, workspace=ws, dev_err=err,
                              stream=stream)

        for _ in range(max(warmup, 3)):
            step()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
        lo, hi = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lo.record(stream)
        for _ in range(steps):
            step()
        hi.record(stream)
        torch.cuda.synchronize(dev)
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item())} at block size {bs}")
        kv = int(lens.sum()) * Hk * D * 2 * 2
        per = statistics.median(a.elapsed_time(b) for a, b in ev)
        loop = lo.elapsed_time(hi) / steps
        res[f"bs{bs}"] = {"step_us": per * 1e3, "loop_step_us": loop * 1e3,
                          "loop_kv_gbs": kv / (loop * 1e-3) / 1e9}
        del kc, vc
    return res


def measure_prefix_sharing(dev, steps: int, warmup: int):
    """The prefix-sharing workload (B=512, lengths lognormal(6, 1) clipped to 1..4096,
    groups of 64 sequences share their first 4 physical blocks, H=16, H_kv=8, D=128) at
    block sizes 16 and 256: the fused decode step timed one launch at a time after an L2
    flush (a read of a 512 MB buffer: a write would leave dirty lines whose write-back
    lands in the timed launch), one launch at a time without the flush (shared blocks may
    then stay in L2 from the step before), and back to back. GB/s are given twice:
    'logical' counts every sequence's K/V rows, 'unique' each physical row once."""
    import torch
    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300 import workloads
    hbm_peak, _, peak_src = measured_peaks()
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)  # 512 MB, read only
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {"peak_gbs": hbm_peak, "peak_source": f"{peak_src} HBM copy GB/s"}
    for bs in (16, 256):
        case = workloads.workload(4, block_size=bs, poison=False)
        tot_ctx, kv_bytes, small_bytes, store_bytes = workload_summary(case)
        Hk, D = case.num_kv_heads, case.head_dim
        rows = {}  # physical block -> rows read from it (the longest reader's share)
        for b in range(case.num_seqs):
            n = int(case.context_lens[b])
            for j in range(-(-n // bs)):
                blk = int(case.block_tables[b, j])
                rows[blk] = max(rows.get(blk, 0), min(bs, n - j * bs))
        uniq_bytes = sum(rows.values()) * Hk * D * 2 * 2
        kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
        q, kn, vn = case.q.to(dev), case.k_new.to(dev), case.v_new.to(dev)
        slots = torch.from_numpy(case.slot_mapping).to(dev)
        bt = torch.from_numpy(case.block_tables).to(dev)
        ctx = torch.from_numpy(case.context_lens).to(dev)
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = pk.DecodeWorkspace(case.num_seqs, case.num_heads, Hk, D, device=dev)

        def step():
            pk.pa_decode_step(out, q, kn, vn, kc, vc, slots, bt, ctx, workspace=ws, dev_err=err,
                              stream=stream)

        def flush_l2():
            torch.amax(flush, dim=0, keepdim=True, out=sink)

        for _ in range(max(warmup, 3)):
            flush_l2()
            step()
        torch.cuda.synchronize(dev)
        times = {}
        for mode in ("flushed", "warm"):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            for a, b in ev:
                if mode == "flushed":
                    flush_l2()
                a.record(stream)
                step()
                b.record(stream)
            torch.cuda.synchronize(dev)
            times[mode] = statistics.median(a.elapsed_time(b) for a, b in ev)
        lo, hi = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lo.record(stream)
        for _ in range(steps):
            step()
        hi.record(stream)
        torch.cuda.synchronize(dev)
        times["loop"] = lo.elapsed_time(hi) / steps
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item())} at block size {bs}")
        entry = {"workload": case.name, "num_seqs": case.num_seqs,
                 "total_context_tokens": tot_ctx, "shared_blocks": case.shared_blocks,
                 "logical_kv_bytes": kv_bytes, "unique_kv_bytes": uniq_bytes}
        for mode, ms in times.items():
            entry[mode] = {"step_us": ms * 1e3,
                           "logical_gbs": kv_bytes / (ms * 1e-3) / 1e9,
                           "unique_gbs": uniq_bytes / (ms * 1e-3) / 1e9,
                           "unique_frac_of_hbm": uniq_bytes / (ms * 1e-3) / 1e9 / hbm_peak}
        res[f"bs{bs}"] = entry
        del kc, vc, case
    del flush
    return res


def fit_stream_and_fixed(points):
    """Least-squares line time = bytes / rate + fixed through (bytes, microseconds) points:
    the streaming rate in GB/s and the fixed cost of a launch in microseconds."""
    import numpy as np
    x = np.array([a for a, _ in points], np.float64)
    y = np.array([b for _, b in points], np.float64)
    slope, icpt = np.polyfit(x, y, 1)  # us per byte, us
    return {"stream_gbs": 1e-3 / slope, "fixed_us": float(icpt)}


def measure_batch_sizes(dev, steps: int, warmup: int):
    """The fused decode step on the first B sequences of the decode-step workload (ctx
    U{100..2048}, H=16, H_kv=8, D=128, bs=256) for B = 1 .. 256: one launch at a time and
    back to back. A least-squares line through (K/V bytes, time) for B >= 16 separates the
    streaming rate from the fixed cost of a launch, which sets the latency of small
    batches."""
    import numpy as np
    import torch
    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300 import workloads
    full = workloads.workload(2, poison=False)
    kc, vc = full.k_cache.to(dev), full.v_cache.to(dev)
    H, Hk, D = full.num_heads, full.num_kv_heads, full.head_dim
    stream = torch.cuda.current_stream(dev)
    res, pts, pts_loop = {}, [], []
    for B in (1, 4, 16, 64, 128, 256):
        q = full.q[:B].to(dev)
        kn, vn = full.k_new[:B].to(dev), full.v_new[:B].to(dev)
        slots = torch.from_numpy(full.slot_mapping[:B].copy()).to(dev)
        bt = torch.from_numpy(full.block_tables[:B].copy()).to(dev)
        ctx = torch.from_numpy(full.context_lens[:B].copy()).to(dev)
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = pk.DecodeWorkspace(B, H, Hk, D, device=dev)

        def step():
            pk.pa_decode_step(out, q, kn, vn, kc, vc, slots, bt, ctx, workspace=ws, dev_err=err,
                              stream=stream)

        for _ in range(max(warmup, 3)):
            step()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
        lo, hi = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lo.record(stream)
        for _ in range(steps):
            step()
        hi.record(stream)
        torch.cuda.synchronize(dev)
        if int(err.item()) != 0:
            raise RuntimeError(f"device error bits {int(err.item())} at batch {B}")
        kv = int(full.context_lens[:B].astype(np.int64).sum()) * Hk * D * 2 * 2
        per = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
        loop = lo.elapsed_time(hi) / steps * 1e3
        res[f"b{B}"] = {"kv_bytes": kv, "step_us": per, "loop_step_us": loop,
                        "kv_gbs": kv / per / 1e3, "loop_kv_gbs": kv / loop / 1e3}
        if B >= 16:
            pts.append((kv, per))
            pts_loop.append((kv, loop))
    for name, p in (("fit_per_launch", pts), ("fit_back_to_back", pts_loop)):
        res[name] = fit_stream_and_fixed(p)
    del kc, vc
    return res


def measure_sampler(dev, steps: int, warmup: int):
    """Gumbel-max sampling of one token per row: B=256 rows of the Qwen3 vocabulary
    (V=151936), fp32 logits N(0, 9), T ~ U[0.3, 1.5], random seeds and offsets. The
    logits rotate over buffers totalling more than L2, so every launch reads from HBM.
    Bytes per launch = the logits read (B*V*4) plus the small per-row inputs/outputs."""
    import numpy as np
    import torch

    import paged_kv_cache_107_gb300 as pk

    B, V = 256, 151936
    rng = np.random.default_rng(107300)
    temps = torch.from_numpy(rng.uniform(0.3, 1.5, size=B).astype(np.float32)).to(dev)
    seeds = torch.from_numpy(rng.integers(0, 2**63, size=B, dtype=np.int64)).to(dev)
    offs = torch.from_numpy(rng.integers(0, 2**40, size=B, dtype=np.int64)).to(dev)
    out = torch.empty(B, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pk.SampleWorkspace(B, device=dev)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, _, peak_src = measured_peaks()
    res = {"workload": "gumbel_sample_b256_v151936", "num_seqs": B, "vocab": V,
           "peak_gbs": hbm_peak, "peak_source": f"{peak_src} HBM copy GB/s"}
    for dtype, name, nbuf in ((torch.float32, "fp32", 3), (torch.bfloat16, "bf16", 5)):
        g = torch.Generator(device=dev)
        g.manual_seed(107300)
        bufs = [(torch.randn((B, V), generator=g, device=dev) * 3).to(dtype) for _ in range(nbuf)]

        def launch(i):
            pk.pa_gumbel_sample(out, bufs[i % nbuf], temps, seeds, offs, workspace=ws,
                                dev_err=err, stream=stream)

        for i in range(max(warmup, 3)):
            launch(i)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            launch(i)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        nbytes = B * V * bufs[0].element_size() + B * (4 + 8 + 8 + 8)
        res[name] = {"kernel_us": ms * 1e3, "bytes_per_launch": nbytes,
                     "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
                     "tokens_per_s": B / (ms * 1e-3)}
        if name == "fp32":
            # bound by instruction issue: warp instructions per launch (committed ncu
            # capture of the same sources) over the live time, against one warp
            # instruction per scheduler per cycle at the maximum SM clock
            inst = profile_value(SAMPLER_SOURCES, "gumbel_sample_b256_v151936.md",
                                 "inst_executed_per_launch")
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            peak = sms * 4 * 2.07e9
            res[name]["roofline"] = {
                "bound": "alu", "unit": "warp instructions/s", "peak": peak,
                "peak_source": f"{sms} SMs x 4 schedulers x 1 instruction/cycle x 2.07 GHz",
                "achieved": inst / (ms * 1e-3) if inst else None,
                "frac": inst / (ms * 1e-3) / peak if inst else None,
                "inst_per_launch": inst}
        del bufs
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the sampler")
    return res


def measure_staged(dev, steps: int, warmup: int):
    """Block-table update through StagedWriteTensor ("Model Runner V2 设计文档", section 4):
    a [1024, 1000] int32 table on the device; each step appends one block id to 256
    sequences (a decode step of 256 sequences). Timed with CUDA events: the apply kernel
    alone, and the one H2D copy of the packed buffer plus the kernel; on the host clock,
    a whole apply_write (staging + native merge/pack + issue). For comparison, a full H2D
    copy of the table from pinned memory."""
    import numpy as np
    import torch

    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300.staged import StagedWriteTensor, pack

    rng = np.random.default_rng(107400)
    R, C, W = 1024, 1000, 256
    init = np.full((R, C), -1, np.int32)
    t = StagedWriteTensor((R, C), dtype=torch.int32, init=torch.from_numpy(init))
    stream = torch.cuda.current_stream(dev)
    n = steps + warmup
    rows_all = [rng.choice(R, size=W, replace=False).astype(np.int32) for _ in range(n)]
    ids_all = [rng.integers(1 << 20, size=W).astype(np.int32) for _ in range(n)]
    col = np.zeros(R, np.int32)

    def cols_for(rows):
        c = col[rows] % C
        col[rows] += 1
        return c

    # host: a whole apply_write per step, the engine's way (arrays of rows, columns, ids)
    for i in range(warmup):
        t.stage_writes(rows_all[i], cols_for(rows_all[i]), ids_all[i])
        t.apply_write(stream)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(warmup, n):
        t.stage_writes(rows_all[i], cols_for(rows_all[i]), ids_all[i])
        t.apply_write(stream)
    host_ms = (time.perf_counter() - t0) * 1e3 / steps
    torch.cuda.synchronize(dev)
    h2d_bytes = t.last_h2d_bytes

    # device: pre-packed buffers, then (copy + kernel) per step and the kernel alone
    packed = []
    for i in range(n):
        buf, lay = pack(rows_all[i], cols_for(rows_all[i]), np.ones(W, np.int32), ids_all[i], 4)
        h = torch.from_numpy(buf.copy()).pin_memory()
        packed.append((h, torch.empty(h.numel(), dtype=torch.uint8, device=dev), lay))

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            fn(i)
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in ev[warmup:])

    def upload_apply(i):
        h, d, lay = packed[i]
        pk.pa_staged_upload_apply(t.gpu, h, d, lay, dev_err=t.dev_err, stream=stream)

    lib = pk.load_library()

    def kernel(i):
        _, d, lay = packed[i]
        base = d.data_ptr()
        rc = lib.pa_staged_write_apply(
            t.gpu.data_ptr(), R, C, C, 4, base + lay.rows_offset, base + lay.starts_offset,
            base + lay.offsets_offset, base + lay.values_offset, lay.num_writes,
            lay.num_values, t.dev_err.data_ptr(), stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"pa_staged_write_apply returned {rc}")

    upload_ms = timed(upload_apply)
    kernel_ms = timed(kernel)
    host_tab = torch.from_numpy(init).pin_memory()
    full_ms = timed(lambda i: t.gpu.copy_(host_tab, non_blocking=True))
    if int(t.dev_err.item()) != 0:
        raise RuntimeError(f"device error bits {int(t.dev_err.item())} in the staged writes")
    return {"workload": "block_table_1024x1000_int32_256_appends", "writes_per_step": W,
            "kernel_us": kernel_ms * 1e3, "upload_apply_device_us": upload_ms * 1e3,
            "apply_write_host_us": host_ms * 1e3, "h2d_bytes_per_step": h2d_bytes,
            "full_table_copy_us": full_ms * 1e3, "full_table_bytes": R * C * 4,
            "bound": "launch latency (1 KB of values per step)"}


def run_ours(args):
    import numpy as np
    import torch

    import paged_kv_cache_107_gb300 as pk
    from paged_kv_cache_107_gb300 import workloads

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk.load_library()
    case = workloads.workload(args.workload, poison=True, num_blocks=args.pool_blocks)
    tot_ctx, kv_bytes, small_bytes, store_bytes = workload_summary(case)
    B, H, Hk, D = case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim

    k_cache = case.k_cache.to(dev)
    v_cache = case.v_cache.to(dev)
    q = case.q.to(dev)
    k_new = case.k_new.to(dev)
    v_new = case.v_new.to(dev)
    slots = torch.from_numpy(case.slot_mapping).to(dev)
    bt = torch.from_numpy(case.block_tables).to(dev)
    ctx = torch.from_numpy(case.context_lens).to(dev)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pk.DecodeWorkspace(B, H, Hk, D, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        # the production step: store of the new tokens and decode in one launch
        pk.pa_decode_step(out, q, k_new, v_new, k_cache, v_cache, slots, bt, ctx,
                          workspace=ws, dev_err=err, stream=stream)

    def store():
        pk.pa_store_kvcache(k_new, v_new, k_cache, v_cache, slots, dev_err=err, stream=stream)

    def decode():
        pk.pa_decode(out, q, k_cache, v_cache, bt, ctx, workspace=ws, dev_err=err, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
        store()
        decode()
    torch.cuda.synchronize(dev)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during warm-up")

    def timed(fns, per_launch=True):
        """K steps back to back on `stream`. Returns the whole region's ms (max over ranks)
        and, with per_launch, the mean ms of each launch from one event pair per launch
        (those events cost a little time between launches, so the step throughput comes
        from a pass without them)."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
              for _ in range(args.steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for i in range(args.steps):
            if per_launch:
                ev[i][0].record(stream)
            for k, fn in enumerate(fns):
                fn()
                if per_launch:
                    ev[i][k + 1].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        total = max_over_ranks(start.elapsed_time(end), world)
        if not per_launch:
            return total, None
        per = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in ev) for k in range(len(fns))]
        return total, per

    # ---- device-timed region: the fused step (throughput pass, then a pass timing each
    # launch), then the same step as two launches ------------------------------------------
    with ClockSampler(dev) as clocks:
        total_ms, _ = timed([step], per_launch=False)
        _, (step_ms,) = timed([step])
        two_total_ms, (store_ms, decode_ms) = timed([store, decode])
    ms_step = total_ms / args.steps
    two_ms_step = two_total_ms / args.steps
    clk = clocks.summary()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} in the timed region")

    value = world * kv_bytes / (ms_step * 1e-3) / 1e9
    seqs_per_s = world * B / (ms_step * 1e-3)
    hbm_peak, _, peak_src = measured_peaks()
    # fused kernel: K/V of every context position (the newest one read from k_new/v_new),
    # q, o, block tables, context lengths, slots, and the new rows written to the cache
    step_alg_bytes = kv_bytes + small_bytes + case.slot_mapping.nbytes + store_bytes // 2
    achieved = step_alg_bytes / (step_ms * 1e-3) / 1e9
    kname = decode_step_kernel(H, Hk, D)
    traffic = kernel_traffic(decode_step_sources(kname), STEP_PROFILES.get(case.name, ""),
                             case.name, kname)

    # ---- end to end through the public API with host buffers ---------------------------
    # every step uploads its inputs from pinned host memory (one packed copy) and copies its
    # output back; DecodeStepPipeline runs those copies on two copy streams so that they
    # overlap the neighbouring steps' kernels, and issues the steps E2E_GROUP at a time so
    # that the steps of a group chain as dependent launches (2 x E2E_GROUP buffer sets)
    from paged_kv_cache_107_gb300.step_io import DecodeStepPipeline
    pipe = DecodeStepPipeline(B, H, Hk, D, case.block_tables.shape[1], dtype=q.dtype,
                              device=dev, compute_stream=stream, depth=2 * E2E_GROUP,
                              group=E2E_GROUP)
    for k in range(pipe.depth):
        hv = pipe.inputs(k)
        hv["q"].copy_(case.q)
        hv["k_new"].copy_(case.k_new)
        hv["v_new"].copy_(case.v_new)
        hv["slot_mapping"].copy_(torch.from_numpy(case.slot_mapping))
        hv["block_tables"].copy_(torch.from_numpy(case.block_tables))
        hv["context_lens"].copy_(torch.from_numpy(case.context_lens))
    h2d = pipe.h2d_bytes
    d2h = pipe.d2h_bytes

    def run(dv, o):
        pk.pa_decode_step(o, dv["q"], dv["k_new"], dv["v_new"], k_cache, v_cache,
                          dv["slot_mapping"], dv["block_tables"], dv["context_lens"],
                          workspace=ws, dev_err=err, stream=stream)

    n_warm = 2 * E2E_GROUP  # every buffer set used once before the timed region
    for i in range(n_warm):
        pipe.submit(i, run)
    pipe.join()
    torch.cuda.synchronize(dev)
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    pipe.start_after(s2)
    for i in range(args.steps):
        pipe.submit(n_warm + i, run)
    pipe.join(stream)
    e2.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(s2.elapsed_time(e2) / args.steps, world)
    barrier(world)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": case.name, "num_seqs": B, "num_heads": H, "num_kv_heads": Hk,
                   "head_dim": D, "block_size": case.block_size, "num_blocks": case.num_blocks,
                   "total_context_tokens": tot_ctx, "kv_bytes_per_step": kv_bytes,
                   "l2": "inputs larger than L2 (K/V read per step >> 129 MB); no flush",
                   "parallelism": f"replicas x{world}"},
        "seqs_per_s": seqs_per_s,
        "pct_of_nominal_hbm": 100.0 * value / world / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": 100.0 * value / world / hbm_peak,
        "kernels_ms": {"decode_step": step_ms},
        "two_launch_step": {
            "value": world * kv_bytes / (two_ms_step * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": two_ms_step, "kernels_ms": {"store": store_ms, "decode": decode_ms},
            "decode_achieved_gbs": (kv_bytes + small_bytes) / (decode_ms * 1e-3) / 1e9},
        "roofline": {"kernel": kname, "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak,
                     "peak_source": f"{peak_src} HBM copy GB/s",
                     "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                     "alg_bytes_per_launch": step_alg_bytes},
        "e2e": {"value": world * kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "per step: one packed upload from pinned memory and one download, "
                          "on two copy streams overlapping the neighbouring steps; steps "
                          f"issued {E2E_GROUP} at a time behind one event wait"},
        # the library's kernels launched in the device-timed region: the fused step in the
        # throughput pass and in the per-launch pass, store + decode in the two-launch pass
        "gpu_launches": 4 * args.steps,
        "clocks": clk,
    }
    if not args.no_prefill:
        line["long_context"] = measure_long_context(dev, steps=min(args.steps, 20),
                                                    warmup=args.warmup)
        cpu_s = 0.0 if (rank != 0 or args.no_cpu_baseline) else args.cpu_seconds / 2
        line["prefill"] = measure_prefill(dev, steps=min(args.steps, 20), warmup=args.warmup,
                                          cpu_seconds=cpu_s)
        line["staged_write"] = measure_staged(dev, steps=min(args.steps, 50), warmup=args.warmup)
        line["sampler"] = measure_sampler(dev, steps=min(args.steps, 50), warmup=args.warmup)
        line["variants"] = measure_variants(dev, steps=min(args.steps, 30), warmup=args.warmup)
        line["prefix_sharing"] = measure_prefix_sharing(dev, steps=min(args.steps, 30),
                                                        warmup=args.warmup)
    if rank == 0 and not args.no_cpu_baseline:
        stored = oracle_store(case)
        cb = cpu_baseline(case, seconds=args.cpu_seconds, stored=stored)
        # the same oracle on one host thread, on a shorter sample
        c1 = cpu_baseline(case, seconds=max(args.cpu_seconds / 3, 1.0), threads=1,
                          stored=stored)
        line["cpu_baseline"] = {"value": cb["gbs"], "unit": "GB/s", "cores": cb["cores"],
                                "kind": "oracle", "sample": cb["sample"],
                                "seqs_per_s": cb["seqs_per_s"],
                                "single_thread": {"value": c1["gbs"], "unit": "GB/s",
                                                  "cores": c1["cores"], "sample": c1["sample"]}}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, choices=[2, 3])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=1.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the secondary chunked-prefill measurement")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the chunked-prefill step (for profiler captures)")
    ap.add_argument("--variants-only", action="store_true",
                    help="time only the head_dim 64 / fp16 variants")
    ap.add_argument("--variant", default=None,
                    choices=["d64_bf16", "d64_fp16", "d128_fp16", "g4", "g8"],
                    help="with --variants-only: time this variant alone")
    ap.add_argument("--sampler-only", action="store_true",
                    help="time only the Gumbel-max sampler (for profiler captures)")
    ap.add_argument("--staged-only", action="store_true",
                    help="time only the staged block-table writes (for profiler captures)")
    ap.add_argument("--batches-only", action="store_true",
                    help="time only the decode step at batch sizes 1..256")
    ap.add_argument("--long-only", action="store_true",
                    help="time only the long-context decode step (for profiler captures)")
    ap.add_argument("--prefix-only", action="store_true",
                    help="time only the prefix-sharing decode step at block sizes 16 and 256")
    ap.add_argument("--pool-blocks", type=int, default=None,
                    help="override the block pool size (a smaller pool for profiler captures)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.variants_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_variants(dev, args.steps, args.warmup, args.variant,
                                          args.pool_blocks)))
    elif args.sampler_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_sampler(dev, args.steps, args.warmup)))
    elif args.staged_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_staged(dev, args.steps, args.warmup)))
    elif args.batches_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_batch_sizes(dev, args.steps, args.warmup)))
    elif args.long_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_long_context(dev, args.steps, args.warmup, args.pool_blocks)))
    elif args.prefix_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_prefix_sharing(dev, args.steps, args.warmup)))
    elif args.prefill_only:
        import torch
        import paged_kv_cache_107_gb300 as pk
        pk.load_library()
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(measure_prefill(dev, args.steps, args.warmup, args.pool_blocks)))
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
