"""Host arithmetic behind the numbers bench.py reports, checked without a GPU: the
prefill FLOP count against a pair-by-pair count, the K/V bytes of a decode step against
a per-token sum, the sha-gated lookup of ncu figures in profiles/, and the line that
separates streaming rate from fixed cost."""
import os

import pytest

import bench
from paged_kv_cache_107_gb300 import workloads


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_flops_counts_every_unmasked_pair(causal):
    case = workloads.prefill_case([0, 17, 300, 5], [1, 40, 129, 256], 16, 8, 128, 16,
                                  seed=5100, causal=causal, poison=False)
    pairs = 0
    for s in range(len(case.cu_seqlens_q) - 1):
        n = int(case.cu_seqlens_q[s + 1] - case.cu_seqlens_q[s])
        k = int(case.cu_seqlens_k[s + 1] - case.cu_seqlens_k[s])
        c = k - n
        for i in range(n):          # query at absolute position c + i
            for t in range(k):
                if not causal or t <= c + i:
                    pairs += 1
    assert bench.prefill_flops(case) == 4.0 * 16 * 128 * pairs


def test_decode_step_bytes_are_per_token_rows():
    case = workloads.decode_case([1, 0, 300, 4097], 32, 8, 64, 16, seed=5200, poison=False)
    tot_ctx, kv, small, store = bench.workload_summary(case)
    assert tot_ctx == 1 + 300 + 4097
    assert kv == sum(int(n) * 8 * 64 * 2 * 2 for n in case.context_lens)
    assert small == (4 * 32 * 64 * 2 * 2 + case.block_tables.nbytes + case.context_lens.nbytes)
    valid = int((case.slot_mapping >= 0).sum())
    assert valid == 3 and store == valid * 8 * 64 * 2 * 2 * 2


def test_fit_recovers_rate_and_fixed_cost():
    rate_gbs, fixed_us = 7400.0, 15.0
    pts = [(b, b / (rate_gbs * 1e3) + fixed_us) for b in (6.6e7, 2.9e8, 5.4e8, 1.16e9)]
    fit = bench.fit_stream_and_fixed(pts)
    assert fit["stream_gbs"] == pytest.approx(rate_gbs, rel=1e-9)
    assert fit["fixed_us"] == pytest.approx(fixed_us, rel=1e-9)


def test_profile_figures_only_while_sources_match(tmp_path, monkeypatch):
    """A committed ncu figure is reported only while the kernel sources it names hash to
    the sha256 recorded beside it, and a traffic figure only for the workload and kernel
    the summary names; any edit of those sources turns it into None."""
    root = tmp_path / "repo"
    csrc = root / "paged_kv_cache_107_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (root / "profiles").mkdir()
    (csrc / "k.cuh").write_text("kernel v1\n")
    (csrc / "h.cuh").write_text("header\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.source_sha256("k.cuh", "h.cuh")
    (root / "profiles" / "p.md").write_text(
        f"source_sha256: {sha}\nworkload: w_a\nkernel: kern/fused\n"
        f"| traffic_bytes_per_launch: 123456 | read + write |\n"
        f"| inst_executed_per_launch: 789 | x |\n")
    src = ("k.cuh", "h.cuh")
    assert bench.kernel_traffic(src, "p.md", "w_a", "kern/fused") == 123456.0
    assert bench.kernel_traffic(src, "p.md", "w_b", "kern/fused") is None  # another workload
    assert bench.kernel_traffic(src, "p.md", "w_a", "kern") is None        # another kernel
    assert bench.profile_value(src, "p.md", "inst_executed_per_launch") == 789.0
    assert bench.kernel_traffic(("h.cuh", "k.cuh"), "p.md", "w_a", "kern/fused") is None
    (csrc / "k.cuh").write_text("kernel v2\n")
    assert bench.kernel_traffic(src, "p.md", "w_a", "kern/fused") is None
    assert bench.kernel_traffic(src, "missing.md", "w_a", "kern/fused") is None
    assert bench.kernel_traffic(src, "", "w_a", "kern/fused") is None


def test_decode_step_kernel_routing():
    """The kernel the roofline names is the one the launcher picks for the shape."""
    assert bench.decode_step_kernel(16, 8, 128) == "paged_decode_kernel/fused"
    assert bench.decode_step_kernel(32, 8, 128) == "paged_decode_tc_kernel/fused"  # long ctx
    assert bench.decode_step_kernel(64, 8, 128) == "paged_decode_tc_kernel/fused"
    assert bench.decode_step_kernel(16, 8, 64) == "paged_decode_tc_kernel/fused"
    assert bench.decode_step_kernel(32, 16, 128) == "paged_decode_tc_kernel/fused"
    assert bench.decode_step_sources("paged_decode_tc_kernel/fused") == bench.DECODE_TC_SOURCES
    assert bench.decode_step_sources("paged_decode_kernel/fused") == bench.DECODE_SOURCES


def test_prefill_cpu_baseline_counts_pairs_of_its_sample():
    """The CPU baseline's FLOPs are 4*D per unmasked pair of the rows it ran: with the
    whole (tiny) chunk sampled they equal the chunk's FLOP count."""
    case = workloads.prefill_case([0, 17, 30], [5, 9, 3], 4, 2, 64, 16, seed=5300,
                                  poison=False)
    r = bench.prefill_cpu_baseline(case, seconds=60.0, threads=1)
    rows = int(case.cu_seqlens_q[-1]) * case.num_heads
    assert r["sample"].startswith(f"{rows} ")
    t = rows / case.num_heads / r["tokens_per_s"]
    assert r["gflops"] * t * 1e9 == pytest.approx(bench.prefill_flops(case), rel=1e-9)


def test_committed_profiles_name_existing_sources():
    """Every sha-gated summary in profiles/ belongs to a source set that exists."""
    for sources in (bench.DECODE_SOURCES, bench.DECODE_TC_SOURCES, bench.PREFILL_SOURCES,
                    bench.STORE_SOURCES, bench.SAMPLER_SOURCES):
        for name in sources:
            assert os.path.exists(os.path.join(bench.ROOT, "paged_kv_cache_107_gb300", "csrc",
                                               name)), name
