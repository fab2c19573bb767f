"""GPU parity of pa_gumbel_sample against the fp64 oracle ("nano-vllm解读", "Gumbel-Max采样";
"Model Runner V2 设计文档", section 6 "Gumbel 采样内核").

The kernel decides in fp32 (logit * log2(e)/T + noise, the noise from the hardware log2
and, for u > 0.9, a fitted cubic in the exact 1 - u), the oracle in fp64 from the same
32-bit random words. So a row must give
exactly the oracle's index whenever the oracle's best score leads the runner-up by more
than the fp32 error bound TOL; inside that bound (a near-tie, where both indices are
correct samples) the kernel's choice must be one of the near-best scores."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_107_gb300 as pk

pytestmark = pytest.mark.gpu


def tol(best):
    # |logit/T| <= ~50 here: product rounding + noise error + sum rounding, with margin
    return 2e-5 * (1.0 + np.abs(best))


def inputs(B, V, seed, dtype=torch.float32, scale=3.0, greedy_every=0, stride_pad=0):
    rng = np.random.default_rng(seed)
    base = rng.standard_normal((B, V + stride_pad), dtype=np.float32) * scale
    logits = torch.from_numpy(base).to(dtype)
    temps = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    if greedy_every:
        temps[::greedy_every] = 0.0
    seeds = rng.integers(0, 2**63, size=B, dtype=np.int64)
    offs = rng.integers(0, 2**40, size=B, dtype=np.int64)
    return logits, temps, seeds, offs


def run(logits, temps, seeds, offs, V=None):
    dev = torch.device("cuda")
    lg = logits.to(dev)
    if V is not None and V != lg.shape[1]:
        lg = lg[:, :V]
    out = torch.full((lg.shape[0],), -7, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pk.pa_gumbel_sample(out, lg, torch.from_numpy(temps).to(dev), torch.from_numpy(seeds).to(dev),
                        torch.from_numpy(offs).to(dev), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.cpu().numpy()


def check(got, logits, temps, seeds, offs, V=None):
    """Greedy rows (exact scores on both sides) must equal the oracle, ties included;
    sampled rows must equal it where the lead is beyond TOL, else pick a near-best score.
    Returns the fraction of sampled rows decided beyond TOL."""
    lg = logits if V is None else logits[:, :V]
    if lg.dtype == torch.bfloat16:
        lg = lg.contiguous()
    else:
        lg = lg.contiguous().numpy()
    idx, best, second = oracle.gumbel_sample(lg, temps, seeds.view(np.uint64), offs.view(np.uint64))
    greedy = ~(temps > 0)
    assert np.array_equal(got[greedy], idx[greedy])
    clear = ~greedy & ((best - second) > tol(best))
    assert np.array_equal(got[clear], idx[clear]), np.flatnonzero(got[clear] != idx[clear])[:5]
    for b in np.flatnonzero(~greedy & ~clear):  # near-ties: any near-best index is correct
        s = oracle.gumbel_scores(lg[b], float(temps[b]), int(seeds.view(np.uint64)[b]),
                                 int(offs.view(np.uint64)[b]))
        assert s[got[b]] >= best[b] - tol(best[b]), (b, got[b], idx[b])
    n = int((~greedy).sum())
    return clear.sum() / n if n else 1.0


def test_qwen3_vocab_fp32_batch256():
    """B=256 rows of V=151936 fp32 logits (N(0,9)), T ~ U[0.3, 1.5], every 8th row greedy,
    random 64-bit seeds and offsets."""
    logits, temps, seeds, offs = inputs(256, 151936, 107300, greedy_every=8)
    got = run(logits, temps, seeds, offs)
    assert check(got, logits, temps, seeds, offs) > 0.99


def test_qwen3_vocab_bf16():
    logits, temps, seeds, offs = inputs(64, 151936, 107301, dtype=torch.bfloat16, greedy_every=5)
    got = run(logits, temps, seeds, offs)
    assert check(got, logits, temps, seeds, offs) > 0.99


@pytest.mark.parametrize("V", [1, 3, 4, 5, 7, 8, 9, 4095, 8191, 8192, 8193, 10239, 10240,
                               10241, 12287, 12288, 12289, 16384, 20001, 20480, 24577])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_vocab_edges(V, dtype):
    """Single element, ragged 16-byte groups, the ring's tile boundaries (10240 fp32 or
    12288 bf16 elements) and the plain-load kernel's chunk boundaries (8192 elements)."""
    logits, temps, seeds, offs = inputs(12, V, 107310 + V, dtype=dtype, greedy_every=4)
    got = run(logits, temps, seeds, offs)
    assert (got >= 0).all() and (got < V).all()
    check(got, logits, temps, seeds, offs)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_unaligned_row_stride(dtype):
    """Rows that do not start on 16 bytes (row stride V + 1): the plain-load path."""
    V = 10001
    logits, temps, seeds, offs = inputs(9, V, 107320, dtype=dtype, stride_pad=1)
    got = run(logits, temps, seeds, offs, V=V)
    check(got, logits, temps, seeds, offs, V=V)


def test_special_values():
    """NaN never wins; a row of -inf (or NaN) gives 0; +inf wins at its lowest index;
    greedy ties go to the lowest index."""
    V = 9000
    logits = torch.zeros((5, V), dtype=torch.float32)
    logits[0, 100] = float("nan")
    logits[0, 8500] = 5.0
    logits[1, :] = float("-inf")
    logits[2, :] = float("nan")
    logits[3, [300, 8200]] = float("inf")
    logits[4, [17, 8999]] = 2.0
    temps = np.array([0.0, 1.0, 1.0, 0.7, 0.0], np.float32)
    seeds = np.arange(5, dtype=np.int64)
    offs = np.zeros(5, np.int64)
    got = run(logits, temps, seeds, offs)
    assert got.tolist() == [8500, 0, 0, 300, 17]


def test_law_on_the_gpu():
    """20000 rows of the same six logits, distinct seeds: the GPU's samples equal the
    oracle's row by row, and their frequencies match softmax(logits / T)."""
    from scipy.stats import chi2
    l = np.array([1.0, 0.5, -0.3, 2.0, 0.0, -1.0], np.float32)
    B, T = 20000, 0.8
    logits = torch.from_numpy(np.tile(l, (B, 1)))
    temps = np.full(B, T, np.float32)
    seeds = np.arange(B, dtype=np.int64) * 104729 + 3
    offs = np.full(B, 9, np.int64)
    got = run(logits, temps, seeds, offs)
    check(got, logits, temps, seeds, offs)
    counts = np.bincount(got, minlength=6).astype(np.float64)
    p = np.exp(l.astype(np.float64) / T)
    p /= p.sum()
    stat = float(((counts - B * p) ** 2 / (B * p)).sum())
    assert chi2.sf(stat, 5) > 1e-4


def test_deterministic_and_offset_dependent():
    logits, temps, seeds, offs = inputs(128, 50000, 107330)
    a = run(logits, temps, seeds, offs)
    b = run(logits, temps, seeds, offs)
    assert np.array_equal(a, b)
    c = run(logits, temps, seeds, offs + 1)
    assert (a != c).mean() > 0.5  # a new step draws new noise
