"""CPU pins of the Gumbel-max sampling oracle ("nano-vllm解读", "Gumbel-Max采样";
"Model Runner V2 设计文档", section 6 "Gumbel 采样内核"): the generator against its
published known-answer vectors, the uniform mapping's closed form, the sampling law
(Gumbel-max theorem: the sample of a row is distributed as softmax(logits / T)) by a
chi-square test, and the greedy, NaN, tie and shift special cases."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def _hex(ws):
    return [int(w, 16) for w in ws]


def test_philox_known_answer_vectors():
    for vec in json.load(open(GOLDEN))["vectors"]:
        got = oracle.philox4x32_10(_hex(vec["counter"]), _hex(vec["key"]))
        assert got.tolist() == _hex(vec["expected"])


def test_element_bits_follow_the_counter_layout():
    """Element i draws word i % 4 of the block at counter (i/4, i/2^34, offset lo, hi)
    under key (seed lo, seed hi); checked at element indexes past 2^34 too."""
    seed, offset = 0x0123456789ABCDEF, 0xFEDCBA9876543210
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in (0, 1, 2, 3, 4, 151935, (1 << 34) + 5):
        g = i >> 2
        words = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, offset & 0xFFFFFFFF, offset >> 32], key)
        assert oracle.philox_bits(seed, offset, i) == int(words[i & 3])


def test_uniform_mapping_closed_form():
    assert oracle.uniform(0) == 2.0 ** -24
    assert oracle.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform(0x1FF) == 2.0 ** -24          # the low 9 bits are dropped
    assert oracle.uniform(0x200) == 3.0 * 2.0 ** -24
    for bits in (0, 1 << 31, 0xDEADBEEF, 0xFFFFFFFF):
        u = oracle.uniform(bits)
        assert 0.0 < u < 1.0 and float(np.float32(u)) == u


def _chi2_pvalue(counts, probs):
    from scipy.stats import chi2
    n = counts.sum()
    exp = probs * n
    stat = float(((counts - exp) ** 2 / exp).sum())
    return float(chi2.sf(stat, len(probs) - 1))


@pytest.mark.parametrize("T", [0.7, 1.0, 2.5])
def test_samples_follow_softmax_over_seeds(T):
    """30000 rows with the same logits and distinct seeds: the frequencies of the samples
    match softmax(logits / T) (chi-square, 5 degrees of freedom)."""
    l = np.array([1.0, 0.5, -0.3, 2.0, 0.0, -1.0], np.float32)
    B = 30000
    logits = np.tile(l, (B, 1))
    idx, _, _ = oracle.gumbel_sample(logits, np.full(B, T, np.float32),
                                     np.arange(B, dtype=np.uint64) * 7919 + 1,
                                     np.full(B, 42, np.uint64))
    counts = np.bincount(idx, minlength=6).astype(np.float64)
    p = np.exp(l.astype(np.float64) / T)
    p /= p.sum()
    assert _chi2_pvalue(counts, p) > 1e-4, (counts / B, p)


def test_samples_follow_softmax_over_offsets():
    """One seed, successive offsets (the per-step counter of a request): same law."""
    l = np.array([0.2, -0.4, 1.1, 0.9], np.float32)
    B = 20000
    idx, _, _ = oracle.gumbel_sample(np.tile(l, (B, 1)), np.ones(B, np.float32),
                                     np.full(B, 1234, np.uint64), np.arange(B, dtype=np.uint64))
    p = np.exp(l.astype(np.float64))
    p /= p.sum()
    assert _chi2_pvalue(np.bincount(idx, minlength=4).astype(np.float64), p) > 1e-4


def test_very_high_temperature_is_uniform():
    l = np.array([3.0, -2.0, 0.5, 1.0, -0.5], np.float32)
    B = 20000
    idx, _, _ = oracle.gumbel_sample(np.tile(l, (B, 1)), np.full(B, 1e6, np.float32),
                                     np.arange(B, dtype=np.uint64), np.zeros(B, np.uint64))
    assert _chi2_pvalue(np.bincount(idx, minlength=5).astype(np.float64),
                        np.full(5, 0.2)) > 1e-4


def test_greedy_is_numpy_argmax_with_lowest_index_on_ties():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((50, 300)).astype(np.float32)
    logits[7, [10, 200]] = 9.0                      # a tie: the lower index wins
    temps = np.where(np.arange(50) % 2 == 0, 0.0, -1.0).astype(np.float32)
    idx, best, _ = oracle.gumbel_sample(logits, temps, np.arange(50, dtype=np.uint64),
                                        np.zeros(50, np.uint64))
    assert np.array_equal(idx, np.argmax(logits, axis=1))
    assert idx[7] == 10 and best[7] == 9.0


def test_nan_never_wins_and_an_empty_row_gives_zero():
    logits = np.zeros((3, 8), np.float32)
    logits[0, 2] = np.nan
    logits[0, 5] = 1.0
    logits[1, :] = np.nan
    logits[2, :] = -np.inf
    idx, _, _ = oracle.gumbel_sample(logits, np.array([0.0, 1.0, 1.0], np.float32),
                                     np.arange(3, dtype=np.uint64), np.zeros(3, np.uint64))
    assert idx.tolist() == [5, 0, 0]


def test_shift_of_all_logits_does_not_change_the_sample():
    """softmax is invariant under adding a constant to every logit of the row."""
    rng = np.random.default_rng(4)
    B, V = 200, 1000
    logits = rng.standard_normal((B, V)).astype(np.float32) * 3
    args = (np.full(B, 0.8, np.float32), np.arange(B, dtype=np.uint64) + 99,
            np.full(B, 5, np.uint64))
    a, best, second = oracle.gumbel_sample(logits, *args)
    b, _, _ = oracle.gumbel_sample(logits + np.float32(4.0), *args)
    clear = (best - second) > 1e-9
    assert np.array_equal(a[clear], b[clear]) and clear.mean() > 0.99


def test_bf16_logits_equal_their_fp32_widening():
    import torch
    rng = np.random.default_rng(5)
    lt = torch.from_numpy(rng.standard_normal((20, 500)).astype(np.float32)).to(torch.bfloat16)
    args = (np.full(20, 1.0, np.float32), np.arange(20, dtype=np.uint64), np.zeros(20, np.uint64))
    a, _, _ = oracle.gumbel_sample(lt, *args)
    b, _, _ = oracle.gumbel_sample(lt.float().numpy(), *args)
    assert np.array_equal(a, b)


def test_scores_of_one_row_agree_with_the_sample():
    rng = np.random.default_rng(6)
    row = rng.standard_normal(4096).astype(np.float32)
    s = oracle.gumbel_scores(row, 0.9, 77, 3)
    idx, best, second = oracle.gumbel_sample(row[None, :], np.array([0.9], np.float32),
                                             np.array([77], np.uint64), np.array([3], np.uint64))
    assert idx[0] == int(np.argmax(s)) and best[0] == s.max()
    assert second[0] == np.sort(s)[-2]
