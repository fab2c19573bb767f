"""The sampler's noise arithmetic above u = 0.9, checked on the CPU over every uniform the
kernel can draw ("nano-vllm解读", "Gumbel-Max采样": G = -ln(-ln u); the kernel ranks in
log2 units and needs -log2 u with relative accuracy, since G amplifies it near u = 1).

The kernel takes u = (2k + 1) / 2^24 from the top 23 random bits k. For u <= 0.9 it uses
the hardware log2; above, it evaluates log2 u = -w P(w) on the exact w = 1 - u with a
fitted cubic P whose coefficients sit in csrc/sample.cu on the line tagged
`log2-uniform-cubic:`. This test reads that line and evaluates the cubic in binary32 the
way the kernel does (Horner with fused multiply-adds, one rounding each), for all 838,861
uniforms above 0.9, against fp64 logarithms. It also checks the integer threshold that
selects between the two forms."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "paged_kv_cache_107_gb300", "csrc", "sample.cu")


def _cubic():
    text = open(SRC).read()
    m = re.search(r"log2-uniform-cubic:((?:\s+-?[0-9.]+f)+)", text)
    assert m, "coefficient line not found"
    return [np.float32(float(t.rstrip("f"))) for t in m.group(1).split()]


def _fma32(a, b, c):
    # a*b is exact in fp64 for binary32 operands; the sum is rounded to fp64, then to fp32
    # (a double rounding that can differ from one fused rounding by at most one ulp)
    return (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(np.float32)


def _uniforms():
    k = np.arange(2 ** 23, dtype=np.int64)
    return k, (2 * k + 1) / 2.0 ** 24


def test_cubic_relative_error_above_0_9():
    coef = _cubic()
    assert len(coef) == 4
    k, u = _uniforms()
    sel = u > 0.9
    u32 = u[sel].astype(np.float32)
    assert np.array_equal(u32.astype(np.float64), u[sel])  # u is exact in binary32
    w = (np.float32(1) - u32).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), 1.0 - u[sel])  # and so is 1 - u
    p = np.full_like(w, coef[0])
    for c in coef[1:]:
        p = _fma32(p, w, c)
    got = (w.astype(np.float64) * p.astype(np.float64)).astype(np.float32).astype(np.float64)
    exact = np.log2(u[sel])
    rel = np.abs(got - exact) / np.abs(exact)
    assert rel.max() < 4e-7, (rel.max(), u[sel][rel.argmax()])
    assert np.all(got < 0)


def test_threshold_selects_u_at_most_0_9():
    text = open(SRC).read()
    m = re.search(r"bits < (\d+)u \? a : w \* p", text)
    assert m
    thr = int(m.group(1))
    k, u = _uniforms()
    # every 32-bit word with top 23 bits k: the lowest and highest of them
    for low in (0, 511):
        bits = (k << 9) | low
        assert np.array_equal(bits < thr, u <= 0.9)
