"""The prefill kernel's software exp2 (common.cuh: exp2_poly2), re-evaluated step by step in
float32 with NumPy from the constants in the source, against the exact 2^x."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "paged_kv_cache_161_gb300", "csrc", "common.cuh")


def _consts():
    txt = open(SRC).read()
    c = {k: np.float32(float(v)) for k, v in re.findall(r"(kExp2C[123]) = ([0-9.e+-]+)f", txt)}
    magic = np.float32(float(re.search(r"kRoundMagic = ([0-9.]+)f", txt).group(1)))
    return c["kExp2C1"], c["kExp2C2"], c["kExp2C3"], magic


def _exp2_poly(x):
    c1, c2, c3, magic = _consts()
    x = np.maximum(x.astype(np.float32), np.float32(-127.0))
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = ((c3 * f + c2) * f + c1).astype(np.float32)
    p = (p * f + np.float32(1.0)).astype(np.float32)
    bits = p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.int32).view(np.float32)


def test_relative_error_over_the_softmax_range():
    x = np.linspace(-126.0, 8.5, 2_000_001).astype(np.float32)
    got = _exp2_poly(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 2e-4  # far below the 2^-9 relative step of the bf16 P it feeds


def test_masked_scores_give_exact_zero():
    x = np.array([-np.inf, -1e30, -127.0, -200.0], np.float32)
    assert (_exp2_poly(x) == 0).all()


def test_integers_are_exact_powers_of_two():
    x = np.arange(-20, 9, dtype=np.float32)
    assert np.array_equal(_exp2_poly(x), np.exp2(x))
