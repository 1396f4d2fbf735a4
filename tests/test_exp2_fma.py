"""The FMA-pipe exponential of the tensor-core backward (exp2_fma in
shared_prompt_tree_gb300/csrc/tc_common.cuh), re-evaluated here step by step in fp32
numpy from the constants in that source: range reduction x = n + f with n = rint(x)
by the 1.5 * 2^23 trick, a degree-3 polynomial for 2^f on [-1/2, 1/2], 2^n added into
the exponent bits.  Its relative error must stay far below the 2^-9 rounding of the
bf16 values it feeds (bound checked: 2e-4)."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "shared_prompt_tree_gb300", "csrc", "tc_common.cuh")


def _coefficients():
    body = open(SRC).read()
    body = body[body.index("float exp2_fma("):]
    body = body[:body.index("}")]
    c = [np.float32(x) for x in re.findall(r"([0-9]+\.[0-9]+)f", body) if x not in ("126.", "12582912.")]
    c = [x for x in c if x < 2.0]
    assert len(c) == 4, c
    c3, c2, c1, c0 = c   # written in Horner order: ((c3 f + c2) f + c1) f + c0
    return c0, c1, c2, c3


def exp2_fma_np(x):
    c0, c1, c2, c3 = _coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = t.view(np.int32) - np.int32(0x4B400000)
    f = (x - (t - magic)).astype(np.float32)
    p = np.float32(c3) * f + np.float32(c2)
    p = (p * f + np.float32(c1)).astype(np.float32)
    p = (p * f + np.float32(c0)).astype(np.float32)
    return (p.view(np.int32) + (n << 23)).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-125.0, 8.0, 3_000_001).astype(np.float32)
    got = exp2_fma_np(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 2e-4


def test_integers_and_clamp():
    x = np.arange(-120, 9, dtype=np.float32)
    got = exp2_fma_np(x).astype(np.float64)
    assert np.all(np.abs(got / np.exp2(x.astype(np.float64)) - 1) < 1e-4)
    # -inf and very negative inputs clamp to about 2^-126: positive, tiny, finite
    low = exp2_fma_np(np.array([-np.inf, -1000.0], dtype=np.float32))
    assert np.all(np.isfinite(low)) and np.all(low > 0) and np.all(low < 2.0 ** -125)
