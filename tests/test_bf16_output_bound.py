"""Where the bf16 forward tolerance comes from, pinned on the CPU.

The stated forward bound (max-abs 1e-2 with bf16 inputs and fp32 accumulation) bounds
the error of the arithmetic.  The output O is stored in the input dtype, bf16, whose
round-to-nearest-even keeps 8 significant bits: storing a value x moves it by at most
2^-8 |x|.  For the N(0,1) configurations |O| stays far below 1 and that rounding is
small; in the large-score stress test of the tensor-core forward (Q and K scaled by 4),
single keys dominate their rows, |O| reaches about 4.3, and the storage rounding alone
reaches 2^-6.

This file models an ideal bf16 tensor-core forward on that exact input - exact scores
and row maxima, the softmax weights P rounded to bf16 (as the PV product consumes
them), exact sums, O rounded to bf16 on output - and checks, against the fp64 oracle:
  1. before output rounding the model stays within 1e-2 (the arithmetic bound holds);
  2. after output rounding it exceeds 1e-2 (so no bf16-output implementation can meet
     the plain bound on this input);
  3. after output rounding it stays within 1e-2 + 2^-8 |O_ref|, the bound the GPU test
     applies to this input;
and pins the rounding fact itself: |bf16(x) - x| <= 2^-8 |x|.
"""
import numpy as np

import workloads as W
from oracle import attention as A

ROUND = 2.0 ** -8


def _bf16(x):
    return W.round_to_bf16(np.asarray(x, dtype=np.float32)).astype(np.float64)


def large_score_inputs():
    """The input of the GPU large-score forward test: Q and K of the prompt and the
    responses scaled by 4 (exact in bf16)."""
    w = W.custom(W.Tree([1000], [[700, 5, 260]]), hq=4, hkv=2, d=128, dtype="bf16", seed=77)
    h = {n: W.tensor_rows_np(w, n) for n in W.TENSORS}
    for n in ("q_p", "k_p", "q_r", "k_r"):
        h[n] = h[n] * 4
    return w, h


def bf16_p_model(w, h, kind):
    """O of every row of side `kind` with P rounded to bf16 and everything else exact."""
    offs = w.tree.offsets()
    scale = A.default_scale(w.d)
    r = w.hq // w.hkv
    q = h["q_" + kind]
    out = np.zeros_like(q)
    for row in range(q.shape[0]):
        (pa, pb), (ra, rb) = A.row_key_set(kind, row, offs)
        for hh in range(w.hq):
            kv = hh // r
            k = np.concatenate([h["k_p"][pa:pb, kv], h["k_r"][ra:rb, kv]])
            v = np.concatenate([h["v_p"][pa:pb, kv], h["v_r"][ra:rb, kv]])
            s = scale * (k @ q[row, hh])
            p = _bf16(np.exp(s - s.max()))
            out[row, hh] = (p @ v) / p.sum()
    return out


def test_bf16_rounding_is_relative_two_to_minus_eight():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.uniform(-3, 3, 200000), [4.3, -4.3, 1.0]])
    err = np.abs(_bf16(x) - x)
    assert np.all(err <= ROUND * np.abs(x))
    # and the bound is attained up to a factor close to 1 (8 significant bits, not 9)
    assert np.max(err / np.abs(x)) > 0.9 * ROUND


def test_large_score_forward_bound_derivation():
    w, h = large_score_inputs()
    ref = A.tree_attention_direct(h, w.tree.offsets(), A.default_scale(w.d), grad=False)
    for kind in ("p", "r"):
        model = bf16_p_model(w, h, kind)
        o_ref = ref["o_" + kind]
        pre = np.abs(model - o_ref)
        post = np.abs(_bf16(model) - o_ref)
        assert pre.max() <= 1e-2, (kind, pre.max())
        assert post.max() > 1e-2, (kind, post.max())
        assert np.all(post <= 1e-2 + ROUND * np.abs(o_ref)), kind
