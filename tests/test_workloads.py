"""The seeded input generators (CPU only): the configurations have the stated shapes,
and the numpy (host) and torch generators give bit-identical values."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def test_config_shapes():
    t = W.workload("tiny")
    assert (t.tree.prompt_lens, t.tree.branch_lens, t.hq, t.hkv, t.d, t.dtype) == ([128], [[64] * 4], 2, 2, 64, "fp32")
    p = W.workload("prompt_heavy")
    assert p.tree.prompt_lens == [32768, 32768] and (p.hq, p.hkv, p.d, p.dtype) == (32, 8, 128, "bf16")
    assert all(len(b) == 8 and all(512 <= x <= 2048 for x in b) for b in p.tree.branch_lens)
    r = W.workload("response_heavy")
    assert r.tree.prompt_lens == [1024] and len(r.tree.branch_lens[0]) == 64
    assert all(1024 <= x <= 16384 for x in r.tree.branch_lens[0])
    m = W.workload("mixed")
    assert m.tree.n_groups == 16
    for lp, bl in zip(m.tree.prompt_lens, m.tree.branch_lens):
        assert len(bl) in (8, 16, 32)
        assert all(lp + x == 65536 // len(bl) for x in bl)
    lg = W.workload("long")
    assert lg.tree.prompt_lens == [262144] and lg.tree.branch_lens == [[8192] * 16]
    assert (lg.hq, lg.hkv) == (64, 8)


def test_pair_count_closed_form():
    tree = W.Tree([3, 0], [[2, 1], [4]])
    # group 0: 3*4/2 + (2*3 + 3) + (1*3 + 1) = 6 + 9 + 4; group 1: 4*5/2 = 10
    assert tree.pair_count() == 6 + 9 + 4 + 10
    assert tree.flattened_tokens() == (3 + 2) + (3 + 1) + 4


def test_bf16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.5 - 2 ** -9, 3.0e38], dtype=np.float32)
    got = W.round_to_bf16(x)
    want = torch.tensor(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("name", ["tiny", "prompt_heavy"])
def test_host_and_torch_generators_agree(name):
    w = W.workload(name)
    if name != "tiny":  # a small slice is enough for the large config
        w = W.custom(W.Tree([40], [[7, 9]]), w.hq, w.hkv, w.d, w.dtype, w.seed, w.scale)
    for tname in W.TENSORS:
        dev = W.tensor_torch(w, tname, "cpu").to(torch.float64).numpy()
        host = W.tensor_rows_np(w, tname)
        np.testing.assert_array_equal(dev, host)
    # Row subsets come out identical to the corresponding slice.
    rows = np.array([0, 5, 13])
    np.testing.assert_array_equal(W.tensor_rows_np(w, "q_r", rows=rows), W.tensor_rows_np(w, "q_r")[rows])


def test_values_are_standard_normal_like():
    w = W.workload("tiny")
    x = W.tensor_rows_np(w, "do_p").ravel()
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    q = W.tensor_rows_np(w, "q_p").ravel()
    assert abs(q.std() - 0.125) < 0.005   # N(0,1)/sqrt(64)
