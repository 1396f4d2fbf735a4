"""Parity of the tcgen05 path, forward and backward (bf16 in, fp32 accumulate), with
the fp64 oracle: relative Frobenius error of every gradient (dQ, dK, dV of prompt and
responses) <= 2e-2, forward max-abs <= 1e-2.  Covers prompt-KV split-K (few and many
splits), response KV tiles that span several branches, and empty pieces."""
import numpy as np
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import compare, run_cuda, run_oracle, device_inputs

pytestmark = pytest.mark.gpu

TREES = [
    W.Tree([300], [[129, 1, 200]]),
    W.Tree([150, 0, 70], [[1, 65, 130], [20, 0], [3]]),
    W.Tree([0, 129], [[64, 1, 2, 200], []]),
    W.Tree([257], [[1] * 9 + [128, 127, 300]]),
    W.Tree([1000], [[700, 5, 260]]),
]


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4)])
def test_tc_forward_backward_matches_oracle(cuda_device, ti, hq, hkv):
    w = W.custom(TREES[ti], hq=hq, hkv=hkv, d=128, dtype="bf16", seed=500 + ti, scale=1.0)
    got = run_cuda(w, kernel=at.KERNEL_TC)
    compare(got, run_oracle(w), "bf16")


@pytest.mark.parametrize("num_sms", [1, 4, 100000])
def test_tc_split_k_variants(cuda_device, num_sms):
    w = W.custom(W.Tree([400], [[300, 520, 90, 7]]), hq=4, hkv=1, d=128, dtype="bf16", seed=9)
    got = run_cuda(w, kernel=at.KERNEL_TC, num_sms=num_sms)
    compare(got, run_oracle(w), "bf16")


def test_tc_prompt_gradient_is_deterministic(cuda_device):
    w = W.custom(TREES[4], hq=8, hkv=2, d=128, dtype="bf16", seed=31)
    t = device_inputs(w, cuda_device)
    a = run_cuda(w, kernel=at.KERNEL_TC, t=t, num_sms=4)
    b = run_cuda(w, kernel=at.KERNEL_TC, t=t, num_sms=4)
    for k in ("dk_p", "dv_p", "dk_r", "dv_r", "o_p", "o_r", "lse_p", "lse_r"):
        assert np.array_equal(a[k], b[k]), k


def test_tc_long_item_pipelines(cuda_device):
    """Items that walk hundreds of query tiles (no prompt-KV splitting): the producer,
    MMA issuer and compute warps run long pipelines over their buffers, and the prompt
    KV items (5000 response rows x 8 heads: 5000 x 8 / 16 = 2500 accumulation steps of
    16 rows) pass the periodic move of dK/dV from TMEM to the fp32 slots (every 2048)."""
    w = W.custom(W.Tree([256], [[3000, 2000]]), hq=16, hkv=2, d=128, dtype="bf16", seed=41)
    got = run_cuda(w, kernel=at.KERNEL_TC, num_sms=100000)
    compare(got, run_oracle(w), "bf16")
