"""Bounded device-side waits: a wait limit far below how long the kernels' legitimate
waits last (a tile landing from HBM, an MMA group finishing, a softmax handing P over)
makes the tensor-core kernels give up.  The call must then report
AUGTREE_ERR_TIMEOUT through augtree_plan_check - not fault, trap or hang - and leave
the device and the plan usable: with the default limit restored, the same plan's next
forward and backward match the oracle.

Every give-up path drains the block's own bulk copies and MMAs (fixed-limit waits,
since those always complete) before it frees tensor memory and exits, so giving up
leaves nothing in flight."""
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import compare, device_inputs, run_cuda, run_oracle

pytestmark = pytest.mark.gpu


def test_wait_limit_is_validated(cuda_device):
    w = W.custom(W.Tree([10], [[5]]), hq=2, hkv=1, d=128, dtype="bf16", seed=1)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    for bad in (0, 60_000_000_001):
        with pytest.raises(at.AugtreeError) as ei:
            plan.set_wait_limit(bad)
        assert ei.value.status == at.ERR_INVALID_ARG
    plan.set_wait_limit(60_000_000_000)
    plan.set_wait_limit(2_000_000_000)


def test_short_wait_limit_times_out_cleanly(cuda_device):
    w = W.custom(W.Tree([3000, 700], [[1500, 700, 1], [900]]), hq=8, hkv=2, d=128, dtype="bf16", seed=31)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, cuda_device)
    plan.set_wait_limit(1)  # 1 ns: any wait not met within a few polls gives up
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                t["do_p"], t["do_r"])
    with pytest.raises(at.AugtreeError) as ei:
        plan.check()
    assert ei.value.status == at.ERR_TIMEOUT
    plan.check()  # the error word was read and cleared
    # The device and the plan stay usable.
    plan.set_wait_limit(2_000_000_000)
    compare(run_cuda(w, plan=plan, t=t), run_oracle(w), "bf16")
