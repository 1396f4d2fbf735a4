"""The persistent schedule (augtree_config.schedule = AUGTREE_SCHED_PERSISTENT) on the
GPU: the key-side and query-side backward kernels run one block per lane of AssignGrid's
placement, re-initialising their barriers between the units of a lane.  Forward and both backward
forms match the oracle on ragged trees, with few lanes (many units per lane, largest-
first greedy lanes) and with lanes from the exact placement (at most 12 units), and the
fused backward's dK/dV are bit-identical across two runs."""
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import compare, device_inputs, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

TREES = [
    W.Tree([300, 129], [[129, 1, 200], [64, 3]]),
    W.Tree([0, 257], [[70, 1], [1] * 5 + [130]]),
    W.Tree([1000], [[700, 5, 260]]),
]


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("sms", [3, 16, 0])
def test_persistent_schedule_matches_oracle(cuda_device, ti, sms):
    w = W.custom(TREES[ti], hq=8, hkv=2, d=128, dtype="bf16", seed=90 + ti)
    ref = run_oracle(w)
    t = device_inputs(w, cuda_device)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC, num_sms=sms,
                             schedule=at.SCHED_PERSISTENT)
    for fused in (True, False):
        compare(run_cuda(w, t=t, plan=plan, fused=fused), ref, "bf16")


def test_persistent_schedule_exact_lanes_and_determinism(cuda_device):
    # 6 prompt rows' worth of units per queue at most: the placement is AssignGrid's exact one.
    w = W.custom(W.Tree([200], [[90, 40]]), hq=4, hkv=2, d=128, dtype="bf16", seed=7)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC, num_sms=2,
                             schedule=at.SCHED_PERSISTENT)
    cfg = at.make_config(w.hq, w.hkv, w.d, at.BF16, 0.0, 2, at.KERNEL_TC)
    assert len(at.schedule_build(w.tree.offsets(), cfg, at.OP_TREE_BWD)) <= at.LANES_EXACT_UNITS
    t = device_inputs(w, cuda_device)
    a = run_cuda(w, t=t, plan=plan)
    b = run_cuda(w, t=t, plan=plan)
    compare(a, run_oracle(w), "bf16")
    for k in ("dk_p", "dv_p", "dk_r", "dv_r", "dq_p", "dq_r"):
        assert (a[k] == b[k]).all(), k
