"""Per-kernel timing of a plan's calls (augtree_plan_set_timing / augtree_plan_kernel_times):
each call reports its kernels in launch order, and their durations add up to the call's
own duration measured around it with CUDA events on the same stream."""
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import device_inputs

pytestmark = pytest.mark.gpu


def test_kernel_times_cover_each_call(cuda_device):
    w = W.custom(W.Tree([700, 300], [[200, 90, 40], [513]]), hq=8, hkv=2, d=128, dtype="bf16", seed=23)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, cuda_device)
    with pytest.raises(at.AugtreeError):
        plan.kernel_times(at.OP_REPLAY_BWD)  # timing is off by default
    plan.set_timing(True)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    ev[0].record(stream)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    ev[1].record(stream)
    at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                t["do_p"], t["do_r"], fused=False)
    ev[2].record(stream)
    torch.cuda.synchronize()
    plan.check()
    # This queue is short for the GPU: the replay forward splits its KV walks, and its
    # partial states and dQ partials are merged and summed by two more kernels.
    fsplit = bool((plan.schedule(at.OP_REPLAY_FWD)[:, 4] > 0).any())
    assert fsplit
    assert [k for k, _ in plan.kernel_times(at.OP_PREFILL_FWD)] == ["fwd_tc"]
    assert [k for k, _ in plan.kernel_times(at.OP_REPLAY_FWD)] == ["fwd_tc", "fwd_split_merge"]
    rb = plan.kernel_times(at.OP_REPLAY_BWD)
    pb = plan.kernel_times(at.OP_PREFILL_BWD)
    assert [k for k, _ in rb] == ["preprocess", "bwd_key_side", "split_reduce", "bwd_query_side", "dq_split_reduce"]
    assert [k for k, _ in pb] == ["preprocess", "bwd_key_side", "bwd_query_side"]
    fwd_ms = sum(m for op in (at.OP_PREFILL_FWD, at.OP_REPLAY_FWD) for _, m in plan.kernel_times(op))
    bwd_ms = sum(m for _, m in rb + pb)
    for part, whole in ((fwd_ms, ev[0].elapsed_time(ev[1])), (bwd_ms, ev[1].elapsed_time(ev[2]))):
        assert 0.0 < part <= whole * 1.02 + 0.02, (part, whole)
    with pytest.raises(at.AugtreeError):
        plan.kernel_times(at.OP_REPLAY_BWD, back=1)  # only one timed call so far
    plan.set_timing(False)


def test_kernel_times_of_the_fused_backward(cuda_device):
    w = W.custom(W.Tree([700, 300], [[200, 90, 40], [513]]), hq=8, hkv=2, d=128, dtype="bf16", seed=29)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, cuda_device)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    plan.set_timing(True)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                t["do_p"], t["do_r"], fused=True)
    e1.record(stream)
    torch.cuda.synchronize()
    plan.check()
    tb = plan.kernel_times(at.OP_TREE_BWD)
    split = bool((plan.schedule(at.OP_TREE_BWD)[:, 4] > 0).any())
    fsplit = bool((plan.schedule(at.OP_REPLAY_FWD)[:, 4] > 0).any())
    want = ["preprocess", "preprocess", "bwd_key_side"] + (["split_reduce"] if split else []) + \
        ["bwd_query_side", "bwd_query_side"] + (["dq_split_reduce"] if fsplit else [])
    assert [k for k, _ in tb] == want
    part = sum(m for _, m in tb)
    assert 0.0 < part <= e0.elapsed_time(e1) * 1.02 + 0.02
    with pytest.raises(at.AugtreeError):
        plan.kernel_times(at.OP_REPLAY_BWD)  # the fused call makes no replay_bwd call
    plan.set_timing(False)
