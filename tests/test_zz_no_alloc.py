"""The allocation-free prefill backward (augtree_prefill_bwd_static).

Some callers cannot call cudaMalloc while they run - for example code inside a
caching-allocator callback, or a step that must never meet an out-of-memory error.
For them the library keeps the prefill backward's scratch in a fixed 64 MiB device
array.  This file checks, through the C ABI, that two calls in a row give the same
results as the workspace-taking augtree_prefill_bwd (within the bf16 gradient
tolerance used throughout: relative Frobenius error <= 2e-2), and that a plan needing
more scratch than the array holds is rejected before any work is queued.  It is named
to run last, and passes alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import TOL, device_inputs, rel_frob

pytestmark = pytest.mark.gpu


def _prefill_inputs(w, dev):
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, dev)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    g = torch.Generator(device="cpu").manual_seed(3)
    dk_acc = torch.randn(t["k_p"].shape, generator=g).to(dev)
    dv_acc = torch.randn(t["v_p"].shape, generator=g).to(dev)
    return plan, t, o_p, lse_p, dk_acc, dv_acc


def test_static_scratch_prefill_backward_matches_workspace_version(cuda_device):
    w = W.custom(W.Tree([700, 300], [[90, 40], [5]]), hq=8, hkv=2, d=128, dtype="bf16", seed=17)
    plan, t, o_p, lse_p, dk_acc, dv_acc = _prefill_inputs(w, cuda_device)
    assert plan.workspace_bytes(at.OP_PREFILL_BWD) <= 64 << 20
    e = lambda x: torch.empty_like(x)
    ref = [e(t["q_p"]), e(t["k_p"]), e(t["v_p"])]
    ws = torch.empty(plan.workspace_bytes(at.OP_PREFILL_BWD), dtype=torch.uint8, device=cuda_device)
    at.augtree_prefill_bwd(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p, t["do_p"], dk_acc, dv_acc, *ref, ws)
    torch.cuda.synchronize()
    tol = TOL["bf16"][1]
    for call in range(2):
        out = [e(t["q_p"]), e(t["k_p"]), e(t["v_p"])]
        at.augtree_prefill_bwd_static(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p, t["do_p"], dk_acc, dv_acc,
                                      *out)
        plan.check()
        for name, a, b in zip(("dq_p", "dk_p", "dv_p"), out, ref):
            err = rel_frob(a.double().cpu().numpy(), b.double().cpu().numpy())
            assert err <= tol, (call, name, err)


def test_static_scratch_rejects_plans_beyond_its_size(cuda_device):
    # 32,768 prompt rows x 32 query heads need about 73 MB of scratch (per-tile row
    # statistics and extra-step rows, plus the dK/dV flush slots), above 64 MiB.
    w = W.custom(W.Tree([32768], [[]]), hq=32, hkv=8, d=128, dtype="bf16", seed=1)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    assert plan.workspace_bytes(at.OP_PREFILL_BWD) > 64 << 20
    z = torch.zeros(1, device=cuda_device)
    with pytest.raises(at.AugtreeError) as ei:
        at.augtree_prefill_bwd_static(plan, z, z, z, z, z, z, None, None, z, z, z)
    assert ei.value.status == at.ERR_WORKSPACE_TOO_SMALL
