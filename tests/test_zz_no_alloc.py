"""The allocation-free prefill backward (augtree_prefill_bwd_static).

Some callers cannot call cudaMalloc while they run - for example code inside a
caching-allocator callback (allocating there would recurse), or a step that must never
meet an out-of-memory error.  For them the library keeps the prefill backward's scratch
in a fixed 64 MiB device array whose address the plan looks up when it is created.

This file checks, through the C ABI, on two calls in a row:
  * the tensor-core family gives results bit-identical to the workspace-taking
    augtree_prefill_bwd (same kernels, same inputs, no atomics anywhere);
  * the SIMT family (fp32) gives bit-identical dK and dV; its dQ is summed with fp32
    atomic adds, whose order varies from run to run, so dQ is held to the fp32 bound
    used throughout (1e-4 relative Frobenius);
  * the calls allocate nothing: the caching allocator's count and the device's free
    memory are unchanged across them;
and that a plan needing more scratch than the array holds is rejected before any work
is queued.  It is named to run last, and passes alone in a fresh process as well as
after the other tests.
"""
import gc

import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import TOL, device_inputs, rel_frob

pytestmark = pytest.mark.gpu


def _prefill_inputs(w, dev, kernel):
    dt = at.BF16 if w.dtype == "bf16" else at.FP32
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=dt, kernel=kernel)
    t = device_inputs(w, dev)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    g = torch.Generator(device="cpu").manual_seed(3)
    dk_acc = torch.randn(t["k_p"].shape, generator=g).to(dev)
    dv_acc = torch.randn(t["v_p"].shape, generator=g).to(dev)
    return plan, t, o_p, lse_p, dk_acc, dv_acc


CASES = [
    # (structure, heads, head_dim, dtype, kernel family)
    (W.Tree([700, 300], [[90, 40], [5]]), 8, 2, 128, "bf16", at.KERNEL_TC),
    (W.Tree([333, 65], [[7], [1, 20]]), 4, 2, 64, "fp32", at.KERNEL_SIMT),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_static_scratch_prefill_backward_matches_workspace_version(cuda_device, ci):
    tree, hq, hkv, d, dtype, kernel = CASES[ci]
    w = W.custom(tree, hq=hq, hkv=hkv, d=d, dtype=dtype, seed=17 + ci)
    plan, t, o_p, lse_p, dk_acc, dv_acc = _prefill_inputs(w, cuda_device, kernel)
    assert plan.workspace_bytes(at.OP_PREFILL_BWD) <= 64 << 20
    e = lambda x: torch.empty_like(x)
    ref = [e(t["q_p"]), e(t["k_p"]), e(t["v_p"])]
    ws = torch.empty(plan.workspace_bytes(at.OP_PREFILL_BWD), dtype=torch.uint8, device=cuda_device)
    at.augtree_prefill_bwd(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p, t["do_p"], dk_acc, dv_acc, *ref, ws)
    outs = [[e(t["q_p"]), e(t["k_p"]), e(t["v_p"])] for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):
        # Tensors of earlier tests held in reference cycles (an exception's traceback,
        # say) are freed whenever Python's cycle collector runs: collect them first and
        # keep the collector off while the call is measured.
        gc.collect()
        gc.disable()
        try:
            alloc0 = torch.cuda.memory_allocated(cuda_device)
            free0 = torch.cuda.mem_get_info(cuda_device)[0]
            at.augtree_prefill_bwd_static(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p, t["do_p"], dk_acc,
                                          dv_acc, *outs[call])
            plan.check()
            alloc1 = torch.cuda.memory_allocated(cuda_device)
            free1 = torch.cuda.mem_get_info(cuda_device)[0]
        finally:
            gc.enable()
        assert alloc1 == alloc0, call
        assert free1 == free0, call
        for name, a, b in zip(("dq_p", "dk_p", "dv_p"), outs[call], ref):
            if kernel == at.KERNEL_SIMT and name == "dq_p":
                err = rel_frob(a.double().cpu().numpy(), b.double().cpu().numpy())
                assert err <= TOL["fp32"][1], (call, name, err)
            else:
                assert torch.equal(a, b), (call, name)


def test_static_scratch_rejects_plans_beyond_its_size(cuda_device):
    # 32,768 prompt rows x 32 query heads need about 73 MB of scratch (per-tile row
    # statistics and extra-MMA rows, plus the dK/dV flush slots), above 64 MiB.
    w = W.custom(W.Tree([32768], [[]]), hq=32, hkv=8, d=128, dtype="bf16", seed=1)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    assert plan.workspace_bytes(at.OP_PREFILL_BWD) > 64 << 20
    z = torch.zeros(1, device=cuda_device)
    with pytest.raises(at.AugtreeError) as ei:
        at.augtree_prefill_bwd_static(plan, z, z, z, z, z, z, None, None, z, z, z)
    assert ei.value.status == at.ERR_WORKSPACE_TOO_SMALL
