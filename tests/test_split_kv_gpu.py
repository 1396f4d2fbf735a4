"""Split-KV replay forward (AugTree paper, Sec. 3.3: the attention of a query over
disjoint key ranges gives partial online-softmax states that merge associatively into
the exact result; MoveQ's global reduction of partial states).  When the replay queue
has too few blocks for the GPU (short responses under long prompts), each query tile's
KV walk is cut into chunks: the forward writes per-chunk states (O / l, lse) and merges
them in split order, and the query-side backward writes per-chunk fp32 dQ and sums them
in split order.  Parity with the fp64 oracle, the split actually taken, determinism,
agreement with the unsplit queue, the persistent schedule, the two-call backward, and
the workspace check."""
import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import compare, device_inputs, rel_frob, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

# (tree, hq, hkv): 1-3-token branches under 4k-8k prompts; a single response row; chunk
# boundaries inside the own-branch tiles; an empty prompt; a 16k prompt whose one query
# tile splits 33 ways (the merge's second group of 32 splits).
CASES = [
    (W.Tree([8192], [[3] * 32]), 32, 8),
    (W.Tree([4000, 8000], [[1, 2, 3, 1], [3, 3, 2]]), 4, 2),
    (W.Tree([8192], [[1]]), 4, 1),
    (W.Tree([300], [[600]]), 2, 2),
    (W.Tree([0], [[1000]]), 2, 1),
    (W.Tree([16384], [[1]]), 2, 1),
]


def _split_items(plan):
    q = plan.schedule(at.OP_REPLAY_FWD)
    return int((q[:, 4] > 0).sum())


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_split_kv_matches_oracle(cuda_device, ci):
    tree, hq, hkv = CASES[ci]
    w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=900 + ci)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    assert _split_items(plan) > 0 and plan.workspace_bytes(at.OP_REPLAY_FWD) > 0
    if ci == len(CASES) - 1:
        assert int(plan.schedule(at.OP_REPLAY_FWD)[:, 4].max()) + 1 == 33
    compare(run_cuda(w, plan=plan), run_oracle(w), "bf16")


def test_split_kv_is_deterministic(cuda_device):
    tree, hq, hkv = CASES[1]
    w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=31)
    t = device_inputs(w, cuda_device)
    a = run_cuda(w, kernel=at.KERNEL_TC, t=t)
    b = run_cuda(w, kernel=at.KERNEL_TC, t=t)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_split_kv_agrees_with_the_unsplit_queue(cuda_device):
    # One SM of balancing width leaves the queue unsplit (it has at least 2 items).
    tree, hq, hkv = CASES[0]
    w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=37)
    t = device_inputs(w, cuda_device)
    split_plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    whole_plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC, num_sms=1)
    assert _split_items(split_plan) > 0 and _split_items(whole_plan) == 0
    assert whole_plan.workspace_bytes(at.OP_REPLAY_FWD) == 0
    a = run_cuda(w, plan=split_plan, t=t)
    b = run_cuda(w, plan=whole_plan, t=t)
    # The prompt side does not depend on the replay queue.
    for k in ("o_p", "lse_p", "dq_p"):
        assert np.array_equal(a[k], b[k]), k
    # Same pairs; the weights P are rounded to bf16 against another running max and
    # summed in another order.  Each side's row sum l carries a relative error of at
    # most 2^-9 (every term rounded to bf16), so lse differs by at most about 2^-8; O
    # by the rounding of P and of the bf16 output, a few 2^-9 of its magnitude.
    assert np.max(np.abs(a["o_r"] - b["o_r"])) <= 2 * 2.0 ** -8 * max(1.0, np.max(np.abs(b["o_r"])))
    assert np.max(np.abs(a["lse_r"] - b["lse_r"])) <= 2.0 ** -8 + 1e-5
    for k in ("dq_r", "dk_r", "dv_r", "dk_p", "dv_p"):
        assert rel_frob(a[k], b[k]) < 1e-2, (k, rel_frob(a[k], b[k]))


def test_split_kv_two_call_backward(cuda_device):
    tree, hq, hkv = CASES[3]
    w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=41)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    assert _split_items(plan) > 0
    compare(run_cuda(w, plan=plan, fused=False), run_oracle(w), "bf16")


def test_split_kv_with_the_persistent_schedule(cuda_device):
    tree, hq, hkv = CASES[1]
    w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=43)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC,
                             schedule=at.SCHED_PERSISTENT)
    assert _split_items(plan) > 0
    compare(run_cuda(w, plan=plan), run_oracle(w), "bf16")


def test_split_kv_forward_rejects_a_small_workspace(cuda_device):
    tree, hq, hkv = CASES[3]
    w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=47)
    t = device_inputs(w, cuda_device)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    need = plan.workspace_bytes(at.OP_REPLAY_FWD)
    assert need > 0
    o_r = torch.empty_like(t["q_r"])
    lse_r = torch.empty(w.hq, w.tree.total_resp, dtype=torch.float32, device=cuda_device)
    for ws in (None, torch.empty(need - 1, dtype=torch.uint8, device=cuda_device)):
        with pytest.raises(at.AugtreeError) as e:
            at.augtree_replay_fwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], o_r, lse_r, ws)
        assert e.value.status in (at.ERR_WORKSPACE_TOO_SMALL, at.ERR_INVALID_ARG)
    # A workspace must start on a 16-byte boundary (its partial states are written in
    # 16-byte vectors).
    big = torch.empty(need + 16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(at.AugtreeError) as e:
        at.augtree_replay_fwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], o_r, lse_r, big[8:])
    assert e.value.status == at.ERR_INVALID_ARG
    del e
