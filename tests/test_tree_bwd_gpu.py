"""The whole backward in one call (augtree_tree_bwd; AugTree paper, Sec. 3.2, Eq. 2): the
prompt K/V gradient is the sum over branches of the replay gradients plus the prompt's
own causal gradient, here accumulated per prompt KV tile in one pass.  Parity with the
fp64 oracle at the bf16 tolerances, agreement with the two-call path, split-K variants,
groups without responses, empty prompts, and determinism."""
import numpy as np
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import GRADS, compare, device_inputs, rel_frob, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

TREES = [
    W.Tree([300], [[129, 1, 200]]),
    W.Tree([150, 0, 70], [[1, 65, 130], [20, 0], [3]]),
    W.Tree([0, 129], [[64, 1, 2, 200], []]),        # empty prompt; a prompt without responses
    W.Tree([257, 40], [[1] * 9 + [128, 127, 300], []]),
    W.Tree([1000], [[700, 5, 260]]),
    W.Tree([333], [[]]),                             # prefill only
]


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4)])
def test_fused_backward_matches_oracle(cuda_device, ti, hq, hkv):
    w = W.custom(TREES[ti], hq=hq, hkv=hkv, d=128, dtype="bf16", seed=700 + ti, scale=1.0)
    compare(run_cuda(w, kernel=at.KERNEL_TC, fused=True), run_oracle(w), "bf16")


@pytest.mark.parametrize("num_sms", [1, 4, 100000])
def test_fused_backward_split_variants(cuda_device, num_sms):
    # 1 and 4 SMs split the prompt KV tiles over chunks of the response query tiles
    # (fp32 partials, reduced in split order into the bf16 gradient); 100000 leaves
    # them whole (written directly).
    w = W.custom(W.Tree([400, 130], [[300, 520, 90, 7], [60]]), hq=4, hkv=1, d=128, dtype="bf16", seed=19)
    compare(run_cuda(w, kernel=at.KERNEL_TC, num_sms=num_sms, fused=True), run_oracle(w), "bf16")


def test_fused_equals_two_call_path(cuda_device):
    w = W.custom(TREES[4], hq=8, hkv=2, d=128, dtype="bf16", seed=71)
    t = device_inputs(w, cuda_device)
    a = run_cuda(w, kernel=at.KERNEL_TC, t=t, fused=True)
    b = run_cuda(w, kernel=at.KERNEL_TC, t=t, fused=False)
    # The response gradients and every dQ come from the same kernels and inputs.
    for k in ("dq_p", "dq_r", "dk_r", "dv_r"):
        assert np.array_equal(a[k], b[k]), k
    # The prompt K/V gradient differs only in fp32 summation order and one bf16
    # rounding (the two-call path rounds the prefill part plus the fp32 replay sum).
    for k in ("dk_p", "dv_p"):
        assert rel_frob(a[k], b[k]) < 5e-3, (k, rel_frob(a[k], b[k]))


def test_fused_backward_is_deterministic(cuda_device):
    w = W.custom(W.Tree([400], [[300, 520, 90, 7]]), hq=4, hkv=1, d=128, dtype="bf16", seed=23)
    t = device_inputs(w, cuda_device)
    a = run_cuda(w, kernel=at.KERNEL_TC, t=t, num_sms=4, fused=True)
    b = run_cuda(w, kernel=at.KERNEL_TC, t=t, num_sms=4, fused=True)
    for k in GRADS:
        assert np.array_equal(a[k], b[k]), k


def test_fused_backward_simt_family(cuda_device):
    # fp32: the SIMT kernels run the two calls inside the one entry point.
    w = W.custom(TREES[1], hq=4, hkv=2, d=64, dtype="fp32", seed=77, scale=0.125)
    compare(run_cuda(w, kernel=at.KERNEL_SIMT, fused=True), run_oracle(w), "fp32")


def test_fused_backward_rejects_small_workspace(cuda_device):
    import torch
    w = W.custom(TREES[0], hq=4, hkv=2, d=128, dtype="bf16", seed=5)
    t = device_inputs(w, cuda_device)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    need = plan.workspace_bytes(at.OP_TREE_BWD)
    assert need > 0
    ws = torch.empty(need - 1, dtype=torch.uint8, device=cuda_device)
    outs = [torch.empty_like(t[k]) for k in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")]
    with pytest.raises(at.AugtreeError) as e:
        at.augtree_tree_bwd(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p, t["do_p"], t["q_r"], t["k_r"], t["v_r"],
                            o_r, lse_r, t["do_r"], *outs, ws)
    assert e.value.status == at.ERR_WORKSPACE_TOO_SMALL


def test_tree_bwd_output_alignment(cuda_device):
    """The query side writes dQ rows (and split-KV fp32 partials) in 32-byte stores when
    the base pointers are 32-byte aligned and in 16-byte stores otherwise: gradients
    and workspace at a 16-byte offset give the same bits as aligned ones (a tree whose
    replay queue splits, so the partial path runs too)."""
    import torch
    w = W.custom(W.Tree([4096, 300], [[2, 3, 1], [200, 9]]), hq=4, hkv=2, d=128, dtype="bf16", seed=83)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    assert int(plan.schedule(at.OP_REPLAY_FWD)[:, 4].max()) > 0
    t = {n: W.tensor_torch(w, n, cuda_device) for n in W.TENSORS}
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    nb = max(1, plan.workspace_bytes(at.OP_TREE_BWD))
    outs = []
    for off in (0, 16):
        def shifted(like):
            raw = torch.empty(like.numel() * like.element_size() + 64, dtype=torch.uint8, device=cuda_device)
            assert raw.data_ptr() % 32 == 0
            return raw[off:off + like.numel() * like.element_size()].view(like.dtype).view(like.shape)
        g = [shifted(t[n]) for n in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")]
        raw = torch.empty(nb + 64, dtype=torch.uint8, device=cuda_device)
        ws = raw[off:off + nb]
        at.augtree_tree_bwd(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p, t["do_p"], t["q_r"], t["k_r"], t["v_r"],
                            o_r, lse_r, t["do_r"], *g, ws)
        torch.cuda.synchronize()
        plan.check()
        outs.append([x.clone() for x in g])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
