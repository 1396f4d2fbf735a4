"""Parity of the tcgen05 forward (prefill + replay, bf16 in, fp32 accumulate) with the
fp64 oracle: ragged trees over several 128-row tiles with tails, one- and
two-head thread blocks (even and odd GQA ratios), empty prompts and branches."""
import numpy as np
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from tests.gpu_util import compare, run_cuda_fwd, run_oracle_fwd

pytestmark = pytest.mark.gpu

TREES = [
    W.Tree([300], [[129, 1, 200]]),
    W.Tree([150, 0, 70], [[1, 65, 130], [20, 0], [3]]),
    W.Tree([0, 129], [[64, 1, 2, 200], []]),
    W.Tree([257], [[1] * 9 + [128, 127, 300]]),
    W.Tree([1000], [[700, 5, 260]]),
]


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4), (6, 2)])
def test_tc_forward_matches_oracle(cuda_device, ti, hq, hkv):
    w = W.custom(TREES[ti], hq=hq, hkv=hkv, d=128, dtype="bf16", seed=400 + ti, scale=1.0)
    got = run_cuda_fwd(w, kernel=at.KERNEL_TC)
    errs = compare(got, run_oracle_fwd(w), "bf16", keys=("o_p", "o_r", "lse_p", "lse_r"))


def test_tc_forward_large_scores(cuda_device):
    """Q and K scaled by 4 (exact in bf16): scores spread 16x wider, so the running max
    grows past the lazy-rescale threshold and O is rescaled in TMEM.  Single keys then
    dominate their rows and |O| reaches about 4.3, where storing O in bf16 (8 significant
    bits) moves it by up to 2^-8 |O|.  The bound is the stated 1e-2 on the arithmetic
    plus that output rounding; tests/test_bf16_output_bound.py derives it on this very
    input (an ideal bf16-P forward exceeds a plain 1e-2 and stays within this bound).
    lse is fp32 and keeps the plain 1e-2."""
    import torch
    from oracle import attention as A
    w = W.custom(TREES[4], hq=4, hkv=2, d=128, dtype="bf16", seed=77)
    t = {n: W.tensor_torch(w, n, cuda_device) for n in W.TENSORS}
    h = {n: W.tensor_rows_np(w, n) for n in W.TENSORS}
    for n in ("q_p", "k_p", "q_r", "k_r"):
        t[n] = t[n] * 4
        h[n] = h[n] * 4
    got = run_cuda_fwd(w, kernel=at.KERNEL_TC, t=t)
    ref = A.tree_attention_direct(h, w.tree.offsets(), A.default_scale(w.d), grad=False)
    for k in ("o_p", "o_r"):
        err = np.abs(got[k] - ref[k])
        assert np.all(err <= 1e-2 + 2.0 ** -8 * np.abs(ref[k])), (k, float(err.max()))
    for k in ("lse_p", "lse_r"):
        assert np.max(np.abs(got[k] - ref[k])) <= 1e-2, k


def test_tc_forward_many_items_per_block(cuda_device):
    """The forward runs one block per SM, each taking items in queue order until the
    queue is exhausted, with consecutive items overlapped.  A queue many times the SM
    count, of items from 1 to 15 KV tiles (short and long prompts, one- to three-tile
    branches), matches the oracle; repeated calls into outputs filled with NaN give
    bit-identical results, so every item is computed on every call (the work counter
    starts from zero each launch) whichever block takes it."""
    import torch
    rng = np.random.default_rng(5)
    prompts = [int(x) for x in rng.integers(0, 1500, size=24)]
    branches = [[int(x) for x in rng.integers(1, 300, size=int(rng.integers(1, 6)))] for _ in prompts]
    w = W.custom(W.Tree(prompts, branches), hq=8, hkv=2, d=128, dtype="bf16", seed=61)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    n_sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    assert len(plan.schedule(at.OP_REPLAY_FWD)) > 4 * n_sms and len(plan.schedule(at.OP_PREFILL_FWD)) > 4 * n_sms
    t = {n: W.tensor_torch(w, n, cuda_device) for n in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")}
    nb = plan.workspace_bytes(at.OP_REPLAY_FWD)
    ws = torch.empty(nb, dtype=torch.uint8, device=cuda_device) if nb else None
    runs = []
    for _ in range(3):
        o_p = torch.full_like(t["q_p"], float("nan"))
        o_r = torch.full_like(t["q_r"], float("nan"))
        lse_p = torch.full((w.hq, w.tree.total_prompt), float("nan"), dtype=torch.float32, device=cuda_device)
        lse_r = torch.full((w.hq, w.tree.total_resp), float("nan"), dtype=torch.float32, device=cuda_device)
        at.augtree_prefill_fwd(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p)
        at.augtree_replay_fwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], o_r, lse_r, ws)
        torch.cuda.synchronize()
        plan.check()
        runs.append({"o_p": o_p, "lse_p": lse_p, "o_r": o_r, "lse_r": lse_r})
    for r in runs[1:]:
        for k in r:
            assert torch.equal(r[k], runs[0][k]), k
    got = {k: v.double().cpu().numpy() for k, v in runs[0].items()}
    compare(got, run_oracle_fwd(w), "bf16", keys=("o_p", "o_r", "lse_p", "lse_r"))


def test_tc_forward_output_alignment(cuda_device):
    """The forward writes each output row in 32-byte stores when the output's base is
    32-byte aligned and in 16-byte stores otherwise: an output that starts 16 bytes into
    an allocation gets the same bits as an aligned one (split-KV replay included, whose
    partial states go to a workspace at a 16-byte offset as well)."""
    import torch
    for tree, hq, hkv in ((TREES[4], 8, 2), (W.Tree([4096], [[2, 3, 1]]), 4, 2)):
        w = W.custom(tree, hq=hq, hkv=hkv, d=128, dtype="bf16", seed=71)
        plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
        t = {n: W.tensor_torch(w, n, cuda_device) for n in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")}
        nb = plan.workspace_bytes(at.OP_REPLAY_FWD)
        outs = []
        for off in (0, 16):
            def shifted(like):
                raw = torch.empty(like.numel() * like.element_size() + 64, dtype=torch.uint8, device=cuda_device)
                assert raw.data_ptr() % 32 == 0
                return raw[off:off + like.numel() * like.element_size()].view(like.dtype).view(like.shape)
            o_p, o_r = shifted(t["q_p"]), shifted(t["q_r"])
            lse_p = torch.empty(w.hq, w.tree.total_prompt, dtype=torch.float32, device=cuda_device)
            lse_r = torch.empty(w.hq, w.tree.total_resp, dtype=torch.float32, device=cuda_device)
            ws = None
            if nb:
                raw = torch.empty(nb + 64, dtype=torch.uint8, device=cuda_device)
                ws = raw[off:off + nb]
            at.augtree_prefill_fwd(plan, t["q_p"], t["k_p"], t["v_p"], o_p, lse_p)
            at.augtree_replay_fwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], o_r, lse_r, ws)
            torch.cuda.synchronize()
            plan.check()
            outs.append([x.clone() for x in (o_p, o_r, lse_p, lse_r)])
        for a, b in zip(*outs):
            assert torch.equal(a, b)
