"""The flattened-per-pair mode through the C ABI (the b=0 ring fallback's semantics,
AugTree Sec. 3.4, and the MegaN/MegaR ablation's no-reuse baseline of Sec. 4.3, on one
GPU): every prompt-response pair runs as its own group with its own copy of the prompt.

The flattened batch is built from a tree batch by copying each group's prompt rows
(Q, K, V) once per branch; the prompt's upstream gradient goes wholly to the group's
first pair (zero in the others).  Checked against the oracle's plain flattened form
(oracle.tree_attention_flat), at the bf16 tolerances:
  * every pair's prompt rows reproduce O_P and lse_P (identical across pairs);
  * response rows and their gradients are the pair's own;
  * the sum over a group's pairs of the per-pair prompt gradients is the tree's dQ_P,
    dK_P, dV_P (Eq. 2), and agrees with the tree run's own prompt gradients."""
import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import attention as A
from tests.gpu_util import TOL, compare, device_inputs, host_inputs, rel_frob, run_cuda

pytestmark = pytest.mark.gpu


def flatten(w, t):
    """(flattened workload tree, flattened device tensors, pair -> (group, branch rows))."""
    po, bb, ro = (np.asarray(x, np.int64) for x in w.tree.offsets())
    prompts, branches, idx, pairs, first = [], [], [], [], []
    for g in range(w.tree.n_groups):
        bl = w.tree.branch_lens[g]
        for k, li in enumerate(bl):
            prompts.append(w.tree.prompt_lens[g])
            branches.append([li])
            idx.append(np.arange(po[g], po[g + 1]))
            pairs.append(g)
            first.append(k == 0)
    tree = W.Tree(prompts, branches)
    gather = torch.as_tensor(np.concatenate(idx) if idx else np.zeros(0, np.int64), device=t["q_p"].device)
    tf = {n: t[n][gather].contiguous() for n in ("q_p", "k_p", "v_p", "do_p")}
    # dO_P enters once: all of it in the group's first pair.
    keep = torch.cat([torch.full((lp,), 1.0 if f else 0.0, device=gather.device)
                      for lp, f in zip(prompts, first)]) if prompts else torch.zeros(0, device=gather.device)
    tf["do_p"] = (tf["do_p"].float() * keep[:, None, None]).to(t["do_p"].dtype)
    for n in ("q_r", "k_r", "v_r", "do_r"):
        tf[n] = t[n]
    return tree, tf, pairs


@pytest.mark.parametrize("tree", [W.Tree([300, 129], [[129, 1, 200], [64, 3]]), W.Tree([700], [[300, 20, 5, 128]])])
def test_flattened_mode_matches_the_flattened_oracle(cuda_device, tree):
    w = W.custom(tree, hq=8, hkv=2, d=128, dtype="bf16", seed=61)
    t = device_inputs(w, cuda_device)
    ftree, tf, pairs = flatten(w, t)
    wf = W.custom(ftree, w.hq, w.hkv, w.d, w.dtype, w.seed, w.scale, name="flattened")
    got = run_cuda(wf, t=tf)
    ref = A.tree_attention_flat(host_inputs(w), w.tree.offsets(), A.default_scale(w.d))
    fwd_tol, grad_tol = TOL["bf16"]
    po = np.asarray(w.tree.offsets()[0], np.int64)
    fo = np.asarray(ftree.offsets()[0], np.int64)
    sums = {k: np.zeros_like(ref[k]) for k in ("dq_p", "dk_p", "dv_p")}
    for pi, g in enumerate(pairs):
        a, b = fo[pi], fo[pi + 1]
        p0, p1 = po[g], po[g + 1]
        assert np.max(np.abs(got["o_p"][a:b] - ref["o_p"][p0:p1]), initial=0) <= fwd_tol, pi
        assert np.max(np.abs(got["lse_p"][:, a:b] - ref["lse_p"][:, p0:p1]), initial=0) <= fwd_tol, pi
        for k in sums:
            sums[k][p0:p1] += got[k][a:b]
    resp = {k: got[k] for k in ("o_r", "lse_r", "dq_r", "dk_r", "dv_r")}
    resp.update(sums)
    compare(resp, ref, "bf16", keys=tuple(resp))
    tree_run = run_cuda(w, t=t)
    for k in ("dq_p", "dk_p", "dv_p"):
        assert rel_frob(sums[k], tree_run[k]) <= grad_tol, k
