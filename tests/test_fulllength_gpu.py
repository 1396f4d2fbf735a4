"""Element-wise parity at the configurations' real lengths, on one KV head.

The first rung of the parity ladder for the large configurations: the fp64 oracle on
one KV head and its query heads, at full length, compared element by element on all
ten outputs (O, lse, dQ, dK, dV of the prompt and of the responses) with the stated
tolerances (bf16: forward max-abs 1e-2, gradients relative Frobenius 2e-2).  Groups
are independent, so a group of a full-size run is compared exactly.

  * prompt-heavy: the full configuration runs on the GPU in the launch configuration
    the benchmark times (default plan, one fused backward call); group 0 (a 32,768-token
    prompt with 8 branches, whose prompt dK/dV sum over all 8 branches, Eq. 2) is
    compared on the last KV head;
  * mixed batch: the full configuration on the GPU, all 16 groups on one KV head;
  * response-heavy: its 1,024-token prompt with every fourth of its 64 branches (16
    branches at their real lengths, 1.3k to 16k tokens), run as its own batch.

The oracle runs per query head in a spawn process pool (tests/oracle_pool.py).
"""
import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import attention as A
from tests.gpu_util import compare, device_inputs
from tests.oracle_pool import oracle_one_kv_head

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(w, dev):
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, dev)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    g = at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                    t["do_p"], t["do_r"])
    plan.check()
    out = dict(o_p=o_p, lse_p=lse_p, o_r=o_r, lse_r=lse_r)
    out.update(dict(zip(("dq_p", "dk_p", "dv_p", "dq_r", "dk_r", "dv_r"), g)))
    del t
    return out


def _check_groups(w, out, groups, kv, dev):
    """Compares groups `groups` of run `out` with the oracle on KV head kv."""
    r = w.hq // w.hkv
    hs = list(range(kv * r, (kv + 1) * r))
    po, bb, ro = w.tree.offsets()
    rows_p = np.concatenate([np.arange(po[g], po[g + 1]) for g in groups]).astype(np.int64)
    rows_r = np.concatenate([np.arange(ro[bb[g]], ro[bb[g + 1]]) for g in groups]).astype(np.int64)
    sub = W.Tree([w.tree.prompt_lens[g] for g in groups], [w.tree.branch_lens[g] for g in groups])
    host = {}
    for n in W.TENSORS:
        rows = rows_p if n.endswith("_p") else rows_r
        host[n] = W.tensor_rows_np(w, n, rows=rows, heads=(hs if n[0] in "qd" else [kv]))
    ref = oracle_one_kv_head(host, sub.offsets(), A.default_scale(w.d))
    ip = torch.as_tensor(rows_p, device=dev)
    ir = torch.as_tensor(rows_r, device=dev)
    ih = torch.as_tensor(hs, device=dev)
    got = {
        "o_p": out["o_p"][ip][:, ih], "o_r": out["o_r"][ir][:, ih],
        "lse_p": out["lse_p"][ih][:, ip], "lse_r": out["lse_r"][ih][:, ir],
        "dq_p": out["dq_p"][ip][:, ih], "dq_r": out["dq_r"][ir][:, ih],
        "dk_p": out["dk_p"][ip, kv:kv + 1], "dv_p": out["dv_p"][ip, kv:kv + 1],
        "dk_r": out["dk_r"][ir, kv:kv + 1], "dv_r": out["dv_r"][ir, kv:kv + 1],
    }
    got = {k: v.double().cpu().numpy() for k, v in got.items()}
    return compare(got, ref, "bf16")


def test_prompt_heavy_group0_full_length_one_kv_head(cuda_device):
    w = W.workload("prompt_heavy")
    out = _run(w, cuda_device)
    errs = _check_groups(w, out, [0], w.hkv - 1, cuda_device)
    print("prompt-heavy group 0:", {k: f"{v:.2e}" for k, v in errs.items()})
    del out
    torch.cuda.empty_cache()


def test_mixed_all_groups_full_length_one_kv_head(cuda_device):
    w = W.workload("mixed")
    out = _run(w, cuda_device)
    errs = _check_groups(w, out, list(range(w.tree.n_groups)), 2, cuda_device)
    print("mixed:", {k: f"{v:.2e}" for k, v in errs.items()})
    del out
    torch.cuda.empty_cache()


def test_response_heavy_sixteen_branches_full_length_one_kv_head(cuda_device):
    full = W.workload("response_heavy")
    tree = W.Tree(full.tree.prompt_lens, [full.tree.branch_lens[0][::4]])
    w = W.custom(tree, full.hq, full.hkv, full.d, full.dtype, full.seed, full.scale, name="response_heavy_16")
    out = _run(w, cuda_device)
    errs = _check_groups(w, out, [0], 5, cuda_device)
    print("response-heavy 16 branches:", {k: f"{v:.2e}" for k, v in errs.items()})
    del out
    torch.cuda.empty_cache()
