"""Parity at the benchmark sizes, in the configuration bench.py times (default plan,
tensor-core path).

The oracle cannot evaluate the full configurations (the long one is about 1 PFLOP of
fp64 work per KV head), so each configuration is checked three ways:
  1. sampled rows: O, lse and dQ of a query row need only that row's valid keys
     (Eq. 1) and its own Delta, so the oracle computes them exactly, row by row, for a
     seeded sample of rows (first/last rows of groups and branches included);
  2. exact gradient identities over every (group, KV head), which hold at any size:
     sum_j dV_j = sum_i dO_i,  sum_j dK_j = 0,  sum_i <dQ_i, q_i> = sum_j <dK_j, k_j>;
  3. full-tensor parity on the same structure scaled down (lengths / 8 or / 16) for one
     KV head and its query heads.
"""
import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import attention as A
from tests.gpu_util import TOL, compare, device_inputs, host_inputs, rel_frob

pytestmark = pytest.mark.gpu

FULL = ["prompt_heavy", "response_heavy", "mixed", "long"]


def run_full(w, dev):
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, dev)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    g = at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                    t["do_p"], t["do_r"])
    plan.check()
    out = dict(o_p=o_p, lse_p=lse_p, o_r=o_r, lse_r=lse_r)
    out.update(dict(zip(("dq_p", "dk_p", "dv_p", "dq_r", "dk_r", "dv_r"), g)))
    return t, out


def sample_rows(w, rng, n=12):
    """Seeded sample of (kind, row): group/branch boundaries plus random rows."""
    po, bb, ro = w.tree.offsets()
    rows = []
    for g in range(w.tree.n_groups):
        if po[g + 1] > po[g]:
            rows += [("p", int(po[g])), ("p", int(po[g + 1]) - 1)]
    for b in range(w.tree.n_branches):
        if ro[b + 1] > ro[b]:
            rows += [("r", int(ro[b])), ("r", int(ro[b + 1]) - 1)]
    rng.shuffle(rows)
    rows = rows[:n]
    if w.tree.total_prompt:
        rows += [("p", int(x)) for x in rng.integers(0, w.tree.total_prompt, size=n // 2)]
    if w.tree.total_resp:
        rows += [("r", int(x)) for x in rng.integers(0, w.tree.total_resp, size=n // 2)]
    return rows


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows_and_identities(cuda_device, name):
    w = W.workload(name)
    t, out = run_full(w, cuda_device)
    fwd_tol, grad_tol = TOL["bf16"]
    offs = w.tree.offsets()
    rng = np.random.default_rng(1234)
    r = w.hq // w.hkv
    scale = A.default_scale(w.d)
    # 1. sampled rows, two query heads (first and last) of one of two sampled KV heads
    kv_heads = sorted(set(int(x) for x in rng.integers(0, w.hkv, size=2)))
    kv_cache = {kv: {n: W.tensor_rows_np(w, n, heads=[kv]) for n in ("k_p", "v_p", "k_r", "v_r")}
                for kv in kv_heads}
    for kind, row in sample_rows(w, rng):
        kv = kv_heads[int(rng.integers(0, len(kv_heads)))]
        c = kv_cache[kv]
        heads = [kv * r, kv * r + r - 1]
        (pa, pb), (ra, rb) = A.row_key_set(kind, row, offs)
        kk = np.concatenate([c["k_p"][pa:pb], c["k_r"][ra:rb]])
        vv = np.concatenate([c["v_p"][pa:pb], c["v_r"][ra:rb]])
        q = W.tensor_rows_np(w, "q_" + kind, rows=[row], heads=heads)
        do = W.tensor_rows_np(w, "do_" + kind, rows=[row], heads=heads)
        o, lse, dq = A.rows_forward_backward(q, np.repeat(kk, len(heads), axis=1),
                                             np.repeat(vv, len(heads), axis=1), scale, do)
        hs = torch.tensor(heads, device=cuda_device)
        go = out["o_" + kind][row, hs].double().cpu().numpy()
        gl = out["lse_" + kind][hs, row].double().cpu().numpy()
        gq = out["dq_" + kind][row, hs].double().cpu().numpy()
        assert np.max(np.abs(go - o[0])) <= fwd_tol, (kind, row)
        assert np.max(np.abs(gl - lse[:, 0])) <= fwd_tol, (kind, row)
        assert rel_frob(gq, dq[0]) <= grad_tol, (kind, row, rel_frob(gq, dq[0]))
    del kv_cache
    # 2. gradient identities per (group, KV head), fp64 sums on the device
    po, bb, ro = offs
    d64 = {k: out[k] for k in ("dq_p", "dk_p", "dv_p", "dq_r", "dk_r", "dv_r")}
    for g in range(w.tree.n_groups):
        p0, p1 = int(po[g]), int(po[g + 1])
        r0, r1 = int(ro[int(bb[g])]), int(ro[int(bb[g + 1])])
        for kv in range(w.hkv):
            hs = slice(kv * r, (kv + 1) * r)
            dv = torch.cat([d64["dv_p"][p0:p1, kv], d64["dv_r"][r0:r1, kv]]).double()
            dk = torch.cat([d64["dk_p"][p0:p1, kv], d64["dk_r"][r0:r1, kv]]).double()
            k = torch.cat([t["k_p"][p0:p1, kv], t["k_r"][r0:r1, kv]]).double()
            do = torch.cat([t["do_p"][p0:p1, hs], t["do_r"][r0:r1, hs]]).double()
            dq = torch.cat([d64["dq_p"][p0:p1, hs], d64["dq_r"][r0:r1, hs]]).double()
            q = torch.cat([t["q_p"][p0:p1, hs], t["q_r"][r0:r1, hs]]).double()
            if dv.numel() == 0:
                continue
            e1 = (dv.sum(0) - do.sum((0, 1))).abs().max() / dv.norm()
            e2 = dk.sum(0).abs().max() / dk.norm()
            e3 = ((dq * q).sum() - (dk * k).sum()).abs() / (dq.norm() * q.norm())
            assert float(e1) <= grad_tol and float(e2) <= grad_tol and float(e3) <= grad_tol, \
                (g, kv, float(e1), float(e2), float(e3))
    del t, out
    torch.cuda.empty_cache()


def scaled(name):
    """The configuration's structure with lengths scaled down, same heads and D."""
    w = W.workload(name)
    div = {"prompt_heavy": 8, "response_heavy": 16, "mixed": 16, "long": 64}[name]
    tree = W.Tree([max(1, x // div) for x in w.tree.prompt_lens],
                  [[max(1, x // div) for x in b] for b in w.tree.branch_lens])
    if name == "mixed":
        tree = W.Tree(tree.prompt_lens[:6], tree.branch_lens[:6])
    return W.custom(tree, w.hq, w.hkv, w.d, w.dtype, w.seed, w.scale, name=name + "_scaled")


@pytest.mark.parametrize("name", FULL)
def test_scaled_structure_full_parity_one_kv_head(cuda_device, name):
    w = scaled(name)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16)
    t = device_inputs(w, cuda_device)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    g = at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                    t["do_p"], t["do_r"])
    plan.check()
    kv = w.hkv - 1
    r = w.hq // w.hkv
    hq_sel = list(range(kv * r, (kv + 1) * r))
    got = dict(o_p=o_p[:, hq_sel], o_r=o_r[:, hq_sel], lse_p=lse_p[hq_sel], lse_r=lse_r[hq_sel],
               dq_p=g[0][:, hq_sel], dk_p=g[1][:, kv:kv + 1], dv_p=g[2][:, kv:kv + 1],
               dq_r=g[3][:, hq_sel], dk_r=g[4][:, kv:kv + 1], dv_r=g[5][:, kv:kv + 1])
    got = {k: v.double().cpu().numpy() for k, v in got.items()}
    host = {n: W.tensor_rows_np(w, n, heads=(hq_sel if n[0] in "qd" else [kv])) for n in W.TENSORS}
    ref = A.tree_attention_direct(host, w.tree.offsets(), A.default_scale(w.d))
    compare(got, ref, "bf16")
