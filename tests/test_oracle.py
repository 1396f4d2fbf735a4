"""Pins of the fp64 oracle against things other than itself (CPU only).

AugTree paper, "Splitting Prompt Prefill from Response Replay for Context-Parallel
Long-Context LLM Post-Training":
  Sec. 2.2      attention O = softmax(Q K^T / sqrt(D_h) + M) V
  Sec. 2.1      replay tree: responses see the whole prompt and their own prefix,
                never a sibling; the prompt never sees a response
  Sec. 3.2 Eq.1 valid KV context of a response token; Eq. 2 prompt gradient = sum
                over branches
  Sec. 3.3      partial online-softmax states merge associatively

Each test checks the oracle against an independent route: a hand-written key-set
table, per-row brute force with math.fsum, torch's scaled_dot_product_attention in
float64 with an explicit tree mask (and its autograd), central finite differences,
closed-form special cases, and exact gradient identities.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import invariants as INV
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(tree, hq, hkv, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    lp, lr = tree.total_prompt, tree.total_resp
    t = {
        "q_p": rng.standard_normal((lp, hq, d)) * scale,
        "k_p": rng.standard_normal((lp, hkv, d)) * scale,
        "v_p": rng.standard_normal((lp, hkv, d)),
        "q_r": rng.standard_normal((lr, hq, d)) * scale,
        "k_r": rng.standard_normal((lr, hkv, d)) * scale,
        "v_r": rng.standard_normal((lr, hkv, d)),
        "do_p": rng.standard_normal((lp, hq, d)),
        "do_r": rng.standard_normal((lr, hq, d)),
    }
    return t


TREES = [
    W.Tree([5], [[3, 4]]),
    W.Tree([7, 3], [[1, 6, 2], [4]]),
    W.Tree([0, 4], [[3, 2], [0, 5]]),          # empty prompt, empty branch
    W.Tree([6, 2, 3], [[], [3], [1, 1, 1]]),   # group without branches
    W.Tree([0], [[0]]),                        # everything empty
]


# ------------------------------------------------------------------------------
# Key sets: the hand-written table of Eq. 1 (tests/golden/eq1_key_sets.json)
# ------------------------------------------------------------------------------
def test_key_sets_match_hand_written_table():
    g = json.load(open(os.path.join(GOLDEN, "eq1_key_sets.json")))
    tree = W.Tree(g["tree"]["prompt_lens"], g["tree"]["branch_lens"])
    offs = tree.offsets()
    lp, lr = tree.total_prompt, tree.total_resp
    names = [f"P{j}" for j in range(lp)] + [f"R{j}" for j in range(lr)]
    nk = lp + lr
    # Zero keys => every valid key gets the same weight; one-hot values reveal the set.
    eye = np.eye(nk)
    t = {
        "q_p": np.ones((lp, 1, nk)), "k_p": np.zeros((lp, 1, nk)), "v_p": eye[:lp, None, :],
        "q_r": np.ones((lr, 1, nk)), "k_r": np.zeros((lr, 1, nk)), "v_r": eye[lp:, None, :],
        "do_p": np.zeros((lp, 1, nk)), "do_r": np.zeros((lr, 1, nk)),
    }
    for fn in (A.tree_attention_flat, A.tree_attention_direct):
        out = fn(t, offs, 1.0, grad=False)
        for kind, rows in (("p", "prompt_rows"), ("r", "response_rows")):
            o = out["o_p"] if kind == "p" else out["o_r"]
            for name, want in g[rows].items():
                i = int(name[1:])
                got = [names[j] for j in range(nk) if o[i, 0, j] > 0]
                assert got == want, (fn.__name__, name, got, want)
                np.testing.assert_allclose(o[i, 0][o[i, 0] > 0], 1.0 / len(want), rtol=1e-15)
    # The per-row key-set function agrees with the table too.
    for kind, rows in (("p", "prompt_rows"), ("r", "response_rows")):
        for name, want in g[rows].items():
            (pa, pb), (ra, rb) = A.row_key_set(kind, int(name[1:]), offs)
            got = [f"P{j}" for j in range(pa, pb)] + [f"R{j}" for j in range(ra, rb)]
            assert got == want


# ------------------------------------------------------------------------------
# Brute force per row (explicit exp / fsum), written from the rules of Sec. 2.1
# ------------------------------------------------------------------------------
def brute_rows(t, tree, hq, hkv, scale):
    """Returns o_p, lse_p, o_r, lse_r by explicit loops over each row's key list."""
    r = hq // hkv
    o_p = np.zeros_like(t["q_p"]); o_r = np.zeros_like(t["q_r"])
    lse_p = np.full((hq, tree.total_prompt), -np.inf); lse_r = np.full((hq, tree.total_resp), -np.inf)
    p_base, r_base = 0, 0
    for lp, bl in zip(tree.prompt_lens, tree.branch_lens):
        jobs = []
        for i in range(lp):   # prompt row i sees prompt keys 0..i of its group
            jobs.append(("p", p_base + i, [("p", p_base + j) for j in range(i + 1)]))
        rb = r_base
        for li in bl:         # response row t sees every prompt key and own keys 0..t
            for tt in range(li):
                keys = [("p", p_base + j) for j in range(lp)] + [("r", rb + j) for j in range(tt + 1)]
                jobs.append(("r", rb + tt, keys))
            rb += li
        for kind, row, keys in jobs:
            for h in range(hq):
                kv = h // r
                q = t["q_" + kind][row, h]
                sc = [scale * math.fsum(q[c] * t["k_" + kk][kr, kv, c] for c in range(q.shape[0]))
                      for kk, kr in keys]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                l = math.fsum(e)
                o = np.array([math.fsum(e[n] * t["v_" + kk][kr, kv, c] for n, (kk, kr) in enumerate(keys)) / l
                              for c in range(q.shape[0])])
                if kind == "p":
                    o_p[row, h] = o; lse_p[h, row] = m + math.log(l)
                else:
                    o_r[row, h] = o; lse_r[h, row] = m + math.log(l)
        p_base += lp
        r_base += sum(bl)
    return o_p, lse_p, o_r, lse_r


@pytest.mark.parametrize("ti", range(4))
def test_forward_matches_brute_force(ti):
    tree = TREES[ti]
    hq, hkv, d = 4, 2, 3
    t = rand_inputs(tree, hq, hkv, d, seed=ti)
    scale = A.default_scale(d)
    o_p, lse_p, o_r, lse_r = brute_rows(t, tree, hq, hkv, scale)
    for fn in (A.tree_attention_flat, A.tree_attention_direct):
        out = fn(t, tree.offsets(), scale, grad=False)
        np.testing.assert_allclose(out["o_p"], o_p, rtol=0, atol=1e-13)
        np.testing.assert_allclose(out["o_r"], o_r, rtol=0, atol=1e-13)
        np.testing.assert_allclose(out["lse_p"], lse_p, rtol=0, atol=1e-13)
        np.testing.assert_allclose(out["lse_r"], lse_r, rtol=0, atol=1e-13)


# ------------------------------------------------------------------------------
# Library special case: torch SDPA (float64, explicit boolean tree mask) + autograd
# ------------------------------------------------------------------------------
def sdpa_tree(t, tree, hq, hkv, scale):
    """Per group: one SDPA call over [P; R_1; ...; R_G] with the tree mask; gradients
    of sum(dO * O) by torch autograd.  Returns a dict like the oracle's."""
    r = hq // hkv
    names = ["q_p", "k_p", "v_p", "q_r", "k_r", "v_r"]
    leaves = {n: torch.tensor(t[n], dtype=torch.float64, requires_grad=True) for n in names}
    outs = {"o_p": [], "o_r": [], "lse_p": [], "lse_r": []}
    loss = 0.0
    prompt_off, branch_begin, resp_off = tree.offsets()
    o_p = torch.zeros_like(leaves["q_p"]); o_r = torch.zeros_like(leaves["q_r"])
    pieces_p, pieces_r = [], []
    for g in range(tree.n_groups):
        p0, p1 = int(prompt_off[g]), int(prompt_off[g + 1])
        rr0, rr1 = int(resp_off[int(branch_begin[g])]), int(resp_off[int(branch_begin[g + 1])])
        lp, lr = p1 - p0, rr1 - rr0
        n = lp + lr
        if n == 0:
            continue
        # branch id per row: -1 for the prompt
        bid = np.full(n, -1)
        for b in range(int(branch_begin[g]), int(branch_begin[g + 1])):
            bid[lp + int(resp_off[b]) - rr0: lp + int(resp_off[b + 1]) - rr0] = b
        idx = np.arange(n)
        qi, kj = idx[:, None], idx[None, :]
        mask = ((bid[kj] == -1) & ((bid[qi] != -1) | (kj <= qi))) | ((bid[kj] == bid[qi]) & (bid[qi] != -1) & (kj <= qi))
        q = torch.cat([leaves["q_p"][p0:p1], leaves["q_r"][rr0:rr1]], 0)
        k = torch.cat([leaves["k_p"][p0:p1], leaves["k_r"][rr0:rr1]], 0)
        v = torch.cat([leaves["v_p"][p0:p1], leaves["v_r"][rr0:rr1]], 0)
        k = k.repeat_interleave(r, dim=1)
        v = v.repeat_interleave(r, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(
            q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
            attn_mask=torch.tensor(mask), scale=scale).transpose(0, 1)
        do = torch.cat([torch.tensor(t["do_p"][p0:p1]), torch.tensor(t["do_r"][rr0:rr1])], 0)
        loss = loss + (o * do).sum()
        pieces_p.append((p0, p1, o[:lp]))
        pieces_r.append((rr0, rr1, o[lp:]))
    if torch.is_tensor(loss):
        loss.backward()
    res = {n.replace("q_", "dq_").replace("k_", "dk_").replace("v_", "dv_"):
           (leaves[n].grad.numpy() if leaves[n].grad is not None else np.zeros_like(t[n]))
           for n in names}
    op = np.zeros_like(t["q_p"]); orr = np.zeros_like(t["q_r"])
    for p0, p1, o in pieces_p:
        op[p0:p1] = o.detach().numpy()
    for r0, r1, o in pieces_r:
        orr[r0:r1] = o.detach().numpy()
    res["o_p"], res["o_r"] = op, orr
    return res


@pytest.mark.parametrize("ti", range(5))
@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (3, 1)])
def test_matches_sdpa_with_tree_mask(ti, heads):
    tree = TREES[ti]
    hq, hkv = heads
    d = 8
    t = rand_inputs(tree, hq, hkv, d, seed=10 + ti)
    scale = A.default_scale(d)
    ref = sdpa_tree(t, tree, hq, hkv, scale)
    for fn in (A.tree_attention_flat, A.tree_attention_direct):
        out = fn(t, tree.offsets(), scale, grad=True)
        for k in ("o_p", "o_r", "dq_p", "dk_p", "dv_p", "dq_r", "dk_r", "dv_r"):
            np.testing.assert_allclose(out[k], ref[k], rtol=0, atol=1e-12, err_msg=f"{fn.__name__} {k}")


# ------------------------------------------------------------------------------
# Central finite differences of L = sum(dO * O)
# ------------------------------------------------------------------------------
def test_backward_matches_finite_differences():
    tree = W.Tree([5], [[3, 4]])
    hq, hkv, d = 2, 1, 4
    t = rand_inputs(tree, hq, hkv, d, seed=3)
    scale = A.default_scale(d)
    offs = tree.offsets()

    def loss(tt):
        o = A.tree_attention_direct(tt, offs, scale, grad=False)
        return float(np.sum(o["o_p"] * tt["do_p"]) + np.sum(o["o_r"] * tt["do_r"]))

    g = A.tree_attention_flat(t, offs, scale, grad=True)
    rng = np.random.default_rng(99)
    eps = 1e-6
    for name in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r"):
        for _ in range(3):
            u = rng.standard_normal(t[name].shape)
            tp = dict(t); tp[name] = t[name] + eps * u
            tm = dict(t); tm[name] = t[name] - eps * u
            fd = (loss(tp) - loss(tm)) / (2 * eps)
            an = float(np.sum(g["d" + name] * u))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


# ------------------------------------------------------------------------------
# The merge (+) of partial states, Sec. 3.3
# ------------------------------------------------------------------------------
def test_merge_of_key_partition_equals_single_pass():
    rng = np.random.default_rng(5)
    m, n, d = 6, 40, 8
    q, k, v = rng.standard_normal((m, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    scale = 0.7
    o_full, lse_full = A.partial_state(q, k, v, scale)
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, n), size=3, replace=False))
        parts = np.split(np.arange(n), cuts)
        states = [A.partial_state(q, k[p], v[p], scale) for p in parts]
        # left fold, right fold and a shuffled order must all agree with one pass
        acc = states[0]
        for s in states[1:]:
            acc = A.lse_merge(*acc, *s)
        racc = states[-1]
        for s in reversed(states[:-1]):
            racc = A.lse_merge(*s, *racc)
        order = rng.permutation(len(states))
        sacc = states[order[0]]
        for i in order[1:]:
            sacc = A.lse_merge(*sacc, *states[i])
        for o, l in (acc, racc, sacc):
            np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l, lse_full, rtol=0, atol=1e-12)


def test_merge_identity_and_empty_states():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((3, 4)); lse = rng.standard_normal(3)
    z, ninf = np.zeros((3, 4)), np.full(3, -np.inf)
    for args in ((o, lse, z, ninf), (z, ninf, o, lse)):
        mo, ml = A.lse_merge(*args)
        np.testing.assert_array_equal(mo, o)
        np.testing.assert_array_equal(ml, lse)
    mo, ml = A.lse_merge(z, ninf, z, ninf)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    # An empty key subset is the identity state.
    eo, el = A.partial_state(rng.standard_normal((3, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert np.all(eo == 0) and np.all(np.isneginf(el))
    # Closed form with two single keys: weights are a logistic of the score gap.
    mo, ml = A.lse_merge(np.ones((1, 1)), np.array([0.0]), np.zeros((1, 1)), np.array([math.log(3.0)]))
    assert abs(mo[0, 0] - 0.25) < 1e-15 and abs(ml[0] - math.log(4.0)) < 1e-15


# ------------------------------------------------------------------------------
# Tree (Eq. 1, prompt once) == flattened per pair (Sec. 2.1 / b=0 fallback)
# ------------------------------------------------------------------------------
def test_tree_equals_flattened_random():
    rng = np.random.default_rng(7)
    for trial in range(6):
        tree = W.random_tree(rng, n_groups=3, max_prompt=9, max_branches=4, max_resp=7)
        hq, hkv, d = 4, 2, 5
        t = rand_inputs(tree, hq, hkv, d, seed=100 + trial)
        scale = A.default_scale(d)
        a = A.tree_attention_flat(t, tree.offsets(), scale, row_block=3)
        b = A.tree_attention_direct(t, tree.offsets(), scale, row_block=2)
        for k in a:
            np.testing.assert_allclose(a[k], b[k], rtol=0, atol=1e-12, err_msg=k)


def test_prompt_gradient_is_sum_over_pairs():
    """Eq. 2: the tree's prompt K/V gradient equals the sum of the per-pair prompt
    gradients, however the prompt's own upstream gradient is split over the pairs."""
    tree = W.Tree([6], [[2, 5, 3]])
    hq, hkv, d = 2, 2, 4
    t = rand_inputs(tree, hq, hkv, d, seed=8)
    scale = A.default_scale(d)
    offs = tree.offsets()
    first = A.tree_attention_flat(t, offs, scale, prompt_do_split="first")
    even = A.tree_attention_flat(t, offs, scale, prompt_do_split="even")
    for k in ("dq_p", "dk_p", "dv_p"):
        np.testing.assert_allclose(first[k], even[k], rtol=0, atol=1e-12)
    # Explicit sum: run each pair alone as a causal sequence and add prompt rows.
    lp = 6
    acc = {k: np.zeros_like(t[k.replace("d", "", 1)]) for k in ("dq_p", "dk_p", "dv_p")}
    r0 = 0
    for pi, li in enumerate(tree.branch_lens[0]):
        seq = {x: np.concatenate([t[x + "_p"], t[x + "_r"][r0:r0 + li]]) for x in ("q", "k", "v")}
        do = np.concatenate([t["do_p"] if pi == 0 else 0 * t["do_p"], t["do_r"][r0:r0 + li]])
        res = A.causal_attention(seq["q"], seq["k"], seq["v"], scale, do=do)
        for x in ("q", "k", "v"):
            acc["d" + x + "_p"] += res["d" + x][:lp]
        r0 += li
    for k in acc:
        np.testing.assert_allclose(first[k], acc[k], rtol=0, atol=1e-12)


# ------------------------------------------------------------------------------
# Special cases that reduce to a textbook routine (SDPA causal)
# ------------------------------------------------------------------------------
def sdpa_causal(q, k, v, do, scale):
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    r = q.shape[1] // k.shape[1]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.transpose(0, 1), kt.repeat_interleave(r, 1).transpose(0, 1),
        vt.repeat_interleave(r, 1).transpose(0, 1), is_causal=True, scale=scale).transpose(0, 1)
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def test_single_branch_is_plain_causal():
    tree = W.Tree([9], [[6]])
    hq, hkv, d = 4, 1, 6
    t = rand_inputs(tree, hq, hkv, d, seed=11)
    scale = A.default_scale(d)
    out = A.tree_attention_direct(t, tree.offsets(), scale)
    cat = {x: np.concatenate([t[x + "_p"], t[x + "_r"]]) for x in ("q", "k", "v", "do")}
    o, dq, dk, dv = sdpa_causal(cat["q"], cat["k"], cat["v"], cat["do"], scale)
    np.testing.assert_allclose(np.concatenate([out["o_p"], out["o_r"]]), o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(np.concatenate([out["dq_p"], out["dq_r"]]), dq, atol=1e-12, rtol=0)
    np.testing.assert_allclose(np.concatenate([out["dk_p"], out["dk_r"]]), dk, atol=1e-12, rtol=0)
    np.testing.assert_allclose(np.concatenate([out["dv_p"], out["dv_r"]]), dv, atol=1e-12, rtol=0)


def test_empty_prompt_is_per_branch_causal_and_no_branches_is_prefill():
    d, scale = 4, 0.5
    tree = W.Tree([0], [[4, 3]])
    t = rand_inputs(tree, 2, 2, d, seed=12)
    out = A.tree_attention_direct(t, tree.offsets(), scale)
    for (a, b) in ((0, 4), (4, 7)):
        o, dq, dk, dv = sdpa_causal(t["q_r"][a:b], t["k_r"][a:b], t["v_r"][a:b], t["do_r"][a:b], scale)
        np.testing.assert_allclose(out["o_r"][a:b], o, atol=1e-12, rtol=0)
        np.testing.assert_allclose(out["dk_r"][a:b], dk, atol=1e-12, rtol=0)
    tree = W.Tree([7], [[]])
    t = rand_inputs(tree, 2, 1, d, seed=13)
    out = A.tree_attention_direct(t, tree.offsets(), scale)
    o, dq, dk, dv = sdpa_causal(t["q_p"], t["k_p"], t["v_p"], t["do_p"], scale)
    np.testing.assert_allclose(out["o_p"], o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(out["dq_p"], dq, atol=1e-12, rtol=0)
    np.testing.assert_allclose(out["dv_p"], dv, atol=1e-12, rtol=0)


# ------------------------------------------------------------------------------
# Per-row form (used for sampled rows of full-size workloads)
# ------------------------------------------------------------------------------
def test_rows_forward_backward_matches_full_oracle():
    tree = W.Tree([6, 4], [[3, 5], [2, 2, 2]])
    hq, hkv, d = 4, 2, 4
    t = rand_inputs(tree, hq, hkv, d, seed=14)
    scale = A.default_scale(d)
    offs = tree.offsets()
    full = A.tree_attention_direct(t, offs, scale)
    for kind, n in (("p", tree.total_prompt), ("r", tree.total_resp)):
        for row in range(n):
            (pa, pb), (ra, rb) = A.row_key_set(kind, row, offs)
            kk = np.concatenate([t["k_p"][pa:pb], t["k_r"][ra:rb]])
            vv = np.concatenate([t["v_p"][pa:pb], t["v_r"][ra:rb]])
            o, lse, dq = A.rows_forward_backward(t["q_" + kind][row:row + 1], kk, vv, scale,
                                                 t["do_" + kind][row:row + 1])
            np.testing.assert_allclose(o[0], full["o_" + kind][row], atol=1e-13, rtol=0)
            np.testing.assert_allclose(lse[:, 0], full["lse_" + kind][:, row], atol=1e-13, rtol=0)
            np.testing.assert_allclose(dq[0], full["dq_" + kind][row], atol=1e-13, rtol=0)


# ------------------------------------------------------------------------------
# Gradient identities (used at full size) hold on the oracle, and catch a mistake
# ------------------------------------------------------------------------------
def _identities(tree, hq, hkv, t, out):
    f = lambda k: out[k]
    return INV.gradient_identities(tree.offsets(), hq, hkv, t["q_p"], t["k_p"], t["q_r"], t["k_r"],
                                   t["do_p"], t["do_r"], f("dq_p"), f("dk_p"), f("dv_p"),
                                   f("dq_r"), f("dk_r"), f("dv_r"))


def _identity_errors(ids):
    e1 = max(np.max(np.abs(x["sum_dv"] - x["sum_do"])) / x["dv_scale"] for x in ids)
    e2 = max(np.max(np.abs(x["sum_dk"])) / x["dk_scale"] for x in ids)
    e3 = max(abs(x["qdq"] - x["kdk"]) / x["ip_scale"] for x in ids)
    return e1, e2, e3


def test_gradient_identities_hold_and_detect_a_dropped_term(monkeypatch):
    tree = W.Tree([5, 3], [[4, 2], [6]])
    hq, hkv, d = 4, 2, 6
    t = rand_inputs(tree, hq, hkv, d, seed=15)
    scale = A.default_scale(d)
    out = A.tree_attention_direct(t, tree.offsets(), scale)
    assert max(_identity_errors(_identities(tree, hq, hkv, t, out))) < 1e-12
    # Plant a mistake in a copy of the oracle's backward (drop Delta): (ii) must fail.
    orig = A.masked_attention_bwd

    def wrong_bwd(q, k, v, mask, sc, o, do):
        return orig(q, k, v, mask, sc, np.zeros_like(o), do)

    monkeypatch.setattr(A, "masked_attention_bwd", wrong_bwd)
    bad = A.tree_attention_direct(t, tree.offsets(), scale)
    assert _identity_errors(_identities(tree, hq, hkv, t, bad))[1] > 1e-3


def test_gqa_equals_mha_with_repeated_kv():
    tree = W.Tree([4], [[3, 2]])
    hq, hkv, d = 6, 2, 4
    t = rand_inputs(tree, hq, hkv, d, seed=16)
    scale = A.default_scale(d)
    gqa = A.tree_attention_direct(t, tree.offsets(), scale)
    tm = dict(t)
    for x in ("k_p", "v_p", "k_r", "v_r"):
        tm[x] = np.repeat(t[x], hq // hkv, axis=1)
    mha = A.tree_attention_direct(tm, tree.offsets(), scale)
    for k in ("o_p", "o_r", "dq_p", "dq_r"):
        np.testing.assert_allclose(gqa[k], mha[k], atol=1e-13, rtol=0)
    for k in ("dk_p", "dv_p", "dk_r", "dv_r"):
        summed = mha[k].reshape(mha[k].shape[0], hkv, hq // hkv, d).sum(2)
        np.testing.assert_allclose(gqa[k], summed, atol=1e-13, rtol=0)


def test_lse_merge_backward_matches_finite_differences():
    """The merge's backward against central differences of the merge itself (fp64), for
    a loss L = <g, O> + <h, lse> with random g, h."""
    rng = np.random.default_rng(31)
    n, d = 6, 5
    oa, ob = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    la, lb = rng.standard_normal(n) * 2, rng.standard_normal(n) * 2
    g, h = rng.standard_normal((n, d)), rng.standard_normal(n)

    def loss(oa_, la_, ob_, lb_):
        o, l = A.lse_merge(oa_, la_, ob_, lb_)
        return float(np.sum(g * o) + np.sum(h * l))

    got = A.lse_merge_backward(oa, la, ob, lb, g, h)
    eps = 1e-6
    for idx, base in enumerate((oa, la, ob, lb)):
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            args_p = [x.copy() for x in (oa, la, ob, lb)]
            args_m = [x.copy() for x in (oa, la, ob, lb)]
            args_p[idx][i] += eps
            args_m[idx][i] -= eps
            num[i] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(got[idx], num, rtol=1e-6, atol=1e-8)


def test_lse_merge_backward_special_cases():
    """An empty partner passes the gradient through; two empty inputs get zeros; equal
    inputs split d_o in halves."""
    rng = np.random.default_rng(32)
    o, do = rng.standard_normal((3, 4)), rng.standard_normal((3, 4))
    l, dl = rng.standard_normal(3), rng.standard_normal(3)
    ninf, z = np.full(3, -np.inf), np.zeros((3, 4))
    doa, dla, dob, dlb = A.lse_merge_backward(o, l, z, ninf, do, dl)
    np.testing.assert_allclose(doa, do, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dla, dl, rtol=0, atol=1e-15)
    assert np.all(dob == 0) and np.all(dlb == 0)
    r = A.lse_merge_backward(z, ninf, z, ninf, do, dl)
    assert all(np.all(x == 0) for x in r)
    doa, dla, dob, dlb = A.lse_merge_backward(o, l, o, l, do, dl)
    np.testing.assert_allclose(doa, do / 2, rtol=1e-15)
    np.testing.assert_allclose(dla, dl / 2, rtol=1e-15)  # <do, oa - ob> = 0
