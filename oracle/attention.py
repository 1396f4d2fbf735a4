"""fp64 reference of exact shared-prompt tree attention (forward and backward).

TEST INFRASTRUCTURE ONLY: imported by tests, the package smoke check and the CPU
baseline of the benchmark, never by the library.

Source: AugTree paper, "Splitting Prompt Prefill from Response Replay for
Context-Parallel Long-Context LLM Post-Training".
  * Sec. 2.2: O = softmax(Q K^T / sqrt(D_h) + M) V for one head.
  * Sec. 2.1 (replay tree, asymmetric KV dependency): the tree is flattened by
    existing stacks into G sequences (P, R_i); each response token attends to the
    full prompt and its own prefix, never to siblings; the prompt never attends to
    responses.
  * Sec. 3.2, Eq. 1: KV(R_{i,t}) = KV_P  U  KV(R_{i,<t}).  Reading: standard causal
    masking, a query at position t also sees its own key (the b=0 fallback of
    Sec. 3.4 runs each (P, R_i) pair with the standard causal mask, and the tree
    result must equal it).
  * Sec. 3.2, Eq. 2: grad KV_P = sum_{i=1..G} grad_{KV_P} L_i (prompt gradients summed
    over all branches, then propagated through the prefill graph).
  * Sec. 3.3: partial online-softmax states S = (m, l, O_acc) merge associatively;
    here they are carried as (O, lse) with lse = m + log l and O = O_acc / l.  The
    merge's backward (lse_merge_backward) is its chain rule, written out.

Layout (token-major, "THD"): q [L, Hq, D], k/v [L, Hkv, D]; query head h uses KV head
floor(h / r), r = Hq / Hkv.  lse is [Hq, L] in natural log.

Gradients are those of the scalar sum(dO * O) for a given upstream dO: with
P = softmax(S),  dV = P^T dO,  dP = dO V^T,  Delta = rowsum(dO * O),
dS = P * (dP - Delta),  dQ = s dS K,  dK = s dS^T Q  (summed over the r query
heads of a KV head).

All arithmetic is float64.  Row blocking only bounds memory: every row's softmax is
computed over its full key set at once; there are no partial or online states in
the forward or backward (only the explicit merge function uses them).
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

NEG_INF = -np.inf


def _gqa_ratio(hq: int, hkv: int) -> int:
    if hkv <= 0 or hq % hkv != 0:
        raise ValueError("Hq must be a positive multiple of Hkv")
    return hq // hkv


# ----------------------------------------------------------------------------------
# Masked attention over explicit key sets
# ----------------------------------------------------------------------------------
def masked_attention_fwd(q, k, v, mask, scale):
    """One head: q [M, D], k/v [N, D], mask [M, N] bool (True = valid key).
    Returns O [M, D] and lse [M].  A row with no valid key gets O = 0, lse = -inf
    (the identity of the merge)."""
    s = scale * (q @ k.T)
    s = np.where(mask, s, NEG_INF)
    m = s.max(axis=1, initial=NEG_INF)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m_safe[:, None])
    p = np.where(mask, p, 0.0)
    l = p.sum(axis=1)
    l_safe = np.where(l > 0, l, 1.0)
    o = (p / l_safe[:, None]) @ v
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m_safe + np.log(l_safe), NEG_INF)
    return o, lse


def masked_attention_bwd(q, k, v, mask, scale, o, do):
    """One head, gradients of sum(do * o) where o = masked_attention_fwd(...).
    Returns dq [M, D], dk [N, D], dv [N, D]."""
    s = scale * (q @ k.T)
    s = np.where(mask, s, NEG_INF)
    m = s.max(axis=1, initial=NEG_INF)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.where(mask, np.exp(s - m_safe[:, None]), 0.0)
    l = p.sum(axis=1)
    p = p / np.where(l > 0, l, 1.0)[:, None]
    dv = p.T @ do
    dp = do @ v.T
    delta = np.sum(do * o, axis=1)
    ds = p * (dp - delta[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


# ----------------------------------------------------------------------------------
# Causal attention on one linear sequence (used per flattened pair)
# ----------------------------------------------------------------------------------
def causal_attention(q, k, v, scale, do=None, row_block: int = 2048):
    """Standard causal attention (key j visible to query i iff j <= i) on one
    sequence, all heads.  q [L, Hq, D], k/v [L, Hkv, D].  Returns dict with o, lse
    and, when do is given, dq, dk, dv.  Rows are processed in blocks of row_block
    queries; each block sees keys [0, block_end)."""
    L, hq, d = q.shape
    hkv = k.shape[1]
    r = _gqa_ratio(hq, hkv)
    o = np.zeros_like(q)
    lse = np.full((hq, L), NEG_INF)
    want = do is not None
    if want:
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
    for h in range(hq):
        kv = h // r
        for a in range(0, L, row_block):
            b = min(L, a + row_block)
            rows = np.arange(a, b)[:, None]
            cols = np.arange(0, b)[None, :]
            mask = cols <= rows
            qb, kb, vb = q[a:b, h], k[:b, kv], v[:b, kv]
            ob, lb = masked_attention_fwd(qb, kb, vb, mask, scale)
            o[a:b, h] = ob
            lse[h, a:b] = lb
            if want:
                gq, gk, gv = masked_attention_bwd(qb, kb, vb, mask, scale, ob, do[a:b, h])
                dq[a:b, h] = gq
                dk[:b, kv] += gk
                dv[:b, kv] += gv
    out = {"o": o, "lse": lse}
    if want:
        out.update(dq=dq, dk=dk, dv=dv)
    return out


# ----------------------------------------------------------------------------------
# Flattened per-pair oracle (the plain definition)
# ----------------------------------------------------------------------------------
def _group_views(prompt_off, branch_begin, resp_off, g):
    p0, p1 = int(prompt_off[g]), int(prompt_off[g + 1])
    b0, b1 = int(branch_begin[g]), int(branch_begin[g + 1])
    branches = [(int(resp_off[b]), int(resp_off[b + 1])) for b in range(b0, b1)]
    return p0, p1, branches


def tree_attention_flat(t: Dict[str, np.ndarray], offsets, scale: float,
                        grad: bool = True, row_block: int = 2048,
                        check_prompt_consistency: bool = True,
                        prompt_do_split: str = "first") -> Dict[str, np.ndarray]:
    """Flatten every prompt-response pair (P_g, R_i) into one linear sequence and run
    causal attention on it (AugTree Sec. 2.1 flattening, Sec. 3.4 b=0 semantics).

    t: dict of float64 arrays q_p, k_p, v_p [sum L_P, H, D], q_r, k_r, v_r
       [sum L_i, H, D] and, when grad, do_p, do_r.
    offsets: (prompt_off, branch_begin, resp_off).

    Tree outputs: O_R / lse_R are the response rows of their own pair; O_P / lse_P
    are the prompt rows (identical in every pair; checked).  Backward: the prompt's
    upstream gradient dO_P enters once, all of it in the group's first pair (zero in
    the others) - or, with prompt_do_split="even", a 1/G share in each pair; by
    linearity both give the same result.  dQ_P, dK_P, dV_P are the sums over pairs of
    the per-pair prompt-row gradients (Eq. 2).  A group without branches is run as
    its prompt alone."""
    prompt_off, branch_begin, resp_off = offsets
    q_p, k_p, v_p = t["q_p"], t["k_p"], t["v_p"]
    q_r, k_r, v_r = t["q_r"], t["k_r"], t["v_r"]
    out = {
        "o_p": np.zeros_like(q_p), "lse_p": np.full((q_p.shape[1], q_p.shape[0]), NEG_INF),
        "o_r": np.zeros_like(q_r), "lse_r": np.full((q_r.shape[1], q_r.shape[0]), NEG_INF),
    }
    if grad:
        for name, ref in (("dq_p", q_p), ("dk_p", k_p), ("dv_p", v_p),
                          ("dq_r", q_r), ("dk_r", k_r), ("dv_r", v_r)):
            out[name] = np.zeros_like(ref)
    n_groups = len(prompt_off) - 1
    for g in range(n_groups):
        p0, p1, branches = _group_views(prompt_off, branch_begin, resp_off, g)
        lp = p1 - p0
        pairs = branches if branches else [(0, 0)]
        for pi, (r0, r1) in enumerate(pairs):
            q = np.concatenate([q_p[p0:p1], q_r[r0:r1]], axis=0)
            k = np.concatenate([k_p[p0:p1], k_r[r0:r1]], axis=0)
            v = np.concatenate([v_p[p0:p1], v_r[r0:r1]], axis=0)
            do = None
            if grad:
                if prompt_do_split == "even":
                    do_prompt = t["do_p"][p0:p1] / len(pairs)
                elif pi == 0:
                    do_prompt = t["do_p"][p0:p1]
                else:
                    do_prompt = np.zeros_like(t["do_p"][p0:p1])
                do = np.concatenate([do_prompt, t["do_r"][r0:r1]], axis=0)
            res = causal_attention(q, k, v, scale, do=do, row_block=row_block)
            if pi == 0:
                out["o_p"][p0:p1] = res["o"][:lp]
                out["lse_p"][:, p0:p1] = res["lse"][:, :lp]
            elif check_prompt_consistency:
                # Same rows, same keys: equal up to the summation order of the matmul.
                assert np.allclose(out["o_p"][p0:p1], res["o"][:lp], rtol=0, atol=1e-12)
                assert np.allclose(out["lse_p"][:, p0:p1], res["lse"][:, :lp], rtol=0, atol=1e-12)
            out["o_r"][r0:r1] = res["o"][lp:]
            out["lse_r"][:, r0:r1] = res["lse"][:, lp:]
            if grad:
                out["dq_p"][p0:p1] += res["dq"][:lp]
                out["dk_p"][p0:p1] += res["dk"][:lp]
                out["dv_p"][p0:p1] += res["dv"][:lp]
                out["dq_r"][r0:r1] = res["dq"][lp:]
                out["dk_r"][r0:r1] = res["dk"][lp:]
                out["dv_r"][r0:r1] = res["dv"][lp:]
    return out


# ----------------------------------------------------------------------------------
# Tree-direct oracle: the valid KV context of Eq. 1, prompt evaluated once
# ----------------------------------------------------------------------------------
def tree_attention_direct(t: Dict[str, np.ndarray], offsets, scale: float,
                          grad: bool = True, row_block: int = 2048) -> Dict[str, np.ndarray]:
    """Same result as tree_attention_flat, computed on the tree (Sec. 3.2):
      prompt rows:   keys = prompt keys j <= i (causal prefill);
      response rows: keys = all prompt keys of the group  U  own-branch keys j <= i
                     (Eq. 1; no sibling keys).
    Backward: every response row's gradient w.r.t. the prompt keys is summed into
    dK_P / dV_P (Eq. 2), alongside the prompt rows' own causal gradient."""
    prompt_off, branch_begin, resp_off = offsets
    q_p, k_p, v_p = t["q_p"], t["k_p"], t["v_p"]
    q_r, k_r, v_r = t["q_r"], t["k_r"], t["v_r"]
    out = {
        "o_p": np.zeros_like(q_p), "lse_p": np.full((q_p.shape[1], q_p.shape[0]), NEG_INF),
        "o_r": np.zeros_like(q_r), "lse_r": np.full((q_r.shape[1], q_r.shape[0]), NEG_INF),
    }
    if grad:
        for name, ref in (("dq_p", q_p), ("dk_p", k_p), ("dv_p", v_p),
                          ("dq_r", q_r), ("dk_r", k_r), ("dv_r", v_r)):
            out[name] = np.zeros_like(ref)
    n_groups = len(prompt_off) - 1
    for g in range(n_groups):
        p0, p1, branches = _group_views(prompt_off, branch_begin, resp_off, g)
        # Prompt prefill: causal self-attention over the prompt, computed once.
        if p1 > p0:
            res = causal_attention(q_p[p0:p1], k_p[p0:p1], v_p[p0:p1], scale,
                                   do=t["do_p"][p0:p1] if grad else None, row_block=row_block)
            out["o_p"][p0:p1] = res["o"]
            out["lse_p"][:, p0:p1] = res["lse"]
            if grad:
                out["dq_p"][p0:p1] += res["dq"]
                out["dk_p"][p0:p1] += res["dk"]
                out["dv_p"][p0:p1] += res["dv"]
        # Response replay: prompt keys (dense) + own-branch keys (causal).
        for (r0, r1) in branches:
            _replay_branch(t, out, p0, p1, r0, r1, scale, grad, row_block)
    return out


def _replay_branch(t, out, p0, p1, r0, r1, scale, grad, row_block):
    q_r, k_r, v_r, k_p, v_p = t["q_r"], t["k_r"], t["v_r"], t["k_p"], t["v_p"]
    hq, hkv = q_r.shape[1], k_r.shape[1]
    r = _gqa_ratio(hq, hkv)
    lp = p1 - p0
    li = r1 - r0
    if li == 0:
        return
    for h in range(hq):
        kv = h // r
        for a in range(0, li, row_block):
            b = min(li, a + row_block)
            keys_k = np.concatenate([k_p[p0:p1, kv], k_r[r0:r0 + b, kv]], axis=0)
            keys_v = np.concatenate([v_p[p0:p1, kv], v_r[r0:r0 + b, kv]], axis=0)
            rows = np.arange(a, b)[:, None]
            own = np.arange(0, b)[None, :]
            mask = np.concatenate([np.ones((b - a, lp), dtype=bool), own <= rows], axis=1)
            qb = q_r[r0 + a:r0 + b, h]
            ob, lb = masked_attention_fwd(qb, keys_k, keys_v, mask, scale)
            out["o_r"][r0 + a:r0 + b, h] = ob
            out["lse_r"][h, r0 + a:r0 + b] = lb
            if grad:
                gq, gk, gv = masked_attention_bwd(qb, keys_k, keys_v, mask, scale, ob,
                                                  t["do_r"][r0 + a:r0 + b, h])
                out["dq_r"][r0 + a:r0 + b, h] = gq
                out["dk_p"][p0:p1, kv] += gk[:lp]
                out["dv_p"][p0:p1, kv] += gv[:lp]
                out["dk_r"][r0:r0 + b, kv] += gk[lp:]
                out["dv_r"][r0:r0 + b, kv] += gv[lp:]


# ----------------------------------------------------------------------------------
# Per-row form (sampled rows of full-size workloads)
# ----------------------------------------------------------------------------------
def row_key_set(kind: str, row: int, offsets):
    """Valid KV context of one query row (Eq. 1 and the causal prefill).
    kind 'p' (prompt row, global prompt index) or 'r' (response row, global response
    index).  Returns ((prompt_key_lo, prompt_key_hi), (resp_key_lo, resp_key_hi)),
    half-open ranges of global key indices."""
    prompt_off, branch_begin, resp_off = offsets
    if kind == "p":
        g = int(np.searchsorted(prompt_off, row, side="right") - 1)
        return (int(prompt_off[g]), row + 1), (0, 0)
    b = int(np.searchsorted(resp_off, row, side="right") - 1)
    g = int(np.searchsorted(branch_begin, b, side="right") - 1)
    return (int(prompt_off[g]), int(prompt_off[g + 1])), (int(resp_off[b]), row + 1)


def rows_forward_backward(q_rows, keys_k, keys_v, scale, do_rows=None):
    """Exact attention of a few query rows over an explicit, fully valid key set.
    q_rows [M, Hq, D]; keys_k / keys_v [N, Hkv, D] (the same key set for every row).
    Returns o [M, Hq, D], lse [Hq, M] and, when do_rows is given, dq [M, Hq, D].
    Each row's dQ needs only its own softmax row and Delta_i = rowsum(dO_i * O_i)."""
    m, hq, d = q_rows.shape
    hkv = keys_k.shape[1]
    r = _gqa_ratio(hq, hkv)
    o = np.zeros_like(q_rows)
    lse = np.zeros((hq, m))
    dq = np.zeros_like(q_rows) if do_rows is not None else None
    mask = np.ones((m, keys_k.shape[0]), dtype=bool)
    for h in range(hq):
        kv = h // r
        ob, lb = masked_attention_fwd(q_rows[:, h], keys_k[:, kv], keys_v[:, kv], mask, scale)
        o[:, h] = ob
        lse[h] = lb
        if do_rows is not None:
            gq, _, _ = masked_attention_bwd(q_rows[:, h], keys_k[:, kv], keys_v[:, kv], mask,
                                            scale, ob, do_rows[:, h])
            dq[:, h] = gq
    return o, lse, dq


# ----------------------------------------------------------------------------------
# Partial softmax states and their merge (Sec. 3.3)
# ----------------------------------------------------------------------------------
def partial_state(q, k, v, scale):
    """Partial state of one head's queries q [M, D] over a key subset k/v [N, D], as
    (O, lse): O = O_acc / l, lse = m + log l.  An empty subset gives (0, -inf)."""
    mask = np.ones((q.shape[0], k.shape[0]), dtype=bool)
    return masked_attention_fwd(q, k, v, mask, scale)


def lse_merge(o_a, lse_a, o_b, lse_b):
    """State merge (+) of two partial states in (O, lse) form:
        lse = log(e^lse_a + e^lse_b),  O = e^(lse_a - lse) O_a + e^(lse_b - lse) O_b.
    o_* [..., D], lse_* [...].  (0, -inf) is the identity; two empty states give
    (0, -inf)."""
    lse = np.logaddexp(lse_a, lse_b)
    fin = np.isfinite(lse)
    lse_safe = np.where(fin, lse, 0.0)
    wa = np.where(fin & np.isfinite(lse_a), np.exp(np.where(np.isfinite(lse_a), lse_a, 0.0) - lse_safe), 0.0)
    wb = np.where(fin & np.isfinite(lse_b), np.exp(np.where(np.isfinite(lse_b), lse_b, 0.0) - lse_safe), 0.0)
    o = wa[..., None] * o_a + wb[..., None] * o_b
    return o, lse


def lse_merge_backward(o_a, lse_a, o_b, lse_b, d_o, d_lse=None):
    """Gradients of the state merge (+) (Sec. 3.3) with respect to its two inputs, given
    the upstream gradient d_o of the merged O and, optionally, d_lse of the merged lse.

    With w_a = e^(lse_a - lse), w_b = e^(lse_b - lse) (so w_a + w_b = 1):
        O = w_a O_a + w_b O_b,   lse = log(e^lse_a + e^lse_b),
        dw_a/dlse_a = w_a w_b,   dw_b/dlse_a = -w_a w_b,   dlse/dlse_a = w_a,
    hence
        dO_a = w_a d_o,   dO_b = w_b d_o,
        dlse_a = w_a w_b <d_o, O_a - O_b> + w_a d_lse,
        dlse_b = w_a w_b <d_o, O_b - O_a> + w_b d_lse.
    An empty input (lse = -inf) has weight 0 and receives zero gradients; the other
    input then passes d_o and d_lse through unchanged."""
    if d_lse is None:
        d_lse = np.zeros(np.shape(lse_a))
    lse = np.logaddexp(lse_a, lse_b)
    fin = np.isfinite(lse)
    lse_safe = np.where(fin, lse, 0.0)
    wa = np.where(fin & np.isfinite(lse_a), np.exp(np.where(np.isfinite(lse_a), lse_a, 0.0) - lse_safe), 0.0)
    wb = np.where(fin & np.isfinite(lse_b), np.exp(np.where(np.isfinite(lse_b), lse_b, 0.0) - lse_safe), 0.0)
    sa = np.sum(d_o * o_a, axis=-1)
    sb = np.sum(d_o * o_b, axis=-1)
    do_a = wa[..., None] * d_o
    do_b = wb[..., None] * d_o
    dl_a = wa * wb * (sa - sb) + wa * d_lse
    dl_b = wa * wb * (sb - sa) + wb * d_lse
    return do_a, dl_a, do_b, dl_b


def to_float64(t: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    return {k: np.asarray(v, dtype=np.float64) for k, v in t.items()}


def default_scale(d: int, scale: Optional[float] = None) -> float:
    """Softmax scale 1/sqrt(D_h) (Sec. 2.2) unless overridden."""
    return float(scale) if scale else 1.0 / np.sqrt(d)
