"""Exact identities of attention gradients, for checks at any size.

TEST INFRASTRUCTURE ONLY: imported by tests, never by the library.

For softmax attention with P = softmax(S), S = s Q K^T (any mask), and the gradient
of sum(dO * O) (AugTree paper, Sec. 2.2 attention; Sec. 3.2, Eq. 2 for the prompt
sums), per KV head and per group, summed over the query heads of that KV head:
  (i)   sum_j dV_j = sum_i dO_i                (every row of P sums to 1)
  (ii)  sum_j dK_j = 0                          (sum_j dS_ij = 0 for every row i)
  (iii) sum_i <dQ_i, q_i> = sum_j <dK_j, k_j>   (both equal s sum_ij dS_ij <q_i, k_j>)
Keys j run over the group's prompt and response keys, rows i over its prompt and
response rows.  Each check returns (lhs, rhs, scale) per (group, KV head) so that a
caller can bound |lhs - rhs| / scale.
"""
from __future__ import annotations

import numpy as np


def _group_rows(offsets, g):
    prompt_off, branch_begin, resp_off = offsets
    p0, p1 = int(prompt_off[g]), int(prompt_off[g + 1])
    r0, r1 = int(resp_off[int(branch_begin[g])]), int(resp_off[int(branch_begin[g + 1])])
    return p0, p1, r0, r1


def gradient_identities(offsets, hq, hkv, q_p, k_p, q_r, k_r, do_p, do_r,
                        dq_p, dk_p, dv_p, dq_r, dk_r, dv_r):
    """All arrays float64 (converted by the caller).  Returns a list of dicts, one per
    (group, kv head), with the three identities' two sides and a magnitude scale."""
    r = hq // hkv
    out = []
    n_groups = len(offsets[0]) - 1
    for g in range(n_groups):
        p0, p1, r0, r1 = _group_rows(offsets, g)
        for kv in range(hkv):
            hs = slice(kv * r, (kv + 1) * r)
            sum_dv = dv_p[p0:p1, kv].sum(0) + dv_r[r0:r1, kv].sum(0)
            sum_do = do_p[p0:p1, hs].sum((0, 1)) + do_r[r0:r1, hs].sum((0, 1))
            sum_dk = dk_p[p0:p1, kv].sum(0) + dk_r[r0:r1, kv].sum(0)
            qdq = float(np.sum(dq_p[p0:p1, hs] * q_p[p0:p1, hs]) + np.sum(dq_r[r0:r1, hs] * q_r[r0:r1, hs]))
            kdk = float(np.sum(dk_p[p0:p1, kv] * k_p[p0:p1, kv]) + np.sum(dk_r[r0:r1, kv] * k_r[r0:r1, kv]))
            dk_scale = float(np.sqrt(np.sum(dk_p[p0:p1, kv] ** 2) + np.sum(dk_r[r0:r1, kv] ** 2)) + 1e-30)
            dv_scale = float(np.sqrt(np.sum(dv_p[p0:p1, kv] ** 2) + np.sum(dv_r[r0:r1, kv] ** 2)) + 1e-30)
            ip_scale = float(np.sqrt(np.sum(dq_p[p0:p1, hs] ** 2) + np.sum(dq_r[r0:r1, hs] ** 2))
                             * np.sqrt(np.sum(q_p[p0:p1, hs] ** 2) + np.sum(q_r[r0:r1, hs] ** 2)) + 1e-30)
            out.append(dict(group=g, kv=kv, sum_dv=sum_dv, sum_do=sum_do, dv_scale=dv_scale,
                            sum_dk=sum_dk, dk_scale=dk_scale, qdq=qdq, kdk=kdk, ip_scale=ip_scale))
    return out
