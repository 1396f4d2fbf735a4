"""The library's host schedule builder against the reference builder on random ragged
trees (AugTree paper, Sec. 3.4: replay units with tile-count weights, largest-first
order), bit for bit, for all five work queues and both kernel families; and the
fused backward queue's brute-force coverage on random small trees.  CPU only."""
import numpy as np
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import schedule as S
from tests.test_schedule_oracle import valid_pairs


@pytest.mark.parametrize("seed", range(40))
def test_random_trees_bit_exact(augtree_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    tree = W.random_tree(rng, n_groups=int(rng.integers(1, 5)), max_prompt=700, max_branches=9, max_resp=600)
    r = int(rng.choice([1, 2, 4, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    hq = r * hkv
    sms = int(rng.choice([1, 3, 16, 152, 100000]))
    for kernel, dtype in ((at.KERNEL_TC, at.BF16), (at.KERNEL_SIMT, at.FP32)):
        cfg = at.make_config(hq, hkv, 128, dtype, 0.0, sms, kernel)
        for op in range(5):
            bm, bn = at.tile_sizes(cfg, op)
            got = at.schedule_build(tree.offsets(), cfg, op)
            want = S.build(tree.offsets(), hq, hkv, op, bm, bn, sms, split_replay_fwd=kernel == at.KERNEL_TC)
            assert got.shape == want.shape and np.array_equal(got, want), (seed, kernel, op)


@pytest.mark.parametrize("seed", range(30))
def test_random_fused_queue_covers_every_pair_once(seed):
    rng = np.random.default_rng(2000 + seed)
    tree = W.random_tree(rng, n_groups=int(rng.integers(1, 4)), max_prompt=40, max_branches=5, max_resp=30)
    bm, bn = [(4, 4), (8, 4), (4, 8), (16, 16)][seed % 4]
    hq, hkv = (4, 2) if seed % 2 else (2, 2)
    sms = [1, 2, 64][seed % 3]
    groups = valid_pairs(tree)
    r = hq // hkv
    covered = set()
    for it in S.build(tree.offsets(), hq, hkv, S.OP_TREE_BWD, bm, bn, sms):
        kind, g, tile, hk, split, cost, a, b = map(int, it)
        grp = groups[g]
        if kind == S.TREE_PROMPT_KV:
            k0, klen = grp["p0"], grp["lp"]
            ranges = [(grp["r0"], grp["r0"] + grp["lr"], a, b, grp["rp"], "rp")]
            if split == 0:
                ranges.append((grp["p0"], grp["p0"] + grp["lp"], (tile * bn) // bm, -(-grp["lp"] // bm),
                               grp["pp"], "pp"))
        else:
            assert kind == S.RESP_KV
            k0, klen = grp["r0"], grp["lr"]
            ranges = [(grp["r0"], grp["r0"] + grp["lr"], a, b, grp["rr"], "rr")]
        keys = range(k0 + tile * bn, min(k0 + (tile + 1) * bn, k0 + klen))
        for rows0, rows1, qa, qb, pairs, side in ranges:
            for qt in range(qa, qb):
                for row in range(rows0 + qt * bm, min(rows0 + (qt + 1) * bm, rows1)):
                    for key in keys:
                        if (row, key) in pairs:
                            for h in range(hk * r, (hk + 1) * r):
                                assert (side, row, key, h) not in covered
                                covered.add((side, row, key, h))
    want = {(side, row, key, h) for grp in groups for side in ("pp", "rp", "rr")
            for (row, key) in grp[side] for h in range(hq)}
    assert covered == want
