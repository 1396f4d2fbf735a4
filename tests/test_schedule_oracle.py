"""Pins of the reference work-queue builder (CPU only).

The queues are the on-chip form of the paper's replay units and largest-first greedy
balancing (AugTree, Sec. 3.4): every valid Q-KV tile interaction implied by Eq. 1
(Sec. 3.2) must be evaluated exactly once, no item may carry an empty tile, and items
come in order of decreasing weight.  These properties are checked here by brute force
over the (query row, key) pairs of small ragged trees, independently of the
builder's own loops.
"""
import numpy as np
import pytest

from oracle import schedule as S
import workloads as W


def valid_pairs(tree):
    """Brute force: per group, the sets of valid (query, key) pairs, in global row
    indices, split by (query side, key side): pp (prompt->prompt), rp (response ->
    prompt), rr (response -> response)."""
    out = []
    p_base = r_base = 0
    for lp, bl in zip(tree.prompt_lens, tree.branch_lens):
        pp = {(p_base + i, p_base + j) for i in range(lp) for j in range(i + 1)}
        rp, rr = set(), set()
        rb = r_base
        for li in bl:
            for t in range(li):
                rp |= {(rb + t, p_base + j) for j in range(lp)}
                rr |= {(rb + t, rb + j) for j in range(t + 1)}
            rb += li
        out.append(dict(pp=pp, rp=rp, rr=rr, p0=p_base, lp=lp, r0=r_base, lr=sum(bl)))
        p_base += lp
        r_base += sum(bl)
    return out


def key_side_stream(tree, bn, it, r=1):
    """The stream an item walks, from the tree alone: a forward item the K/V of (group,
    KV head = head // r, -1); a key-side item the Q/dO tiles of (group, KV head, -1) for
    prompt keys, (group, KV head, branch) for response keys (the branch holding the
    tile's first key, empty branches skipped)."""
    kind, g, tile = int(it[0]), int(it[1]), int(it[2])
    if kind in (S.PREFILL_Q, S.REPLAY_Q):
        return (g, int(it[3]) // r, -1)
    if kind != S.RESP_KV:
        return (g, int(it[3]), -1)
    key = tile * bn
    pos = 0
    for i, li in enumerate(tree.branch_lens[g]):
        if pos <= key < pos + li:
            return (g, int(it[3]), i)
        pos += li
    raise AssertionError("tile outside its group's branches")


def first_row_branch(tree, bm, it):
    """Replay forward item: the branch (index within its group) of its query tile's
    first row; -1 for every other item."""
    if int(it[0]) != S.REPLAY_Q:
        return -1
    g, row = int(it[1]), int(it[2]) * bm
    pos = 0
    for i, li in enumerate(tree.branch_lens[g]):
        if pos <= row < pos + li:
            return i
        pos += li
    raise AssertionError("query tile outside its group's branches")


def check_key_side_order(q, tree, bn, r=1, bm=None):
    """Every queue: the items of one stream are contiguous; streams come in order of
    decreasing total cost (ties by group, KV head, branch); within a stream, the replay
    forward items of one first-row branch are contiguous, those sub-streams come by
    decreasing total cost (ties by branch), and items within a sub-stream come largest
    first (ties by tile, kind, split, head)."""
    streams = [key_side_stream(tree, bn, it, r) for it in q]
    subs = [s_ + (first_row_branch(tree, bm if bm is not None else bn, it),) for s_, it in zip(streams, q)]
    total, sub_total = {}, {}
    for s_, sb, it in zip(streams, subs, q):
        total[s_] = total.get(s_, 0) + int(it[5])
        sub_total[sb] = sub_total.get(sb, 0) + int(it[5])
    for seq in (streams, subs):
        seen, prev = set(), None
        for s_ in seq:
            if s_ != prev:
                assert s_ not in seen, "a stream's items are split apart"
                seen.add(s_)
                prev = s_
    keys = [(-total[s_], s_, -sub_total[sb], sb[3], -int(it[5]), int(it[2]), int(it[0]), int(it[4]), int(it[3]))
            for s_, sb, it in zip(streams, subs, q)]
    assert keys == sorted(keys)


TREES = [
    W.Tree([5], [[3, 4]]),
    W.Tree([70, 33], [[1, 60, 25], [40]]),
    W.Tree([0, 41], [[30, 20], [0, 57]]),
    W.Tree([64, 2, 30], [[], [31], [1, 1, 1, 17]]),
    W.Tree([130], [[9] * 7 + [65]]),
]
TILES = [(4, 4), (8, 4), (4, 8), (16, 16), (8, 16)]


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("bm,bn", TILES)
@pytest.mark.parametrize("hq,hkv", [(4, 2), (2, 2)])
@pytest.mark.parametrize("split", [False, True])
def test_forward_queues_cover_valid_pairs_once(ti, bm, bn, hq, hkv, split):
    """Every valid (row, key) pair of every head exactly once; with the split-KV rule
    (1000 SMs, so that the short replay queues split into small chunks), split k of a
    tile walks the chunk [k C, k C + cost) of the tile's KV walk, C the cost of its
    split 0."""
    tree = TREES[ti]
    groups = valid_pairs(tree)
    offs = tree.offsets()
    sms = 1000 if split else 3
    for op, kind, side in ((S.OP_PREFILL_FWD, S.PREFILL_Q, "pp"), (S.OP_REPLAY_FWD, S.REPLAY_Q, None)):
        q = S.build(offs, hq, hkv, op, bm, bn, num_sms=sms, split_replay_fwd=split)
        check_key_side_order(q, tree, bn, hq // hkv, bm)
        chunk, nsplit = {}, {}
        for it in q:
            k, g, tile, h, sp, cost, a, b = map(int, it)
            if sp == 0:
                chunk[(g, tile, h)] = cost
            nsplit[(g, tile, h)] = max(nsplit.get((g, tile, h), 0), sp + 1)
        walked = {}
        covered = {}
        for it in q:
            k, g, tile, h, sp, cost, a, b = map(int, it)
            assert k == kind and (sp == 0 or (split and op == S.OP_REPLAY_FWD))
            walked[(g, tile, h)] = walked.get((g, tile, h), 0) + cost
            grp = groups[g]
            if op == S.OP_PREFILL_FWD:
                rows = range(grp["p0"] + tile * bm, min(grp["p0"] + (tile + 1) * bm, grp["p0"] + grp["lp"]))
                tiles = [("p", grp["p0"] + j * bn) for j in range(a)]
                assert b == 0 and cost == a
            else:
                rows = range(grp["r0"] + tile * bm, min(grp["r0"] + (tile + 1) * bm, grp["r0"] + grp["lr"]))
                first = rows[0]
                # own-branch keys start at the first row's branch start (brute force)
                bstart = min(y for (rr, y) in grp["rr"] if rr == first)
                tiles = [("p", grp["p0"] + j * bn) for j in range(a)] + \
                        [("r", bstart + j * bn) for j in range(b)]
                if nsplit[(g, tile, h)] == 1:
                    assert cost == a + b
                else:
                    c = chunk[(g, tile, h)]
                    assert nsplit[(g, tile, h)] == -(-(a + b) // c) and 0 < cost <= c
                    assert cost == min(c, a + b - sp * c)
                    tiles = tiles[sp * c: sp * c + cost]
            assert len(rows) > 0
            for (side_k, k0) in tiles:
                keys = range(k0, k0 + bn)
                hit = 0
                for row in rows:
                    for key in keys:
                        if op == S.OP_PREFILL_FWD:
                            ok = (row, key) in grp["pp"]
                        else:
                            ok = (row, key) in (grp["rp"] if side_k == "p" else grp["rr"])
                        if ok:
                            assert (side_k, row, key, h) not in covered, "pair covered twice"
                            covered[(side_k, row, key, h)] = 1
                            hit += 1
                assert hit > 0, "empty KV tile in an item"
        if op == S.OP_REPLAY_FWD:
            for (g, tile, h), n in walked.items():
                it = [x for x in q if x[1] == g and x[2] == tile and x[3] == h][0]
                assert n == int(it[6]) + int(it[7])  # the splits walk a + b tiles in all
        # every valid pair, every head
        for grp in groups:
            for h in range(hq):
                if op == S.OP_PREFILL_FWD:
                    for (row, key) in grp["pp"]:
                        assert ("p", row, key, h) in covered
                else:
                    for (row, key) in grp["rp"]:
                        assert ("p", row, key, h) in covered
                    for (row, key) in grp["rr"]:
                        assert ("r", row, key, h) in covered


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("bm,bn", TILES)
@pytest.mark.parametrize("hq,hkv,sms", [(4, 2, 1), (4, 2, 64), (2, 2, 2), (8, 1, 1)])
def test_backward_queues_cover_valid_pairs_once(ti, bm, bn, hq, hkv, sms):
    tree = TREES[ti]
    groups = valid_pairs(tree)
    offs = tree.offsets()
    r = hq // hkv
    for op in (S.OP_REPLAY_BWD, S.OP_PREFILL_BWD):
        q = S.build(offs, hq, hkv, op, bm, bn, num_sms=sms)
        check_key_side_order(q, tree, bn)
        covered = set()
        split_ranges = {}
        for it in q:
            kind, g, tile, hk, split, cost, a, b = map(int, it)
            grp = groups[g]
            assert cost == (b - a) * r and b > a
            if kind == S.PREFILL_KV:
                assert op == S.OP_PREFILL_BWD
                k0, rows0, rows1, pairs, side = grp["p0"], grp["p0"], grp["p0"] + grp["lp"], grp["pp"], "pp"
            elif kind == S.PROMPT_KV:
                assert op == S.OP_REPLAY_BWD
                k0, rows0, rows1, pairs, side = grp["p0"], grp["r0"], grp["r0"] + grp["lr"], grp["rp"], "rp"
                split_ranges.setdefault((g, tile, hk), []).append((split, a, b))
            else:
                assert kind == S.RESP_KV and op == S.OP_REPLAY_BWD and split == 0
                k0, rows0, rows1, pairs, side = grp["r0"], grp["r0"], grp["r0"] + grp["lr"], grp["rr"], "rr"
            keys = range(k0 + tile * bn, min(k0 + (tile + 1) * bn, k0 + (grp["lp"] if side != "rr" else grp["lr"])))
            assert len(keys) > 0
            for qt in range(a, b):
                rows = range(rows0 + qt * bm, min(rows0 + (qt + 1) * bm, rows1))
                hit = 0
                for row in rows:
                    for key in keys:
                        if (row, key) in pairs:
                            for h in range(hk * r, (hk + 1) * r):
                                assert (side, row, key, h) not in covered
                                covered.add((side, row, key, h))
                            hit += 1
                assert hit > 0, "empty query tile in an item"
        for grp in groups:
            sides = ("pp",) if op == S.OP_PREFILL_BWD else ("rp", "rr")
            for side in sides:
                for (row, key) in grp[side]:
                    for h in range(hq):
                        assert (side, row, key, h) in covered
        # splits of one prompt KV tile partition the group's query tiles, in order
        for (g, tile, hk), lst in split_ranges.items():
            lst.sort()
            assert [s for s, _, _ in lst] == list(range(len(lst)))
            assert lst[0][1] == 0 and all(lst[i][2] == lst[i + 1][1] for i in range(len(lst) - 1))
            assert lst[-1][2] == -(-groups[g]["lr"] // bm)


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("bm,bn", TILES)
@pytest.mark.parametrize("hq,hkv,sms", [(4, 2, 1), (4, 2, 64), (2, 2, 2), (8, 1, 1)])
def test_fused_backward_queue_covers_every_pair_once(ti, bm, bn, hq, hkv, sms):
    """The fused backward's queue (all of the backward in one call) covers the pairs of
    both backward queues: prompt->prompt, response->prompt and response->response, each
    exactly once per query head; a prompt KV tile's split 0 carries its prompt rows."""
    tree = TREES[ti]
    groups = valid_pairs(tree)
    offs = tree.offsets()
    r = hq // hkv
    q = S.build(offs, hq, hkv, S.OP_TREE_BWD, bm, bn, num_sms=sms)
    check_key_side_order(q, tree, bn)
    rb = S.build(offs, hq, hkv, S.OP_REPLAY_BWD, bm, bn, num_sms=sms)
    nsplit = {}
    for it in rb:
        if it[0] == S.PROMPT_KV:
            nsplit[int(it[1])] = max(nsplit.get(int(it[1]), 0), int(it[4]) + 1)
    covered = set()
    for it in q:
        kind, g, tile, hk, split, cost, a, b = map(int, it)
        grp = groups[g]
        assert kind in (S.TREE_PROMPT_KV, S.RESP_KV)
        ranges = []
        if kind == S.TREE_PROMPT_KV:
            k0, klen = grp["p0"], grp["lp"]
            assert split < max(1, nsplit.get(g, 1))  # the replay backward's split rule
            ranges.append((grp["r0"], grp["r0"] + grp["lr"], a, b, grp["rp"], "rp"))
            own = 0
            if split == 0:
                qa2, qb2 = (tile * bn) // bm, -(-grp["lp"] // bm)
                own = qb2 - qa2
                ranges.append((grp["p0"], grp["p0"] + grp["lp"], qa2, qb2, grp["pp"], "pp"))
            assert cost == (b - a + own) * r and cost > 0
        else:
            assert split == 0 and cost == (b - a) * r
            k0, klen = grp["r0"], grp["lr"]
            ranges.append((grp["r0"], grp["r0"] + grp["lr"], a, b, grp["rr"], "rr"))
        keys = range(k0 + tile * bn, min(k0 + (tile + 1) * bn, k0 + klen))
        assert len(keys) > 0
        for rows0, rows1, qa, qb, pairs, side in ranges:
            for qt in range(qa, qb):
                rows = range(rows0 + qt * bm, min(rows0 + (qt + 1) * bm, rows1))
                hit = 0
                for row in rows:
                    for key in keys:
                        if (row, key) in pairs:
                            for h in range(hk * r, (hk + 1) * r):
                                assert (side, row, key, h) not in covered
                                covered.add((side, row, key, h))
                            hit += 1
                assert hit > 0, "empty query tile in an item"
    for grp in groups:
        for side in ("pp", "rp", "rr"):
            for (row, key) in grp[side]:
                for h in range(hq):
                    assert (side, row, key, h) in covered


def test_lpt_order_meets_the_list_scheduling_bound():
    """Items are taken largest first within each stream (Sec. 3.4).  Any list schedule
    on m lanes has makespan <= total/m + largest item."""
    import heapq
    tree = W.Tree([300, 20], [[37, 200, 5, 90], [400, 3]])
    offs = tree.offsets()
    for op in (S.OP_PREFILL_FWD, S.OP_REPLAY_FWD, S.OP_REPLAY_BWD, S.OP_PREFILL_BWD, S.OP_TREE_BWD):
        q = S.build(offs, 4, 2, op, 16, 16, num_sms=4)
        costs = [int(c) for c in q[:, 5]]
        check_key_side_order(q, tree, 16, 2, 16)
        m = 8
        lanes = [0] * m
        for c in costs:
            heapq.heappush(lanes, heapq.heappop(lanes) + c)
        assert max(lanes) <= sum(costs) / m + max(costs)


def test_replay_split_rule_worked_examples():
    """The split-KV rule on hand-worked cases (one replay query tile of 65 KV tiles:
    an 8,192-token prompt is 64 tiles, 32 three-token branches one own tile; 32 query
    heads, one block per head and split; 152 SMs).  Candidates T = ceil(65 / s): s = 3
    gives T = 22, 96 blocks, one wave, time 22 + 2 = 24; s = 4 gives T = 17, 128
    blocks, one wave, time 19; s = 5 gives T = 13, 160 blocks, two waves, time
    2 x 15 = 30; s = 9 gives T = 8, 288 blocks, two waves, time 20.  So 4 splits
    (17 + 17 + 17 + 14 tiles)."""
    assert S.replay_fwd_splits([65], 32, 8, 152) == [4]
    # Enough items (2 * 152 or more) for the GPU: nothing splits.
    assert S.replay_fwd_splits([65] * 10, 32, 8, 152) == [1] * 10
    # Four such tiles: 128 blocks whole, one wave, time 65 + 2 = 67; two splits give
    # 256 blocks in two waves, time 2 x 35 = 70, and more splits longer still.
    assert S.replay_fwd_splits([65] * 4, 32, 8, 152) == [1] * 4
    # Three heads: every candidate down to T = 4 (17 splits of 4 tiles, 51 blocks) fits
    # in one wave, and the smallest chunk is then the fastest: time 4 + 2.
    assert S.replay_fwd_splits([65], 3, 1, 152) == [17]
    q = S.build(W.Tree([8192], [[3] * 32]).offsets(), 32, 8, S.OP_REPLAY_FWD, 128, 128, 152,
                split_replay_fwd=True)
    assert len(q) == 4 * 32
    assert sorted(set(int(c) for c in q[:, 5])) == [14, 17]
