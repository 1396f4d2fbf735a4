"""Reference builder of the tile work queues (bit-exact target of the library's).

TEST INFRASTRUCTURE ONLY: imported by tests, never by the library.

AugTree paper, Sec. 3.4: the response paths of a tree become bounded replay units,
each with a work estimate from its query length and its valid Q-KV tile count, and
units are assigned to lanes so that the most loaded lane is as light as possible
(by largest-first greedy balancing when the exact subset DP is not used).  On one GPU
a lane is a thread block: a unit is a (query tile, head) item in the forward and a
(KV tile, KV head, split) item in the backward, its weight is its number of valid
tile interactions, and blocks take items in order of decreasing weight.

The item encoding, split rule and tie-break order are the library contract written
out below in plain Python loops; the comparison with the library is bit for bit.

Order.  Every item walks the tiles of one stream: a forward item the K/V of its
group's KV head (query head h uses KV head h // r); a key-side item the Q/dO tiles of
its group for its KV head (prompt keys) or of its own branch (response keys).  The
items of a stream form a chunk; chunks go largest first by their total cost (ties by
group, KV head, branch, with -1 for a group-wide stream).  Within a chunk, replay
forward items form sub-chunks by the branch of their query tile's first row (the
branch whose keys their own-branch tiles are), largest first (ties by branch); every
other item is its chunk's only sub-chunk.  Items within a sub-chunk go largest first
(ties by tile, kind, split, head).  This keeps largest-first balancing within a
sub-chunk and makes the blocks that run side by side share one stream (cache locality
of the on-chip scheduling; the pages' balancing is across lanes of a multi-node
cluster and says nothing about it).
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

PREFILL_Q, REPLAY_Q, PROMPT_KV, RESP_KV, PREFILL_KV, TREE_PROMPT_KV = 0, 1, 2, 3, 4, 5
OP_PREFILL_FWD, OP_REPLAY_FWD, OP_REPLAY_BWD, OP_PREFILL_BWD, OP_TREE_BWD = 0, 1, 2, 3, 4
MAX_SPLIT = 64
FWD_MIN_CHUNK = 4      # KV tiles per split of a replay query tile, at least
MAX_FWD_PARTS = 4096   # partial states (query tile x head x split) of one plan, at most
FWD_BLOCK_OVERHEAD = 2  # a block's fixed cost in KV tiles, for the choice of the chunk


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def _groups(offsets):
    prompt_off, branch_begin, resp_off = [list(map(int, x)) for x in offsets]
    out = []
    for g in range(len(prompt_off) - 1):
        p0, p1 = prompt_off[g], prompt_off[g + 1]
        b0, b1 = branch_begin[g], branch_begin[g + 1]
        starts = [resp_off[b] for b in range(b0, b1)]
        ends = [resp_off[b + 1] for b in range(b0, b1)]
        r0, r1 = resp_off[b0], resp_off[b1]
        out.append(dict(p0=p0, lp=p1 - p0, r0=r0, lr=r1 - r0, starts=starts, ends=ends))
    return out


def _branch_of(grp, row: int) -> int:
    """Index (within the group) of the branch holding global response row `row`;
    empty branches are skipped."""
    for i, (s, e) in enumerate(zip(grp["starts"], grp["ends"])):
        if s <= row < e:
            return i
    raise ValueError("row outside the group's branches")


def _fwd_split_count(cost: int, target: int) -> int:
    """Splits of one replay query tile walking `cost` KV tiles, at about `target` tiles
    each (at most MAX_SPLIT; equal chunks of ceil(cost / s) tiles, the last shorter)."""
    s = min(MAX_SPLIT, max(1, _cdiv(cost, target)))
    return _cdiv(cost, _cdiv(cost, s)) if cost > 0 else 1


def replay_fwd_splits(costs: List[int], hq: int, hkv: int, num_sms: int) -> List[int]:
    """Split-KV rule of the replay forward (tensor-core kernels), per replay query tile
    with `costs[i]` KV tiles (prompt tiles, then own-branch tiles).

    AugTree paper, Sec. 3.3: a query's attention over disjoint key ranges gives partial
    online-softmax states that merge associatively into the exact result (MoveQ's
    global reduction of partial states).  Splitting a long query tile's KV walk over
    several blocks is worth it only when the queue has too few blocks for the GPU: with
    fewer than 2 * num_sms items (query tile x head) the tiles are cut into chunks of
    about T KV tiles; otherwise every tile keeps one item.  T is chosen among
    ceil(c_max / s), s = 1..64 (c_max the largest cost; T >= FWD_MIN_CHUNK when s > 1;
    at most MAX_FWD_PARTS partial states, tiles x heads x splits over split tiles), as
    the one with the least estimated time
        ceil(blocks / num_sms) * (largest chunk + FWD_BLOCK_OVERHEAD),
    the first (largest T) on ties.  A block is one split of a tile for one query head
    (Hq blocks per split of a tile); hkv does not enter."""
    n_items = len(costs) * hq
    if n_items == 0 or n_items >= 2 * num_sms:
        return [1] * len(costs)
    per_tile = hq
    cmax = max(costs)
    best_t, best_time = cmax, None
    for sc in range(1, MAX_SPLIT + 1):
        t = _cdiv(cmax, sc)
        if sc > 1 and t < FWD_MIN_CHUNK:
            break
        splits = [_fwd_split_count(c, t) for c in costs]
        if sum(s * hq for s in splits if s > 1) > MAX_FWD_PARTS:
            continue
        blocks = sum(per_tile * s for s in splits)
        chunk_max = max(_cdiv(c, s) for c, s in zip(costs, splits))
        time = _cdiv(blocks, num_sms) * (chunk_max + FWD_BLOCK_OVERHEAD)
        if best_time is None or time < best_time:
            best_t, best_time = t, time
    return [_fwd_split_count(c, best_t) for c in costs]


def build(offsets, hq: int, hkv: int, op: int, bm: int, bn: int, num_sms: int,
          split_replay_fwd: bool = False) -> np.ndarray:
    """Work queue of `op` as an int32 array [n_items, 8]:
    kind, group, tile, head, split, cost, a, b.

    split_replay_fwd: apply the split-KV rule (replay_fwd_splits) to the replay forward
    queue, as the tensor-core kernels do.  A split item k of a tile with s splits walks
    the tile's KV tiles [k C, min((k + 1) C, a + b)), C = ceil((a + b) / s), in the
    order prompt tiles then own-branch tiles; its cost is that count; a and b stay the
    tile's own."""
    r = hq // hkv
    groups = _groups(offsets)
    items: List[Tuple[int, ...]] = []
    branch_of_item = {}  # response-key items: index of the branch whose tiles they walk
    row_branch_of_item = {}  # replay forward items: branch of the query tile's first row
    if op == OP_PREFILL_FWD:
        for g, grp in enumerate(groups):
            for t in range(_cdiv(grp["lp"], bm)):
                row_end = min(grp["p0"] + (t + 1) * bm, grp["p0"] + grp["lp"])
                a = _cdiv(row_end - grp["p0"], bn)
                for h in range(hq):
                    items.append((PREFILL_Q, g, t, h, 0, a, a, 0))
    elif op == OP_REPLAY_FWD:
        tiles = []
        for g, grp in enumerate(groups):
            a = _cdiv(grp["lp"], bn)
            for t in range(_cdiv(grp["lr"], bm)):
                row_begin = grp["r0"] + t * bm
                row_end = min(row_begin + bm, grp["r0"] + grp["lr"])
                br = _branch_of(grp, row_begin)
                bstart = grp["starts"][br]
                b = _cdiv(row_end - bstart, bn)
                tiles.append((g, t, a, b, br))
        splits = replay_fwd_splits([a + b for (_, _, a, b, _) in tiles], hq, hkv, num_sms) if split_replay_fwd \
            else [1] * len(tiles)
        for (g, t, a, b, br), s in zip(tiles, splits):
            cost = a + b
            c = _cdiv(cost, s)
            for k in range(s):
                kc = cost if s == 1 else min(c, cost - k * c)
                for h in range(hq):
                    items.append((REPLAY_Q, g, t, h, k, kc, a, b))
                    row_branch_of_item[len(items) - 1] = br
    elif op in (OP_REPLAY_BWD, OP_TREE_BWD):
        # Unsplit costs first, to fix the split target.  The fused backward (all of the
        # backward in one call) uses the replay backward's split rule; split 0 of a
        # prompt KV tile also walks the prompt's own causal query tiles of that tile.
        tree = op == OP_TREE_BWD
        total = 0
        resp_items = []
        for g, grp in enumerate(groups):
            nq = _cdiv(grp["lr"], bm)
            nkp = _cdiv(grp["lp"], bn) if nq > 0 else 0
            total += nkp * nq * r * hkv
            for j in range(_cdiv(grp["lr"], bn)):
                k_lo = grp["r0"] + j * bn
                k_hi = min(k_lo + bn, grp["r0"] + grp["lr"])
                e = grp["ends"][_branch_of(grp, k_hi - 1)]
                qa = (k_lo - grp["r0"]) // bm
                qb = _cdiv(e - grp["r0"], bm)
                resp_items.append((g, j, qa, qb, _branch_of(grp, k_lo)))
                total += (qb - qa) * r * hkv
        target = max(r, _cdiv(total, 2 * num_sms))
        for g, grp in enumerate(groups):
            nq = _cdiv(grp["lr"], bm)
            nqp = _cdiv(grp["lp"], bm)
            if grp["lp"] == 0 or (nq == 0 and not tree):
                continue
            if nq == 0:
                for j in range(_cdiv(grp["lp"], bn)):
                    for h in range(hkv):
                        items.append((TREE_PROMPT_KV, g, j, h, 0, (nqp - (j * bn) // bm) * r, 0, 0))
                continue
            s = min(MAX_SPLIT, max(1, _cdiv(nq * r, target)))
            c = _cdiv(nq, s)
            s = _cdiv(nq, c)
            for j in range(_cdiv(grp["lp"], bn)):
                for k in range(s):
                    qa, qb = k * c, min((k + 1) * c, nq)
                    own = nqp - (j * bn) // bm if (tree and k == 0) else 0
                    for h in range(hkv):
                        items.append((TREE_PROMPT_KV if tree else PROMPT_KV, g, j, h, k, (qb - qa + own) * r, qa, qb))
        for (g, j, qa, qb, br) in resp_items:
            for h in range(hkv):
                items.append((RESP_KV, g, j, h, 0, (qb - qa) * r, qa, qb))
                branch_of_item[len(items) - 1] = br
    elif op == OP_PREFILL_BWD:
        for g, grp in enumerate(groups):
            nq = _cdiv(grp["lp"], bm)
            for j in range(_cdiv(grp["lp"], bn)):
                qa = (j * bn) // bm
                for h in range(hkv):
                    items.append((PREFILL_KV, g, j, h, 0, (nq - qa) * r, qa, nq))
    else:
        raise ValueError(op)
    # Chunks of one stream: (group, KV head, branch or -1), largest chunk first; within a
    # chunk, sub-chunks by the branch of a replay forward item's first query row (-1 for
    # every other item), largest first; items within a sub-chunk largest first, ties by
    # (tile, kind, split, head).
    fwd = op in (OP_PREFILL_FWD, OP_REPLAY_FWD)
    chunk = [(it[1], it[3] // r if fwd else it[3], branch_of_item.get(i, -1)) for i, it in enumerate(items)]
    sub = [c + (row_branch_of_item.get(i, -1),) for i, c in enumerate(chunk)]
    total, sub_total = {}, {}
    for c, sc, it in zip(chunk, sub, items):
        total[c] = total.get(c, 0) + it[5]
        sub_total[sc] = sub_total.get(sc, 0) + it[5]
    order = sorted(range(len(items)), key=lambda i: (-total[chunk[i]], chunk[i], -sub_total[sub[i]], sub[i][3],
                                                     -items[i][5], items[i][2], items[i][0], items[i][4],
                                                     items[i][3]))
    return np.array([items[i] for i in order], dtype=np.int32).reshape(-1, 8)


def splits_per_group(queue: np.ndarray, n_groups: int) -> List[int]:
    """Number of prompt-KV splits of each group in a replay_bwd queue."""
    s = [1] * n_groups
    for it in queue:
        if it[0] == PROMPT_KV:
            s[it[1]] = max(s[it[1]], int(it[4]) + 1)
    return s
