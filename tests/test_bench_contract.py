"""The benchmark's JSON contract and its host-side arithmetic (CPU only).

The reference arm (the fp64 oracle on the host cores) runs end to end here; the GPU
arm's line is produced on a GPU machine, so its pieces that need no GPU are checked one by
one: the useful-FLOP count (AugTree paper, Sec. 3.2: valid pairs with the prompt counted
once), the replica throughput over ranks, and the launch count of one step."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def brute_pairs(tree):
    """Valid (query, key) pairs of Eq. 1 counted by enumeration: prompt causal, response
    rows over the whole prompt and their own branch up to themselves."""
    n = 0
    for lp, bl in zip(tree.prompt_lens, tree.branch_lens):
        n += sum(i + 1 for i in range(lp))
        for li in bl:
            n += sum(lp + t + 1 for t in range(li))
    return n


def test_useful_flops_count_each_valid_pair_once():
    for tree in (W.Tree([5], [[3, 4]]), W.Tree([0, 7], [[2], [1, 0, 9]]), W.Tree([12], [[]])):
        w = W.custom(tree, hq=4, hkv=2, d=64)
        n = brute_pairs(tree)
        assert tree.pair_count() == n
        # forward 4 D Hq per pair (QK^T, PV), backward 10 D Hq (five products)
        assert bench.useful_flops(w) == 14 * 64 * 4 * n


def test_reference_arm_prints_the_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 1 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert cb["full_step_s_extrapolated"] > 0 and cb["cpu_model"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_replica_throughput_single_process():
    rate, ms = bench.replica_throughput(1000.0, 250.0, 1)
    assert ms == 250.0 and rate == 4000.0


class _FakePlan:
    """Stand-in for a plan: queue shapes and totals only."""

    def __init__(self, tree, split):
        self.total_prompt, self.total_resp = tree.total_prompt, tree.total_resp
        self.split = split

    def schedule(self, op):
        q = np.zeros((3, 8), dtype=np.int32)
        if op == 4 and self.split:
            q[1, 4] = 1
        return q


class _Ops:
    OP_PREFILL_FWD, OP_REPLAY_FWD, OP_REPLAY_BWD, OP_PREFILL_BWD, OP_TREE_BWD = 0, 1, 2, 3, 4


def test_launch_count_of_one_step():
    tree = W.Tree([40], [[10, 20]])
    # two forwards; fused backward: 2 preprocess, key side, (split reduce), 2 query side
    assert bench.count_launches(_FakePlan(tree, False), _Ops, fused=True) == 2 + 5
    assert bench.count_launches(_FakePlan(tree, True), _Ops, fused=True) == 2 + 6
    # two calls: replay 4 (preprocess, key side, split reduce, query side), prefill 3
    assert bench.count_launches(_FakePlan(tree, False), _Ops, fused=False) == 2 + 4 + 3


def test_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` without a launcher re-runs itself under torch.distributed.run
    with two ranks (CPU here: the reference arm, whose rank 0 alone works and prints)."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--workload", "tiny",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
