"""The checked build (-DAUGTREE_CHECKED=1): every kernel validates its work item against
the plan's geometry before it uses any index the item implies; a failing item sets a
bit of the plan's error word (augtree_plan_check returns AUGTREE_ERR_DEVICE_CHECK) and
is skipped, never trapped.  It stands in for a sanitizer on a GPU where none may run.

Built into a temporary directory and run in a child process (the binding loads one
library per process):
  * CPU: the checked variant compiles for sm_103a;
  * GPU: with it, forward and backward match the oracle on ragged trees for both kernel
    families, no check fails, and the fused backward's dK/dV are bit-identical across
    two runs (the prompt gradient's reduction is atomic-free).
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, sys.argv[2])
import shared_prompt_tree_gb300 as at
at.LIB_PATH = sys.argv[1]
import torch
import workloads as W
from tests.gpu_util import compare, device_inputs, run_cuda, run_oracle
torch.cuda.set_device(0)
cases = [
    (W.Tree([300, 129], [[129, 1, 200], [64, 3]]), 8, 2, 128, "bf16", at.KERNEL_TC),
    (W.Tree([0, 257], [[70, 1], [1] * 5 + [130]]), 6, 2, 128, "bf16", at.KERNEL_TC),
    (W.Tree([150, 33], [[65, 1, 20], [40]]), 4, 2, 64, "fp32", at.KERNEL_SIMT),
]
for tree, hq, hkv, d, dt, kernel in cases:
    w = W.custom(tree, hq=hq, hkv=hkv, d=d, dtype=dt, seed=23)
    ref = run_oracle(w)
    for fused in (True, False):
        got = run_cuda(w, kernel=kernel, fused=fused)  # plan.check() inside: raises on a failed check
        compare(got, ref, dt)
    if kernel == at.KERNEL_TC:
        t = device_inputs(w, "cuda")
        plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=kernel)
        a = run_cuda(w, kernel=kernel, t=t, plan=plan)
        b = run_cuda(w, kernel=kernel, t=t, plan=plan)
        for k in ("dk_p", "dv_p", "dk_r", "dv_r"):
            assert (a[k] == b[k]).all(), k
print("checked build ok")
'''


def _build(tmp_path):
    sys.path.insert(0, ROOT)
    from shared_prompt_tree_gb300 import build
    return build.build_variant(["-DAUGTREE_CHECKED=1"], str(tmp_path / "checked"))


def test_checked_variant_compiles(tmp_path):
    lib = _build(tmp_path)
    assert os.path.getsize(lib) > 0


@pytest.mark.gpu
def test_checked_build_matches_oracle_and_records_no_failure(tmp_path, cuda_device):
    lib = _build(tmp_path)
    r = subprocess.run([sys.executable, "-c", CHILD, lib, ROOT], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "checked build ok" in r.stdout
