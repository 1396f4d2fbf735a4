"""The C-ABI library without a GPU: it loads, exports every entry point the header
declares, builds the work queues bit-exactly like the reference builder, and rejects
bad descriptors and configs on the host."""
import ctypes
import os
import re

import numpy as np
import pytest

import shared_prompt_tree_gb300 as at
from oracle import schedule as S
import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "augtree.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(augtree_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(augtree_lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(augtree_lib, n), n
    assert at.lib().augtree_version() >= 100
    assert at.status_string(at.ERR_WORKSPACE_TOO_SMALL) == "workspace too small"


TREES = [
    W.Tree([5], [[3, 4]]),
    W.Tree([700, 33], [[1, 600, 250], [400]]),
    W.Tree([0, 410], [[300, 200], [0, 570]]),
    W.Tree([640, 2, 300], [[], [310], [1, 1, 1, 170]]),
    W.Tree([1300], [[9] * 70 + [650]]),
]


@pytest.mark.parametrize("ti", range(len(TREES)))
@pytest.mark.parametrize("kernel,dtype", [(at.KERNEL_SIMT, at.FP32), (at.KERNEL_TC, at.BF16), (at.KERNEL_AUTO, at.FP32)])
@pytest.mark.parametrize("hq,hkv,sms", [(4, 2, 3), (32, 8, 152), (2, 2, 1)])
def test_schedule_bit_exact_with_reference_builder(augtree_lib, ti, kernel, dtype, hq, hkv, sms):
    tree = TREES[ti]
    cfg = at.make_config(hq, hkv, 128, dtype, 0.0, sms, kernel)
    for op in range(5):
        bm, bn = at.tile_sizes(cfg, op)
        got = at.schedule_build(tree.offsets(), cfg, op)
        want = S.build(tree.offsets(), hq, hkv, op, bm, bn, sms, split_replay_fwd=kernel == at.KERNEL_TC)
        assert got.shape == want.shape and np.array_equal(got, want), (op, bm, bn)


def test_schedule_bit_exact_on_the_benchmark_shapes(augtree_lib):
    for name in ("response_heavy", "mixed", "prompt_heavy"):
        w = W.workload(name)
        cfg = at.make_config(w.hq, w.hkv, w.d, at.BF16, 0.0, 152, at.KERNEL_TC)
        for op in range(5):
            bm, bn = at.tile_sizes(cfg, op)
            got = at.schedule_build(w.tree.offsets(), cfg, op)
            want = S.build(w.tree.offsets(), w.hq, w.hkv, op, bm, bn, 152, split_replay_fwd=True)
            assert np.array_equal(got, want), (name, op)


def _status(offsets, cfg, op=0, cap=10 ** 6):
    d, keep = at.make_desc(*offsets)
    n = ctypes.c_size_t()
    out = np.zeros((max(cap, 1), 8), dtype=np.int32)
    return at.lib().augtree_schedule_build(ctypes.byref(d), ctypes.byref(cfg), op, out.ctypes.data, cap,
                                           ctypes.byref(n)), n.value


def test_host_validation_errors(augtree_lib):
    good = W.Tree([5, 3], [[2, 2], [4]]).offsets()
    cfg = at.make_config(4, 2, 128, at.BF16, 0.0, 8)
    assert _status(good, cfg)[0] == at.OK
    po, bb, ro = good
    # decreasing prompt offsets, nonzero first offsets, branch count mismatch
    assert _status((np.array([0, 5, 4]), bb, ro), cfg)[0] == at.ERR_INVALID_ARG
    assert _status((np.array([1, 5, 8]), bb, ro), cfg)[0] == at.ERR_INVALID_ARG
    assert _status((po, np.array([0, 2, 2]), ro), cfg)[0] == at.ERR_INVALID_ARG
    assert _status((po, bb, np.array([0, 2, 1, 5])), cfg)[0] == at.ERR_INVALID_ARG
    # unsupported configs
    assert _status(good, at.make_config(4, 3, 128, at.BF16, 0.0, 8))[0] == at.ERR_UNSUPPORTED
    assert _status(good, at.make_config(4, 2, 96, at.BF16, 0.0, 8))[0] == at.ERR_UNSUPPORTED
    assert _status(good, at.make_config(4, 2, 128, 7, 0.0, 8))[0] == at.ERR_UNSUPPORTED
    assert _status(good, at.make_config(4, 2, 128, at.FP32, 0.0, 8, at.KERNEL_TC))[0] == at.ERR_UNSUPPORTED
    # bad values
    assert _status(good, at.make_config(0, 2, 128, at.BF16, 0.0, 8))[0] == at.ERR_INVALID_ARG
    assert _status(good, at.make_config(4, 2, 128, at.BF16, -1.0, 8))[0] == at.ERR_INVALID_ARG
    assert _status(good, at.make_config(4, 2, 128, at.BF16, 0.0, 0))[0] == at.ERR_INVALID_ARG  # host build needs SMs
    assert _status(good, at.make_config(4, 2, 128, at.BF16, 0.0, 8, 9))[0] == at.ERR_INVALID_ARG
    assert _status(good, cfg, op=at.OP_TREE_BWD)[0] == at.OK
    assert _status(good, cfg, op=5)[0] == at.ERR_INVALID_ARG
    # capacity
    st, n = _status(good, cfg, cap=1)
    assert st == at.ERR_CAPACITY and n > 1
    # null pointers
    n = ctypes.c_size_t()
    assert at.lib().augtree_schedule_build(None, ctypes.byref(cfg), 0, None, 0, ctypes.byref(n)) == at.ERR_INVALID_ARG
    assert at.lib().augtree_plan_destroy(None) == at.ERR_INVALID_ARG
    assert at.lib().augtree_lse_merge(-1, 1, 1, None, None, None, None, None, None, None) == at.ERR_INVALID_ARG
    assert at.lib().augtree_lse_merge(0, 1, 1, None, None, None, None, None, None, None) == at.OK


def test_empty_structures_build_empty_queues(augtree_lib):
    cfg = at.make_config(2, 1, 64, at.FP32, 0.0, 4)
    for tree in (W.Tree([0], [[0]]), W.Tree([], []), W.Tree([3], [[]])):
        for op in range(5):
            q = at.schedule_build(tree.offsets(), cfg, op)
            want = S.build(tree.offsets(), 2, 1, op, 64, 64, 4)
            assert np.array_equal(q, want)


def declared_param_counts():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(augtree_\w+)\s*\(([^)]*)\)\s*;", src):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_binding_signatures_match_the_header(augtree_lib):
    counts = declared_param_counts()
    assert set(counts) == set(at._SIGS), set(counts) ^ set(at._SIGS)
    for name, n in counts.items():
        assert len(at._SIGS[name]) == n, (name, len(at._SIGS[name]), n)
