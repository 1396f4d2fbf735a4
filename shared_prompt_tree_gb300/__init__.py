"""Exact, differentiable shared-prompt tree attention on one GB300 (sm_103a).

A thin binding over the C ABI of libaugtree.so (include/augtree.h): argument
marshalling only.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and importing an op without the built library
raises.  PyTorch supplies device memory and the current stream.

AugTree, "Splitting Prompt Prefill from Response Replay for Context-Parallel
Long-Context LLM Post-Training": a group is a replay tree (P, {R_i}) (Sec. 3.1); the
prompt is prefilled once with causal attention and its K/V are shared by every
branch (Sec. 3.2); a response row attends to the whole prompt and to its own branch
up to itself (Eq. 1); the prompt K/V gradient is the sum over all branches and flows
back through the prefill (Eq. 2).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libaugtree.so")

# augtree_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_DEVICE_CHECK, ERR_TIMEOUT, \
    ERR_CAPACITY = range(8)
FP32, BF16 = 0, 1
KERNEL_AUTO, KERNEL_SIMT, KERNEL_TC = 0, 1, 2
SCHED_QUEUE, SCHED_PERSISTENT = 0, 1
LANES_EXACT_UNITS = 12
KID_FWD_TC, KID_BWD_KEY_SIDE, KID_BWD_QUERY_SIDE = 1, 4, 6
OP_PREFILL_FWD, OP_REPLAY_FWD, OP_REPLAY_BWD, OP_PREFILL_BWD, OP_TREE_BWD = 0, 1, 2, 3, 4
# augtree_kernel_id: kinds reported by augtree_plan_kernel_times
KERNEL_IDS = {1: "fwd_tc", 2: "fwd_simt", 3: "preprocess", 4: "bwd_key_side", 5: "split_reduce",
              6: "bwd_query_side", 7: "dq_convert", 8: "bwd_simt", 9: "fwd_split_merge", 10: "dq_split_reduce"}
TIMING_RING = 64
ITEM_WORDS = 8


class AugtreeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Desc(ctypes.Structure):
    _fields_ = [("prompt_off", ctypes.POINTER(ctypes.c_int32)),
                ("branch_begin", ctypes.POINTER(ctypes.c_int32)),
                ("resp_off", ctypes.POINTER(ctypes.c_int32)),
                ("n_groups", ctypes.c_int32),
                ("n_branches", ctypes.c_int32)]


class Config(ctypes.Structure):
    _fields_ = [("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("softmax_scale", ctypes.c_float), ("num_sms", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("schedule", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_SZ = ctypes.c_size_t

# name -> argument types (all return int32 status unless listed in _RESTYPE)
_SIGS = {
    "augtree_tile_sizes": [ctypes.POINTER(Config), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                           ctypes.POINTER(ctypes.c_int32)],
    "augtree_schedule_build": [ctypes.POINTER(Desc), ctypes.POINTER(Config), ctypes.c_int32, _P, _SZ,
                               ctypes.POINTER(_SZ)],
    "augtree_schedule_lanes": [ctypes.POINTER(Desc), ctypes.POINTER(Config), ctypes.c_int32, ctypes.c_int32, _P, _SZ,
                               _P, _SZ, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)],
    "augtree_assign_grid": [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P,
                            ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)],
    "augtree_plan_create": [ctypes.POINTER(Desc), ctypes.POINTER(Config), ctypes.POINTER(_P)],
    "augtree_plan_destroy": [_P],
    "augtree_plan_workspace_bytes": [_P, ctypes.c_int32, ctypes.POINTER(_SZ)],
    "augtree_schedule_export": [_P, ctypes.c_int32, _P, _SZ, ctypes.POINTER(_SZ)],
    "augtree_prefill_fwd": [_P] * 7 + [_SZ, _P],
    "augtree_replay_fwd": [_P] * 8 + [_P, _SZ, _P],
    "augtree_replay_bwd": [_P] * 15 + [_SZ, _P],
    "augtree_prefill_bwd": [_P] * 13 + [_SZ, _P],
    "augtree_prefill_bwd_static": [_P] * 13,
    "augtree_tree_bwd": [_P] * 20 + [_SZ, _P],
    "augtree_lse_merge": [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32] + [_P] * 6 + [_P],
    "augtree_lse_merge_bwd": [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32] + [_P] * 10 + [_P],
    "augtree_plan_check": [_P, _P],
    "augtree_plan_set_wait_limit": [_P, ctypes.c_uint64],
    "augtree_plan_set_timing": [_P, ctypes.c_int32],
    "augtree_plan_kernel_times": [_P, ctypes.c_int32, ctypes.c_int32, _P, _P, ctypes.c_int32,
                                  ctypes.POINTER(ctypes.c_int32)],
    "augtree_status_string": [ctypes.c_int32],
    "augtree_version": [],
}
_RESTYPE = {"augtree_status_string": ctypes.c_char_p, "augtree_version": ctypes.c_int32}


def lib():
    """The loaded C library.  Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with shared_prompt_tree_gb300.build.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _RESTYPE.get(name, ctypes.c_int32)
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().augtree_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status: int, where: str):
    if status != OK:
        raise AugtreeError(status, where)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def make_desc(prompt_off, branch_begin, resp_off):
    """Desc struct plus the int32 arrays it points into (keep them alive together)."""
    po, bb, ro = _i32(prompt_off), _i32(branch_begin), _i32(resp_off)
    ip = ctypes.POINTER(ctypes.c_int32)
    d = Desc(po.ctypes.data_as(ip), bb.ctypes.data_as(ip), ro.ctypes.data_as(ip), len(po) - 1, len(ro) - 1)
    return d, (po, bb, ro)


def make_config(hq, hkv, head_dim, dtype=BF16, softmax_scale=0.0, num_sms=0, kernel=KERNEL_AUTO,
                schedule=SCHED_QUEUE):
    return Config(hq, hkv, head_dim, dtype, softmax_scale, num_sms, kernel, schedule)


def tile_sizes(cfg: Config, op: int):
    bm, bn = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().augtree_tile_sizes(ctypes.byref(cfg), op, ctypes.byref(bm), ctypes.byref(bn)), "augtree_tile_sizes")
    return bm.value, bn.value


def schedule_build(offsets, cfg: Config, op: int) -> np.ndarray:
    """Host-only work queue of `op` as int32 [n_items, 8] (no GPU needed)."""
    d, keep = make_desc(*offsets)
    n = _SZ()
    st = lib().augtree_schedule_build(ctypes.byref(d), ctypes.byref(cfg), op, None, 0, ctypes.byref(n))
    if st not in (OK, ERR_CAPACITY):
        _check(st, "augtree_schedule_build")
    out = np.zeros((max(1, n.value), ITEM_WORDS), dtype=np.int32)
    _check(lib().augtree_schedule_build(ctypes.byref(d), ctypes.byref(cfg), op, out.ctypes.data, n.value,
                                        ctypes.byref(n)), "augtree_schedule_build")
    return out[:n.value]


def schedule_lanes(offsets, cfg: Config, op: int, kernel_id: int):
    """Host-only persistent-schedule placement of a kernel's work units on lanes
    (AssignGrid over the queue's unit costs).  Returns (lane_off int32 [n_lanes+1],
    units int32 [n_units]): lane l runs units[lane_off[l]:lane_off[l+1]] in order."""
    d, keep = make_desc(*offsets)
    nl, nu = _SZ(), _SZ()
    st = lib().augtree_schedule_lanes(ctypes.byref(d), ctypes.byref(cfg), op, kernel_id, None, 0, None, 0,
                                      ctypes.byref(nl), ctypes.byref(nu))
    if st not in (OK, ERR_CAPACITY):
        _check(st, "augtree_schedule_lanes")
    off = np.zeros(nl.value + 1, dtype=np.int32)
    units = np.zeros(max(1, nu.value), dtype=np.int32)
    _check(lib().augtree_schedule_lanes(ctypes.byref(d), ctypes.byref(cfg), op, kernel_id, off.ctypes.data,
                                        off.size, units.ctypes.data, units.size, ctypes.byref(nl),
                                        ctypes.byref(nu)), "augtree_schedule_lanes")
    return off, units[:nu.value]


ASSIGN_GRID_MAX_EXACT = 16


def assign_grid(w, rounds: int, lanes: int, u_max: int = 12):
    """AssignGrid (host only): places replay units with work estimates `w` on a grid of
    `rounds` x `lanes` cells, one unit per cell, minimising the largest lane total;
    exact for len(w) <= u_max, largest-first greedy otherwise (u_max=0: always greedy).
    Returns (round int32 [U], lane int32 [U], makespan, exact)."""
    wa = np.ascontiguousarray(np.asarray(w, dtype=np.int64))
    n = int(wa.size)
    rnd = np.zeros(max(1, n), dtype=np.int32)
    lane = np.zeros(max(1, n), dtype=np.int32)
    mk, ex = ctypes.c_int64(), ctypes.c_int32()
    _check(lib().augtree_assign_grid(wa.ctypes.data if n else None, n, int(rounds), int(lanes), int(u_max),
                                     rnd.ctypes.data, lane.ctypes.data, ctypes.byref(mk), ctypes.byref(ex)),
           "augtree_assign_grid")
    return rnd[:n], lane[:n], int(mk.value), bool(ex.value)


class Plan:
    """A plan: validated descriptors plus the device work queues (augtree_plan_create).
    Must be created with the target CUDA device current."""

    def __init__(self, prompt_off, branch_begin, resp_off, hq, hkv, head_dim, dtype=BF16, softmax_scale=0.0,
                 num_sms=0, kernel=KERNEL_AUTO, schedule=SCHED_QUEUE):
        self.cfg = make_config(hq, hkv, head_dim, dtype, softmax_scale, num_sms, kernel, schedule)
        d, (po, bb, ro) = make_desc(prompt_off, branch_begin, resp_off)
        self.prompt_off, self.branch_begin, self.resp_off = po, bb, ro
        self.total_prompt, self.total_resp = int(po[-1]), int(ro[-1])
        self.hq, self.hkv, self.head_dim, self.dtype = hq, hkv, head_dim, dtype
        self.softmax_scale = softmax_scale
        h = _P()
        _check(lib().augtree_plan_create(ctypes.byref(d), ctypes.byref(self.cfg), ctypes.byref(h)),
               "augtree_plan_create")
        self.handle = h

    @classmethod
    def from_tree(cls, tree, hq, hkv, head_dim, **kw):
        return cls(*tree.offsets(), hq, hkv, head_dim, **kw)

    def workspace_bytes(self, op: int) -> int:
        n = _SZ()
        _check(lib().augtree_plan_workspace_bytes(self.handle, op, ctypes.byref(n)), "augtree_plan_workspace_bytes")
        return n.value

    def schedule(self, op: int) -> np.ndarray:
        n = _SZ()
        st = lib().augtree_schedule_export(self.handle, op, None, 0, ctypes.byref(n))
        if st not in (OK, ERR_CAPACITY):
            _check(st, "augtree_schedule_export")
        out = np.zeros((max(1, n.value), ITEM_WORDS), dtype=np.int32)
        _check(lib().augtree_schedule_export(self.handle, op, out.ctypes.data, n.value, ctypes.byref(n)),
               "augtree_schedule_export")
        return out[:n.value]

    def set_timing(self, enable: bool):
        """Per-kernel timing of this plan's calls (CUDA events around each launch)."""
        _check(lib().augtree_plan_set_timing(self.handle, 1 if enable else 0), "augtree_plan_set_timing")

    def kernel_times(self, op: int, back: int = 0):
        """[(kind, ms)] of the kernels of the back-th most recent timed call of op."""
        kind = (ctypes.c_int32 * 8)()
        ms = (ctypes.c_float * 8)()
        n = ctypes.c_int32()
        _check(lib().augtree_plan_kernel_times(self.handle, op, back, ctypes.cast(kind, _P), ctypes.cast(ms, _P), 8,
                                               ctypes.byref(n)), "augtree_plan_kernel_times")
        return [(KERNEL_IDS.get(kind[i], str(kind[i])), float(ms[i])) for i in range(n.value)]

    def set_wait_limit(self, ns: int):
        """Limit in nanoseconds of a device-side wait on another warp's work (2 s by
        default); a kernel that runs past it gives up and check() raises ERR_TIMEOUT."""
        _check(lib().augtree_plan_set_wait_limit(self.handle, int(ns)), "augtree_plan_set_wait_limit")

    def check(self, stream=None):
        """Synchronize and raise if a kernel of this plan recorded a device-side error."""
        _check(lib().augtree_plan_check(self.handle, _stream(stream)), "augtree_plan_check")

    def close(self):
        if getattr(self, "handle", None):
            lib().augtree_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------------------------
# Compute calls: the C entry points with the same names.  Tensors are torch CUDA
# tensors (or None); `stream` is a torch.cuda.Stream or None (the current stream).
# ------------------------------------------------------------------------------------
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def augtree_prefill_fwd(plan: Plan, qp, kp, vp, op, lse_p, ws=None, stream=None):
    _check(lib().augtree_prefill_fwd(plan.handle, _ptr(qp), _ptr(kp), _ptr(vp), _ptr(op), _ptr(lse_p), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "augtree_prefill_fwd")


def augtree_replay_fwd(plan: Plan, qr, kp, vp, kr, vr, or_, lse_r, ws=None, stream=None):
    _check(lib().augtree_replay_fwd(plan.handle, _ptr(qr), _ptr(kp), _ptr(vp), _ptr(kr), _ptr(vr), _ptr(or_),
                                    _ptr(lse_r), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                    _stream(stream)), "augtree_replay_fwd")


def augtree_replay_bwd(plan: Plan, qr, kp, vp, kr, vr, or_, lse_r, dor, dqr, dkr, dvr, dkp_sum, dvp_sum, ws,
                       stream=None):
    _check(lib().augtree_replay_bwd(plan.handle, _ptr(qr), _ptr(kp), _ptr(vp), _ptr(kr), _ptr(vr), _ptr(or_),
                                    _ptr(lse_r), _ptr(dor), _ptr(dqr), _ptr(dkr), _ptr(dvr), _ptr(dkp_sum),
                                    _ptr(dvp_sum), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                    _stream(stream)), "augtree_replay_bwd")


def augtree_prefill_bwd(plan: Plan, qp, kp, vp, op, lse_p, dop, dkp_acc, dvp_acc, dqp, dkp, dvp, ws, stream=None):
    _check(lib().augtree_prefill_bwd(plan.handle, _ptr(qp), _ptr(kp), _ptr(vp), _ptr(op), _ptr(lse_p), _ptr(dop),
                                     _ptr(dkp_acc), _ptr(dvp_acc), _ptr(dqp), _ptr(dkp), _ptr(dvp), _ptr(ws),
                                     0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "augtree_prefill_bwd")


def augtree_tree_bwd(plan: Plan, qp, kp, vp, op, lse_p, dop, qr, kr, vr, or_, lse_r, dor, dqp, dkp, dvp, dqr, dkr, dvr,
                     ws, stream=None):
    _check(lib().augtree_tree_bwd(plan.handle, *(_ptr(t) for t in (qp, kp, vp, op, lse_p, dop, qr, kr, vr, or_, lse_r,
                                                                  dor, dqp, dkp, dvp, dqr, dkr, dvr, ws)),
                                  0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "augtree_tree_bwd")


def augtree_prefill_bwd_static(plan: Plan, qp, kp, vp, op, lse_p, dop, dkp_acc, dvp_acc, dqp, dkp, dvp,
                               stream=None):
    """augtree_prefill_bwd without a workspace: the library's fixed 64 MiB scratch array
    is used instead, and the call allocates nothing."""
    _check(lib().augtree_prefill_bwd_static(plan.handle, _ptr(qp), _ptr(kp), _ptr(vp), _ptr(op), _ptr(lse_p),
                                            _ptr(dop), _ptr(dkp_acc), _ptr(dvp_acc), _ptr(dqp), _ptr(dkp), _ptr(dvp),
                                            _stream(stream)), "augtree_prefill_bwd_static")


def augtree_lse_merge(oa, lse_a, ob, lse_b, o, lse, stream=None):
    """(O, lse) state merge of fp32 tensors oa/ob/o [rows, h, d], lse [h, rows]."""
    rows, h, d = oa.shape
    _check(lib().augtree_lse_merge(rows, h, d, _ptr(oa), _ptr(lse_a), _ptr(ob), _ptr(lse_b), _ptr(o), _ptr(lse),
                                   _stream(stream)), "augtree_lse_merge")


def augtree_lse_merge_bwd(oa, lse_a, ob, lse_b, dout, dlse, doa, dlse_a, dob, dlse_b, stream=None):
    """Gradients of the (O, lse) merge with respect to its inputs (dlse may be None)."""
    rows, h, d = oa.shape
    _check(lib().augtree_lse_merge_bwd(rows, h, d, _ptr(oa), _ptr(lse_a), _ptr(ob), _ptr(lse_b), _ptr(dout),
                                       _ptr(dlse), _ptr(doa), _ptr(dlse_a), _ptr(dob), _ptr(dlse_b),
                                       _stream(stream)), "augtree_lse_merge_bwd")


# ------------------------------------------------------------------------------------
# Autograd
# ------------------------------------------------------------------------------------
def _torch_dtype(plan: Plan):
    import torch
    return torch.bfloat16 if plan.dtype == BF16 else torch.float32


def _empty(shape, plan, device, dtype=None):
    import torch
    return torch.empty(shape, dtype=dtype or _torch_dtype(plan), device=device)


def forward(plan: Plan, q_p, k_p, v_p, q_r, k_r, v_r):
    """Prefill + replay forward.  Returns o_p, lse_p, o_r, lse_r."""
    import torch
    dev = (q_p if q_p.numel() else q_r).device
    o_p = _empty(q_p.shape, plan, dev)
    o_r = _empty(q_r.shape, plan, dev)
    lse_p = _empty((plan.hq, plan.total_prompt), plan, dev, torch.float32)
    lse_r = _empty((plan.hq, plan.total_resp), plan, dev, torch.float32)
    augtree_prefill_fwd(plan, q_p, k_p, v_p, o_p, lse_p)
    # Split-KV partial states of the replay forward (only when its queue is split).
    n_ws = plan.workspace_bytes(OP_REPLAY_FWD)
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev) if n_ws else None
    augtree_replay_fwd(plan, q_r, k_p, v_p, k_r, v_r, o_r, lse_r, ws)
    return o_p, lse_p, o_r, lse_r


def backward(plan: Plan, q_p, k_p, v_p, q_r, k_r, v_r, o_p, lse_p, o_r, lse_r, do_p, do_r, fused: bool = True):
    """The tree backward (the prompt K/V gradient sums every branch's replay gradient and
    the prompt's own causal part, Eq. 2).  fused: one augtree_tree_bwd call; otherwise
    the replay backward, then the prefill backward that adds its sums.
    Returns dq_p, dk_p, dv_p, dq_r, dk_r, dv_r."""
    import torch
    dev = (q_p if q_p.numel() else q_r).device
    if fused:
        dq_p, dk_p, dv_p = _empty(q_p.shape, plan, dev), _empty(k_p.shape, plan, dev), _empty(v_p.shape, plan, dev)
        dq_r, dk_r, dv_r = _empty(q_r.shape, plan, dev), _empty(k_r.shape, plan, dev), _empty(v_r.shape, plan, dev)
        ws = torch.empty(max(1, plan.workspace_bytes(OP_TREE_BWD)), dtype=torch.uint8, device=dev)
        augtree_tree_bwd(plan, q_p, k_p, v_p, o_p, lse_p, do_p, q_r, k_r, v_r, o_r, lse_r, do_r, dq_p, dk_p, dv_p,
                         dq_r, dk_r, dv_r, ws)
        return dq_p, dk_p, dv_p, dq_r, dk_r, dv_r
    f32 = torch.float32
    dq_r, dk_r, dv_r = _empty(q_r.shape, plan, dev), _empty(k_r.shape, plan, dev), _empty(v_r.shape, plan, dev)
    dkp_sum = _empty(k_p.shape, plan, dev, f32)
    dvp_sum = _empty(v_p.shape, plan, dev, f32)
    ws = torch.empty(max(1, plan.workspace_bytes(OP_REPLAY_BWD)), dtype=torch.uint8, device=dev)
    augtree_replay_bwd(plan, q_r, k_p, v_p, k_r, v_r, o_r, lse_r, do_r, dq_r, dk_r, dv_r, dkp_sum, dvp_sum, ws)
    dq_p, dk_p, dv_p = _empty(q_p.shape, plan, dev), _empty(k_p.shape, plan, dev), _empty(v_p.shape, plan, dev)
    ws2 = torch.empty(max(1, plan.workspace_bytes(OP_PREFILL_BWD)), dtype=torch.uint8, device=dev)
    augtree_prefill_bwd(plan, q_p, k_p, v_p, o_p, lse_p, do_p, dkp_sum, dvp_sum, dq_p, dk_p, dv_p, ws2)
    return dq_p, dk_p, dv_p, dq_r, dk_r, dv_r


def _autograd_fn():
    import torch

    class TreeAttentionFn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, plan, q_p, k_p, v_p, q_r, k_r, v_r):
            ts = [t.contiguous() for t in (q_p, k_p, v_p, q_r, k_r, v_r)]
            o_p, lse_p, o_r, lse_r = forward(plan, *ts)
            ctx.plan = plan
            ctx.save_for_backward(*ts, o_p, lse_p, o_r, lse_r)
            ctx.mark_non_differentiable(lse_p, lse_r)
            return o_p, o_r, lse_p, lse_r

        @staticmethod
        def backward(ctx, do_p, do_r, _dlse_p, _dlse_r):
            q_p, k_p, v_p, q_r, k_r, v_r, o_p, lse_p, o_r, lse_r = ctx.saved_tensors
            if do_p is None:
                do_p = torch.zeros_like(o_p)
            if do_r is None:
                do_r = torch.zeros_like(o_r)
            g = backward(ctx.plan, q_p, k_p, v_p, q_r, k_r, v_r, o_p, lse_p, o_r, lse_r,
                         do_p.contiguous(), do_r.contiguous())
            return (None,) + g

    return TreeAttentionFn


_FN = None


_MERGE_FN = None


def _merge_fn():
    import torch

    class LseMergeFn(torch.autograd.Function):
        """(O, lse) merge of two partial attention states as a differentiable operator."""

        @staticmethod
        def forward(ctx, oa, lse_a, ob, lse_b):
            oa, lse_a, ob, lse_b = (x.contiguous() for x in (oa, lse_a, ob, lse_b))
            o, lse = torch.empty_like(oa), torch.empty_like(lse_a)
            augtree_lse_merge(oa, lse_a, ob, lse_b, o, lse)
            ctx.save_for_backward(oa, lse_a, ob, lse_b)
            return o, lse

        @staticmethod
        def backward(ctx, do, dlse):
            oa, lse_a, ob, lse_b = ctx.saved_tensors
            do = torch.zeros_like(oa) if do is None else do.contiguous()
            dlse = None if dlse is None else dlse.contiguous()
            doa, dob = torch.empty_like(oa), torch.empty_like(ob)
            dla, dlb = torch.empty_like(lse_a), torch.empty_like(lse_b)
            augtree_lse_merge_bwd(oa, lse_a, ob, lse_b, do, dlse, doa, dla, dob, dlb)
            return doa, dla, dob, dlb

    return LseMergeFn


def lse_merge(oa, lse_a, ob, lse_b):
    """Differentiable (O, lse) merge of fp32 CUDA tensors oa/ob [rows, h, d], lse [h, rows]."""
    global _MERGE_FN
    if _MERGE_FN is None:
        _MERGE_FN = _merge_fn()
    return _MERGE_FN.apply(oa, lse_a, ob, lse_b)


def tree_attention(plan: Plan, q_p, k_p, v_p, q_r, k_r, v_r):
    """Differentiable tree attention: returns (o_p, o_r, lse_p, lse_r).  Gradients
    reach q/k/v of both the prompt and the responses; the prompt K/V gradient is the
    sum over every branch plus the prompt's own causal part."""
    global _FN
    if _FN is None:
        _FN = _autograd_fn()
    return _FN.apply(plan, q_p, k_p, v_p, q_r, k_r, v_r)
