"""Helpers of the GPU parity tests: run the CUDA path through the binding on seeded
inputs and compare with the fp64 oracle on the same values."""
import numpy as np
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import attention as A

GRADS = ("dq_p", "dk_p", "dv_p", "dq_r", "dk_r", "dv_r")

# Tolerances: bf16 inputs with fp32 accumulation: forward max-abs <= 1e-2 (O and lse),
# gradients relative Frobenius <= 2e-2; fp32 mode: 1e-4 for both.
TOL = {"bf16": (1e-2, 2e-2), "fp32": (1e-4, 1e-4)}


def device_inputs(w, device):
    return {n: W.tensor_torch(w, n, device) for n in W.TENSORS}


def host_inputs(w):
    return {n: W.tensor_rows_np(w, n) for n in W.TENSORS}


def run_cuda(w, kernel=at.KERNEL_AUTO, device="cuda", num_sms=0, t=None, plan=None, fused=True):
    """Forward + backward of workload w through the C ABI (fused: one augtree_tree_bwd
    call; otherwise replay_bwd then prefill_bwd).  Returns numpy float64 arrays keyed
    like the oracle's output."""
    dt = at.BF16 if w.dtype == "bf16" else at.FP32
    if plan is None:
        plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=dt, kernel=kernel, num_sms=num_sms)
    if t is None:
        t = device_inputs(w, device)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    g = at.backward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"], o_p, lse_p, o_r, lse_r,
                    t["do_p"], t["do_r"], fused=fused)
    torch.cuda.synchronize()
    plan.check()
    out = {"o_p": o_p, "lse_p": lse_p, "o_r": o_r, "lse_r": lse_r}
    out.update(dict(zip(GRADS, g)))
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def run_oracle(w, heads_q=None, heads_kv=None):
    t = host_inputs(w)
    return A.tree_attention_direct(t, w.tree.offsets(), A.default_scale(w.d))


def rel_frob(x, ref):
    n = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / n if n > 0 else np.linalg.norm(x)


def compare(got, ref, dtype, keys=None):
    """Returns a dict of errors and asserts the tolerance."""
    fwd_tol, grad_tol = TOL[dtype]
    errs = {}
    for k in ("o_p", "o_r", "lse_p", "lse_r"):
        if keys and k not in keys:
            continue
        a, b = got[k], ref[k]
        assert a.shape == b.shape, k
        fin = np.isfinite(b)
        assert np.array_equal(np.isfinite(a), fin), f"{k}: finite pattern differs"
        errs[k] = float(np.max(np.abs(a[fin] - b[fin]))) if fin.any() else 0.0
        assert errs[k] <= fwd_tol, (k, errs[k])
    for k in GRADS:
        if keys and k not in keys:
            continue
        assert got[k].shape == ref[k].shape, k
        errs[k] = float(rel_frob(got[k], ref[k]))
        assert errs[k] <= grad_tol, (k, errs[k])
    return errs


def run_cuda_fwd(w, kernel=at.KERNEL_AUTO, device="cuda", t=None):
    """Forward only (prefill + replay) through the C ABI."""
    dt = at.BF16 if w.dtype == "bf16" else at.FP32
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=dt, kernel=kernel)
    if t is None:
        t = device_inputs(w, device)
    o_p, lse_p, o_r, lse_r = at.forward(plan, t["q_p"], t["k_p"], t["v_p"], t["q_r"], t["k_r"], t["v_r"])
    plan.check()
    out = {"o_p": o_p, "lse_p": lse_p, "o_r": o_r, "lse_r": lse_r}
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def run_oracle_fwd(w):
    t = host_inputs(w)
    return A.tree_attention_direct(t, w.tree.offsets(), A.default_scale(w.d), grad=False)
