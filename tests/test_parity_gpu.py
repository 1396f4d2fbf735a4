"""GPU parity of the CUDA path (through the C ABI) with the fp64 oracle, element by
element, on seeded inputs that span several tiles and ragged tails, plus edge cases:
empty prompts, empty branches, groups without branches, one-token branches."""
import numpy as np
import pytest
import torch

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import attention as A
from tests.gpu_util import compare, run_cuda, run_oracle, device_inputs, GRADS

pytestmark = pytest.mark.gpu

RAGGED = [
    W.Tree([150, 0, 70], [[1, 65, 130], [20, 0], [3]]),
    W.Tree([0, 129], [[64, 1, 2, 200], []]),
    W.Tree([257], [[1] * 9 + [128, 127, 300]]),
    W.Tree([63, 1, 190], [[5, 64], [1], [0, 33, 70]]),
]


def test_tiny_config_fp32_simt(cuda_device):
    w = W.workload("tiny")
    got = run_cuda(w, kernel=at.KERNEL_SIMT)
    compare(got, run_oracle(w), "fp32")


@pytest.mark.parametrize("ti", range(len(RAGGED)))
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_fp32_simt(cuda_device, ti, d):
    w = W.custom(RAGGED[ti], hq=4, hkv=2, d=d, dtype="fp32", seed=200 + ti, scale=1.0)
    got = run_cuda(w, kernel=at.KERNEL_SIMT)
    compare(got, run_oracle(w), "fp32")


@pytest.mark.parametrize("ti", range(len(RAGGED)))
def test_ragged_bf16_simt(cuda_device, ti):
    w = W.custom(RAGGED[ti], hq=8, hkv=2, d=128, dtype="bf16", seed=300 + ti, scale=1.0)
    got = run_cuda(w, kernel=at.KERNEL_SIMT)
    compare(got, run_oracle(w), "bf16")


def test_split_k_paths_agree(cuda_device):
    """Forcing many prompt-KV splits (small balancing width) or none (large width)
    gives the same prompt gradient sums up to fp32 rounding (Eq. 2)."""
    w = W.custom(W.Tree([140], [[300, 200, 90]]), hq=4, hkv=1, d=64, dtype="fp32", seed=9)
    a = run_cuda(w, kernel=at.KERNEL_SIMT, num_sms=1)
    b = run_cuda(w, kernel=at.KERNEL_SIMT, num_sms=100000)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.FP32, kernel=at.KERNEL_SIMT, num_sms=100000)
    assert plan.workspace_bytes(at.OP_REPLAY_BWD) > 0
    for k in GRADS:
        np.testing.assert_allclose(a[k], b[k], rtol=0, atol=1e-5)
    compare(a, run_oracle(w), "fp32")


def test_prompt_gradient_is_deterministic(cuda_device):
    """The prompt dK/dV reduction has no atomics: two runs are bit-identical."""
    w = W.custom(RAGGED[0], hq=4, hkv=2, d=64, dtype="fp32", seed=11)
    t = device_inputs(w, cuda_device)
    a = run_cuda(w, kernel=at.KERNEL_SIMT, t=t, num_sms=2)
    b = run_cuda(w, kernel=at.KERNEL_SIMT, t=t, num_sms=2)
    for k in ("dk_p", "dv_p", "dk_r", "dv_r", "o_p", "o_r", "lse_p", "lse_r"):
        assert np.array_equal(a[k], b[k]), k


def test_lse_merge_matches_oracle(cuda_device):
    rng = np.random.default_rng(4)
    rows, h, d = 37, 3, 64
    oa, ob = rng.standard_normal((rows, h, d)), rng.standard_normal((rows, h, d))
    la, lb = rng.standard_normal((h, rows)) * 3, rng.standard_normal((h, rows)) * 3
    la[0, :5] = -np.inf
    lb[0, 3:8] = -np.inf
    dev = cuda_device
    T = lambda x: torch.tensor(x, dtype=torch.float32, device=dev)
    o, l = torch.empty(rows, h, d, device=dev), torch.empty(h, rows, device=dev)
    at.augtree_lse_merge(T(oa), T(la), T(ob), T(lb), o, l)
    # oracle in (O, lse) form, per head
    f32 = lambda x: x.astype(np.float32).astype(np.float64)
    ro, rl = A.lse_merge(f32(oa).transpose(1, 0, 2), f32(la), f32(ob).transpose(1, 0, 2), f32(lb))
    np.testing.assert_allclose(o.cpu().numpy().transpose(1, 0, 2), ro, atol=1e-5, rtol=0)
    got = l.cpu().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(got[fin], rl[fin], atol=1e-5, rtol=0)
    # in-place (aliasing the first operand)
    oa_t, la_t = T(oa), T(la)
    at.augtree_lse_merge(oa_t, la_t, T(ob), T(lb), oa_t, la_t)
    np.testing.assert_allclose(oa_t.cpu().numpy(), o.cpu().numpy(), atol=0, rtol=0)


def test_lse_merge_backward_matches_oracle(cuda_device):
    """The merge's backward (C ABI and the differentiable merge) against the fp64 oracle,
    with empty states on either side and on both."""
    rng = np.random.default_rng(5)
    rows, h, d = 41, 3, 64
    oa, ob = rng.standard_normal((rows, h, d)), rng.standard_normal((rows, h, d))
    la, lb = rng.standard_normal((h, rows)) * 3, rng.standard_normal((h, rows)) * 3
    la[0, :5] = -np.inf
    lb[0, 3:8] = -np.inf
    g, gl = rng.standard_normal((rows, h, d)), rng.standard_normal((h, rows))
    dev = cuda_device
    f32 = lambda x: x.astype(np.float32).astype(np.float64)
    T = lambda x: torch.tensor(x, dtype=torch.float32, device=dev)
    want = A.lse_merge_backward(f32(oa).transpose(1, 0, 2), f32(la), f32(ob).transpose(1, 0, 2), f32(lb),
                                f32(g).transpose(1, 0, 2), f32(gl))
    outs = [torch.empty(rows, h, d, device=dev), torch.empty(h, rows, device=dev),
            torch.empty(rows, h, d, device=dev), torch.empty(h, rows, device=dev)]
    at.augtree_lse_merge_bwd(T(oa), T(la), T(ob), T(lb), T(g), T(gl), *outs)
    got = [x.cpu().numpy().astype(np.float64) for x in outs]
    got[0], got[2] = got[0].transpose(1, 0, 2), got[2].transpose(1, 0, 2)
    for name, a, b in zip(("doa", "dlse_a", "dob", "dlse_b"), got, want):
        np.testing.assert_allclose(a, b, atol=1e-4, rtol=1e-5, err_msg=name)
    # through autograd
    ta, tla, tb, tlb = (T(x).requires_grad_() for x in (oa, la, ob, lb))
    o, l = at.lse_merge(ta, tla, tb, tlb)
    (o * T(g)).sum().add((torch.where(torch.isfinite(l), l, torch.zeros_like(l)) * T(gl)).sum()).backward()
    fin = np.isfinite(np.logaddexp(la, lb))
    gl_eff = np.where(fin, gl, 0.0)
    want2 = A.lse_merge_backward(f32(oa).transpose(1, 0, 2), f32(la), f32(ob).transpose(1, 0, 2), f32(lb),
                                 f32(g).transpose(1, 0, 2), gl_eff)
    for name, t, b, tr in (("oa", ta, want2[0], True), ("la", tla, want2[1], False), ("ob", tb, want2[2], True),
                           ("lb", tlb, want2[3], False)):
        a = t.grad.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(a.transpose(1, 0, 2) if tr else a, b, atol=1e-4, rtol=1e-5, err_msg=name)


def test_schedule_export_matches_host_build(cuda_device):
    w = W.custom(RAGGED[2], hq=8, hkv=2, d=128, dtype="bf16", seed=1)
    for kernel in (at.KERNEL_SIMT, at.KERNEL_TC):
        plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=kernel, num_sms=152)
        cfg = at.make_config(w.hq, w.hkv, w.d, at.BF16, 0.0, 152, kernel)
        for op in range(4):
            assert np.array_equal(plan.schedule(op), at.schedule_build(w.tree.offsets(), cfg, op))


def test_device_side_errors_are_reported(cuda_device):
    w = W.custom(RAGGED[0], hq=4, hkv=2, d=64, dtype="fp32", seed=2)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.FP32, kernel=at.KERNEL_SIMT)
    t = device_inputs(w, cuda_device)
    need = plan.workspace_bytes(at.OP_REPLAY_BWD)
    small = torch.empty(max(1, need - 256), dtype=torch.uint8, device=cuda_device)
    z = lambda x: torch.empty_like(x)
    with pytest.raises(at.AugtreeError) as e:
        at.augtree_replay_bwd(plan, t["q_r"], t["k_p"], t["v_p"], t["k_r"], t["v_r"], z(t["q_r"]),
                              torch.empty(4, w.tree.total_resp, device=cuda_device), t["do_r"], z(t["q_r"]),
                              z(t["k_r"]), z(t["v_r"]), z(t["k_p"]), z(t["v_p"]), small)
    assert e.value.status == at.ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(at.AugtreeError) as e:
        at.augtree_prefill_fwd(plan, None, t["k_p"], t["v_p"], z(t["q_p"]), None)
    assert e.value.status == at.ERR_INVALID_ARG


def test_autograd_binding_matches_oracle(cuda_device):
    w = W.custom(RAGGED[3], hq=4, hkv=1, d=64, dtype="fp32", seed=21)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.FP32, kernel=at.KERNEL_SIMT)
    t = device_inputs(w, cuda_device)
    leaves = {k: t[k].clone().requires_grad_(True) for k in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")}
    o_p, o_r, lse_p, lse_r = at.tree_attention(plan, *(leaves[k] for k in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")))
    ((o_p * t["do_p"]).sum() + (o_r * t["do_r"]).sum()).backward()
    got = {"o_p": o_p, "o_r": o_r, "lse_p": lse_p, "lse_r": lse_r}
    got.update({"d" + k: leaves[k].grad for k in leaves})
    got = {k: v.detach().double().cpu().numpy() for k, v in got.items()}
    compare(got, run_oracle(w), "fp32")


def test_autograd_binding_tensor_cores_matches_oracle(cuda_device):
    # The differentiable operator on the bf16 tensor-core kernels (its backward is one
    # augtree_tree_bwd call).
    w = W.custom(RAGGED[3], hq=8, hkv=2, d=128, dtype="bf16", seed=22)
    plan = at.Plan.from_tree(w.tree, w.hq, w.hkv, w.d, dtype=at.BF16, kernel=at.KERNEL_TC)
    t = device_inputs(w, cuda_device)
    leaves = {k: t[k].clone().requires_grad_(True) for k in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")}
    o_p, o_r, lse_p, lse_r = at.tree_attention(plan, *(leaves[k] for k in ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r")))
    ((o_p.float() * t["do_p"].float()).sum() + (o_r.float() * t["do_r"].float()).sum()).backward()
    plan.check()
    got = {"o_p": o_p, "o_r": o_r, "lse_p": lse_p, "lse_r": lse_r}
    got.update({"d" + k: leaves[k].grad for k in leaves})
    got = {k: v.detach().double().cpu().numpy() for k, v in got.items()}
    compare(got, run_oracle(w), "bf16")
