"""Seeded synthetic workloads for shared-prompt tree attention.

This module only produces inputs: tree shapes (prompt and branch lengths), their
offset descriptors, and tensor values.  It contains none of the attention arithmetic,
so that the fp64 oracle and the CUDA path can both read identical inputs without
sharing any of the method's code.

Tree shapes follow the AugTree paper ("Splitting Prompt Prefill from Response Replay
for Context-Parallel Long-Context LLM Post-Training"), Sec. 2.1 and 3.1: a replay
tree is one prompt P and G response branches R_1..R_G.  Groups are laid out one
after another; inside a group the branches are contiguous (THD packing).

Tensor values come from a counter-based generator so that any subset of rows can be
regenerated on the host (numpy) or the whole tensor on the device (torch), giving
bit-identical values:

    h(i)  = element hash of (seed, tensor id, flat element index i), built from the
            32-bit "lowbias32" integer hash (C. Wellons, hash-prospector);
    value = scale * T[h(i) >> 16]

where T is a 65536-entry table of standard-normal quantiles,
T[k] = Phi^-1((k + 0.5) / 65536), rounded to the tensor's storage dtype.  The values
are therefore N(0,1) quantised to 65536 levels (tails cut at |z| = 4.32); for bf16
storage this is indistinguishable from rounding an N(0,1) draw to bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

# Tensor ids used by the element hash.
TENSORS = ("q_p", "k_p", "v_p", "q_r", "k_r", "v_r", "do_p", "do_r")
TENSOR_ID = {name: i for i, name in enumerate(TENSORS)}

_M32 = 0xFFFFFFFF


# ----------------------------------------------------------------------------------
# Tree shapes
# ----------------------------------------------------------------------------------
@dataclasses.dataclass
class Tree:
    """A batch of replay trees: group g has prompt length prompt_lens[g] and
    branches with lengths branch_lens[g][0..G_g-1]."""

    prompt_lens: List[int]
    branch_lens: List[List[int]]

    def __post_init__(self):
        assert len(self.prompt_lens) == len(self.branch_lens)
        for lp in self.prompt_lens:
            assert lp >= 0
        for bl in self.branch_lens:
            for li in bl:
                assert li >= 0

    @property
    def n_groups(self) -> int:
        return len(self.prompt_lens)

    @property
    def n_branches(self) -> int:
        return sum(len(b) for b in self.branch_lens)

    @property
    def total_prompt(self) -> int:
        return int(sum(self.prompt_lens))

    @property
    def total_resp(self) -> int:
        return int(sum(sum(b) for b in self.branch_lens))

    def offsets(self):
        """(prompt_off[n_groups+1], branch_begin[n_groups+1], resp_off[n_branches+1])
        as int32 arrays: the ragged descriptors of the C ABI."""
        prompt_off = np.zeros(self.n_groups + 1, dtype=np.int64)
        prompt_off[1:] = np.cumsum(self.prompt_lens)
        branch_begin = np.zeros(self.n_groups + 1, dtype=np.int64)
        branch_begin[1:] = np.cumsum([len(b) for b in self.branch_lens])
        flat = [li for b in self.branch_lens for li in b]
        resp_off = np.zeros(len(flat) + 1, dtype=np.int64)
        resp_off[1:] = np.cumsum(flat)
        for a in (prompt_off, branch_begin, resp_off):
            assert a[-1] < 2**31
        return (prompt_off.astype(np.int32), branch_begin.astype(np.int32),
                resp_off.astype(np.int32))

    def pair_count(self) -> int:
        """Number of valid (query, key) pairs with the prompt counted once."""
        n = 0
        for lp, bl in zip(self.prompt_lens, self.branch_lens):
            n += lp * (lp + 1) // 2
            for li in bl:
                n += li * lp + li * (li + 1) // 2
        return n

    def flattened_tokens(self) -> int:
        """Tokens a per-pair flattening would process: sum over pairs of L_P + L_i
        (a group without branches counts its prompt once)."""
        t = 0
        for lp, bl in zip(self.prompt_lens, self.branch_lens):
            t += sum(lp + li for li in bl) if bl else lp
        return t


@dataclasses.dataclass
class Workload:
    name: str
    tree: Tree
    hq: int
    hkv: int
    d: int
    dtype: str          # "fp32" or "bf16"
    seed: int           # tensor seed
    scale: float        # multiplier of Q/K/V values (exact power of 2); dO is unscaled

    @property
    def tokens(self) -> int:
        return self.tree.total_prompt + self.tree.total_resp

    def useful_flops(self, fwd: bool = True, bwd: bool = True) -> float:
        n = self.tree.pair_count()
        return float((4 if fwd else 0) + (10 if bwd else 0)) * self.d * self.hq * n

    def value_scale(self, name: str) -> float:
        return 1.0 if name.startswith("do") else self.scale

    def shape(self, name: str):
        rows = self.tree.total_prompt if name.endswith("_p") else self.tree.total_resp
        heads = self.hkv if name[0] in "kv" else self.hq
        return (rows, heads, self.d)


def _tiny_tree() -> Tree:
    return Tree([128], [[64, 64, 64, 64]])


def _prompt_heavy_tree(seed: int = 2) -> Tree:
    rng = np.random.default_rng(seed)
    branches = [[int(x) for x in rng.integers(512, 2049, size=8)] for _ in range(2)]
    return Tree([32768, 32768], branches)


def _response_heavy_tree(seed: int = 3) -> Tree:
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(1024.0), math.log(16384.0), size=64)
    return Tree([1024], [[int(round(math.exp(x))) for x in u]])


def _mixed_tree(seed: int = 4) -> Tree:
    rng = np.random.default_rng(seed)
    prompts, branches = [], []
    for _ in range(16):
        g = int(rng.choice([8, 16, 32]))
        rho = 10.0 ** float(rng.uniform(-3.0, 3.0))
        budget = 65536 // g
        lp = min(max(int(round(budget * rho / (1.0 + rho))), 1), budget - 1)
        prompts.append(lp)
        branches.append([budget - lp] * g)
    return Tree(prompts, branches)


def _long_tree() -> Tree:
    return Tree([262144], [[8192] * 16])


def workload(name: str) -> Workload:
    """The five seeded configurations (tiny, prompt-heavy, response-heavy, mixed, long)."""
    if name == "tiny":
        return Workload("tiny", _tiny_tree(), 2, 2, 64, "fp32", 0, 0.125)
    if name == "prompt_heavy":
        return Workload("prompt_heavy", _prompt_heavy_tree(2), 32, 8, 128, "bf16", 102, 1.0)
    if name == "response_heavy":
        return Workload("response_heavy", _response_heavy_tree(3), 32, 8, 128, "bf16", 103, 1.0)
    if name == "mixed":
        return Workload("mixed", _mixed_tree(4), 32, 8, 128, "bf16", 104, 1.0)
    if name == "long":
        return Workload("long", _long_tree(), 64, 8, 128, "bf16", 105, 1.0)
    raise KeyError(name)


WORKLOADS = ("tiny", "prompt_heavy", "response_heavy", "mixed", "long")


def custom(tree: Tree, hq: int, hkv: int, d: int, dtype: str = "bf16", seed: int = 7,
           scale: float = 1.0, name: str = "custom") -> Workload:
    return Workload(name, tree, hq, hkv, d, dtype, seed, scale)


def random_tree(rng: np.random.Generator, n_groups: int, max_prompt: int, max_branches: int,
                max_resp: int, allow_empty: bool = True) -> Tree:
    """A random ragged tree for edge-case tests."""
    lo = 0 if allow_empty else 1
    prompts = [int(rng.integers(lo, max_prompt + 1)) for _ in range(n_groups)]
    branches = []
    for _ in range(n_groups):
        g = int(rng.integers(lo, max_branches + 1))
        branches.append([int(rng.integers(lo, max_resp + 1)) for _ in range(g)])
    return Tree(prompts, branches)


# ----------------------------------------------------------------------------------
# Value table and element hash
# ----------------------------------------------------------------------------------
_TABLE64: Optional[np.ndarray] = None


def _table64() -> np.ndarray:
    global _TABLE64
    if _TABLE64 is None:
        from scipy.special import ndtri
        k = np.arange(65536, dtype=np.float64)
        _TABLE64 = ndtri((k + 0.5) / 65536.0)
    return _TABLE64


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return them as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def value_table(dtype: str, scale: float) -> np.ndarray:
    """The 65536 representable input values, as float32 holding the stored (rounded)
    value.  scale is applied in fp64 before rounding."""
    t = (_table64() * scale).astype(np.float32)
    if dtype == "bf16":
        t = round_to_bf16(t)
    elif dtype != "fp32":
        raise ValueError(dtype)
    return t


def _lowbias32_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint32)
    x ^= x >> np.uint32(16)
    x *= np.uint32(0x7FEB352D)
    x ^= x >> np.uint32(15)
    x *= np.uint32(0x846CA68B)
    x ^= x >> np.uint32(16)
    return x


def _stream_key(seed: int, tensor_id: int) -> int:
    s = (seed * 0x9E3779B9 + tensor_id * 0x85EBCA6B + 0x165667B1) & _M32
    return int(_lowbias32_np(np.array([s], dtype=np.uint32))[0])


def hash_index_np(seed: int, tensor_id: int, idx: np.ndarray) -> np.ndarray:
    """16-bit table index for flat element indices idx (int64 array)."""
    idx = np.asarray(idx, dtype=np.int64)
    key = np.uint32(_stream_key(seed, tensor_id))
    lo = (idx & _M32).astype(np.uint32)
    hi = (idx >> 32).astype(np.uint32)
    h = _lowbias32_np(lo ^ key)
    h = _lowbias32_np(h ^ hi ^ np.uint32(0x27D4EB2F))
    return (h >> np.uint32(16)).astype(np.int64)


def tensor_rows_np(w: Workload, name: str, rows: Optional[np.ndarray] = None,
                   heads: Optional[Sequence[int]] = None) -> np.ndarray:
    """Values of tensor `name` of workload w as float64, for the given token rows
    (default all) and heads (default all): shape [len(rows), len(heads), D]."""
    n_rows, n_heads, d = w.shape(name)
    rows = np.arange(n_rows, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    heads = np.arange(n_heads, dtype=np.int64) if heads is None else np.asarray(heads, np.int64)
    idx = ((rows[:, None, None] * n_heads + heads[None, :, None]) * d
           + np.arange(d, dtype=np.int64)[None, None, :])
    table = value_table(w.dtype, w.value_scale(name)).astype(np.float64)
    return table[hash_index_np(w.seed, TENSOR_ID[name], idx)]


def all_tensors_np(w: Workload, heads_q=None, heads_kv=None) -> Dict[str, np.ndarray]:
    out = {}
    for name in TENSORS:
        heads = heads_kv if name[0] in "kv" else heads_q
        out[name] = tensor_rows_np(w, name, heads=heads)
    return out


# ----------------------------------------------------------------------------------
# Device-side generation (torch).  Same hash, emulated in int64 without overflow.
# ----------------------------------------------------------------------------------
def _mul32_t(a, b: int):
    """(a * b) mod 2^32 for a int64 tensor holding uint32 values and a 32-bit constant."""
    b_lo = b & 0xFFFF
    b_hi = b >> 16
    return (a * b_lo + (((a * b_hi) & 0xFFFF) << 16)) & _M32


def _lowbias32_t(x):
    x = x ^ (x >> 16)
    x = _mul32_t(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32_t(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def hash_index_torch(seed: int, tensor_id: int, idx):
    key = _stream_key(seed, tensor_id)
    lo = idx & _M32
    hi = idx >> 32
    h = _lowbias32_t(lo ^ key)
    h = _lowbias32_t(h ^ hi ^ 0x27D4EB2F)
    return h >> 16


def tensor_torch(w: Workload, name: str, device, chunk: int = 1 << 27):
    """The whole tensor `name` on `device` in its storage dtype (torch.float32 or
    torch.bfloat16), generated in chunks of flat indices."""
    import torch
    n_rows, n_heads, d = w.shape(name)
    n = n_rows * n_heads * d
    tdtype = torch.float32 if w.dtype == "fp32" else torch.bfloat16
    table = torch.from_numpy(value_table(w.dtype, w.value_scale(name))).to(device).to(tdtype)
    out = torch.empty(n, dtype=tdtype, device=device)
    tid = TENSOR_ID[name]
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        idx = torch.arange(s, e, dtype=torch.int64, device=device)
        out[s:e] = table[hash_index_torch(w.seed, tid, idx)]
    return out.view(n_rows, n_heads, d)


def all_tensors_torch(w: Workload, device) -> Dict[str, "object"]:
    return {name: tensor_torch(w, name, device) for name in TENSORS}
