"""Seeded synthetic workloads: rollout segment trees and KDA input tensors.

This module only draws inputs. It holds none of the method's arithmetic (no
recurrence, no planner), so that the fp64 oracle and the CUDA path can both be fed
from it without sharing any of the computation they are compared on.

Workloads follow the problem statement of HARTS (arXiv 2608.28158): a rollout tree
is contracted into fork-free segments (page "HARTS ... 精读", section 4.2); each
root-to-leaf path is a training trajectory (section 1.1).  The pages' SWE-bench
rollout trees are not available, so seeded trees with the same shape statistics
stand in for them (about 5.6x trajectory-to-compact expansion, section 1.1;
real trees finish in 2-3 calls, section 6 "因果链四").

Tree format: ``parent[i] < i`` (-1 for a root; forests allowed) and
``seg_len[i] >= 1`` tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "fig1_tree", "make_tree", "tree_stats", "make_inputs",
    "expand_rows", "WORKLOAD_ORDER",
]


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    dk: int
    dv: int
    chunk: int
    dtype: str            # "fp32" or "bf16": the dtype of q, k, v, g, beta, o and grads
    backward: bool
    n_trees: int
    target_C: int | None = None
    target_S_over_C: float | None = None
    note: str = ""


# The five workloads: sizes, heads, head dims, chunk length and dtypes as the
# benchmark statement gives them.
WORKLOADS: dict[str, Workload] = {
    "fig1_fp32": Workload("fig1_fp32", H=1, dk=32, dv=32, chunk=16, dtype="fp32",
                          backward=True, n_trees=1,
                          note="Fig. 1 tree: A=100; B=50, C=70 under A; D=90, E=40 under B"),
    "fwd16k_bf16": Workload("fwd16k_bf16", H=16, dk=128, dv=128, chunk=64, dtype="bf16",
                            backward=False, n_trees=8, target_C=16384,
                            note="8 trees, depth 3-6, fanout 1-4, segments 32-2048"),
    "fb64k_bf16": Workload("fb64k_bf16", H=16, dk=128, dv=128, chunk=64, dtype="bf16",
                           backward=True, n_trees=32, target_C=65536, target_S_over_C=5.6,
                           note="32 trees as fwd16k, two-factor scaled to S/C = 5.6"),
    "wide256k_bf16": Workload("wide256k_bf16", H=32, dk=128, dv=128, chunk=64, dtype="bf16",
                              backward=True, n_trees=64, target_C=262144,
                              target_S_over_C=1_400_000 / 262_144,
                              note="64 trees, shared root 8K-16K, 3-10 levels of fanout 2-8, "
                                   "branches 64-4096"),
    "deep128k_bf16": Workload("deep128k_bf16", H=16, dk=128, dv=128, chunk=64, dtype="bf16",
                              backward=True, n_trees=16, target_C=131072,
                              note="16 chain-heavy trees, every fork at chunk offset 1-63, "
                                   "nested side branches (Strahler 6-8 rounds)"),
}
WORKLOAD_ORDER = ["fig1_fp32", "fwd16k_bf16", "fb64k_bf16", "wide256k_bf16", "deep128k_bf16"]


def fig1_tree():
    """The tree of Fig. 1(a) with token counts: root A, children B and C of A,
    children D and E of B (segment ids 0..4 = A..E)."""
    parent = np.array([-1, 0, 0, 1, 1], dtype=np.int32)
    seg_len = np.array([100, 50, 70, 90, 40], dtype=np.int64)
    return parent, seg_len


def _loguniform(rng, lo, hi, size=None):
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=size))


def _chain_heavy_tree(rng, levels, fan_lo, fan_hi, len_lo, len_hi, root_len):
    """One agentic-style tree: at each fork level the frontier segment draws a
    fanout f; f = 1 extends the frontier, otherwise it forks into f children of
    which one (drawn at random) becomes the next frontier and the rest are leaves."""
    parent = [-1]
    length = [float(root_len)]
    frontier = 0
    for _ in range(levels):
        f = int(rng.integers(fan_lo, fan_hi + 1))
        if f == 1:
            length[frontier] += float(_loguniform(rng, len_lo, len_hi))
            continue
        kids = []
        for _ in range(f):
            parent.append(frontier)
            length.append(float(_loguniform(rng, len_lo, len_hi)))
            kids.append(len(parent) - 1)
        frontier = kids[int(rng.integers(0, f))]
    return parent, length


def _leaf_counts(parent):
    n = len(parent)
    nkids = np.zeros(n, np.int64)
    for i in range(n):
        if parent[i] >= 0:
            nkids[parent[i]] += 1
    leaves = (nkids == 0).astype(np.int64)
    cnt = leaves.copy()
    for i in range(n - 1, -1, -1):
        if parent[i] >= 0:
            cnt[parent[i]] += cnt[i]
    return cnt, nkids == 0


def _forest(trees):
    parent, length = [], []
    for p, l in trees:
        base = len(parent)
        parent.extend([-1 if x < 0 else x + base for x in p])
        length.extend(l)
    return parent, length


def _scale_two_factor(parent, length, target_C, target_ratio):
    """Scale internal segments by a and leaves by b so that C and S hit their
    targets (the 2x2 linear system in the two unknowns).  Returns None if the
    system has no positive solution."""
    mult, is_leaf = _leaf_counts(parent)
    L = np.asarray(length, np.float64)
    Ci = L[~is_leaf].sum(); Cl = L[is_leaf].sum()
    Si = (L * mult)[~is_leaf].sum(); Sl = L[is_leaf].sum()
    Ct, St = float(target_C), float(target_C) * target_ratio
    det = Ci * Sl - Cl * Si
    if det == 0:
        return None
    a = (Ct * Sl - Cl * St) / det
    b = (Ci * St - Si * Ct) / det
    if a <= 0 or b <= 0:
        return None
    out = np.where(is_leaf, L * b, L * a)
    return np.maximum(1, np.rint(out)).astype(np.int64)


def _strahler_tree(rng, k, spine_forks, B, leaf_budget):
    """A chain-heavy tree whose minimum call count is the Horton-Strahler number k:
    a top spine of `spine_forks` forks with leaf side children, then nested binary
    forks.  Every internal segment crosses a chunk boundary and ends at offset 1..B-1
    within a chunk, so every side branch replays 1..B-1 tokens."""
    parent, length, start = [], [], []
    internal = []

    def add(par, internal_seg):
        s = 0 if par < 0 else start[par] + length[par]
        if internal_seg:
            off = int(rng.integers(1, B))
            e = (s // B + 1) * B + off
            ln = e - s
        else:
            ln = 1  # set later from the leaf budget
        parent.append(par); length.append(ln); start.append(s)
        internal.append(internal_seg)
        return len(parent) - 1

    def gen(par, level_k, nf):
        if level_k == 1:
            add(par, False)
            return
        v = par
        for _ in range(nf):
            v_new = add(v, True)
            add(v_new, False)          # side leaf
            v = v_new
        b = add(v, True)               # binary fork: two subtrees of Strahler k-1
        gen(b, level_k - 1, 0)
        gen(b, level_k - 1, 0)

    # the root is itself an internal segment of the top spine
    root = add(-1, True)
    add(root, False)
    gen(root, k, spine_forks - 1)
    leaves = [i for i in range(len(parent)) if not internal[i]]
    w = _loguniform(rng, 1.0, 16.0, size=len(leaves))
    w = w / w.sum() * max(leaf_budget, len(leaves))
    for i, x in zip(leaves, w):
        length[i] = max(1, int(round(x)))
    return parent, length


def make_tree(name: str, seed: int | None = None):
    """Seeded segment forest for a workload.  Returns (parent int32[n], seg_len int64[n])."""
    wl = WORKLOADS[name]
    if seed is None:
        seed = WORKLOAD_ORDER.index(name)
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "fig1_fp32":
        return fig1_tree()
    if name in ("fwd16k_bf16", "fb64k_bf16"):
        for _ in range(200):
            trees = []
            for _ in range(wl.n_trees):
                levels = int(rng.integers(3, 7))
                trees.append(_chain_heavy_tree(rng, levels, 1, 4, 32, 2048,
                                               _loguniform(rng, 32, 2048)))
            parent, length = _forest(trees)
            if wl.target_S_over_C is None:
                L = np.asarray(length)
                seg = np.maximum(1, np.rint(L * wl.target_C / L.sum())).astype(np.int64)
                break
            seg = _scale_two_factor(parent, length, wl.target_C, wl.target_S_over_C)
            if seg is not None:
                break
        else:
            raise RuntimeError("no feasible draw")
        return np.asarray(parent, np.int32), seg
    if name == "wide256k_bf16":
        for _ in range(200):
            trees = []
            for _ in range(wl.n_trees):
                levels = int(rng.integers(3, 11))
                trees.append(_chain_heavy_tree(rng, levels, 2, 8, 64, 4096,
                                               rng.uniform(8192, 16384)))
            parent, length = _forest(trees)
            seg = _scale_two_factor(parent, length, wl.target_C, wl.target_S_over_C)
            if seg is not None:
                break
        else:
            raise RuntimeError("no feasible draw")
        return np.asarray(parent, np.int32), seg
    if name == "deep128k_bf16":
        trees = []
        per_tree = wl.target_C // wl.n_trees
        for _ in range(wl.n_trees):
            k = int(rng.integers(6, 8))
            nf = int(rng.integers(20, 41)) - (k - 1)
            # internal segments cost about B tokens each; leaves take the rest
            n_internal = nf + (2 ** (k - 1) - 1)
            budget = per_tree - n_internal * wl.chunk
            trees.append(_strahler_tree(rng, k, nf, wl.chunk, budget))
        parent, length = _forest(trees)
        return np.asarray(parent, np.int32), np.asarray(length, np.int64)
    raise KeyError(name)


def tree_stats(parent, seg_len):
    """C (compact tokens), S (expanded trajectory tokens), segments, leaves, roots."""
    parent = np.asarray(parent)
    seg_len = np.asarray(seg_len, np.int64)
    mult, is_leaf = _leaf_counts(list(parent))
    return dict(C=int(seg_len.sum()), S=int((seg_len * mult).sum()), n_seg=len(parent),
                n_leaves=int(is_leaf.sum()), n_roots=int((parent < 0).sum()))


_TENSOR_IDS = dict(q=1, k=2, v=3, g=4, beta=5, W=6)


def make_inputs(C, H, dk, dv, dtype, seed, device="cpu"):
    """Seeded KDA inputs in the compact layout ``[C, H, d]`` (``beta``: ``[C, H]``).

    q, k ~ N(0,1) L2-normalised per (token, head); v ~ N(0,1); beta = sigmoid(N(0,1));
    g = -softplus(N(0,1)) per channel (natural-log decay); W ~ N(0,1) is the fixed
    loss weight (the output gradient).  Normalisation happens before the cast, as the
    workloads specify.  Each tensor draws from its own torch generator seeded
    ``1000*seed + id``."""
    import torch
    td = {"fp32": torch.float32, "bf16": torch.bfloat16}[dtype]
    dev = torch.device(device)
    out = {}
    shapes = dict(q=(C, H, dk), k=(C, H, dk), v=(C, H, dv), g=(C, H, dk), beta=(C, H),
                  W=(C, H, dv))
    for name, tid in _TENSOR_IDS.items():
        gen = torch.Generator(device=dev)
        gen.manual_seed(1000 * seed + tid)
        x = torch.randn(shapes[name], generator=gen, device=dev, dtype=torch.float32)
        if name in ("q", "k"):
            x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        elif name == "g":
            x = -torch.nn.functional.softplus(x)
        elif name == "beta":
            x = torch.sigmoid(x)
        out[name] = x.to(td).contiguous()
        del x
    return out


def expand_rows(parent, seg_len, seg_offset):
    """Compact row indices of every trajectory, leaves in increasing segment id.
    Returns (rows int64[S], traj_ptr int64[n_leaves+1], leaf ids)."""
    parent = np.asarray(parent)
    n = len(parent)
    nk = np.zeros(n, np.int64)
    for i in range(n):
        if parent[i] >= 0:
            nk[parent[i]] += 1
    leaves = [i for i in range(n) if nk[i] == 0]
    rows, ptr = [], [0]
    for lf in leaves:
        path = []
        v = lf
        while v >= 0:
            path.append(v)
            v = parent[v]
        for v in reversed(path):
            rows.append(np.arange(seg_offset[v], seg_offset[v] + seg_len[v], dtype=np.int64))
        ptr.append(ptr[-1] + sum(int(seg_len[v]) for v in path))
    return np.concatenate(rows), np.asarray(ptr, np.int64), np.asarray(leaves, np.int64)
