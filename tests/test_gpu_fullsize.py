"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

The whole forest runs through the library; sampled trajectories (the deepest one, the
one with the most replay, a random one) are checked against the fp64 oracle run on
that trajectory alone, for a few heads:
  * forward: o on every row of the trajectory, and the final state of the sequence
    that ends at its leaf;
  * backward: the loss is restricted to the trajectory's rows (dO = W there, 0
    elsewhere), so the oracle's gradients over the trajectory are the exact ones, and
    every row off the trajectory's path must get exactly zero gradient.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from oracle import plan_twin
from prefix_shared_chunkwise_gb300.api import Plan, kda_bwd, kda_fwd
from prefix_shared_chunkwise_gb300.synth import WORKLOADS, expand_rows, make_inputs, make_tree
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2
# heads compared with the oracle: where the sequential passes group four heads per block
# (the second round of the 256K-token forest), 0 opens a group, 5 and 30 follow one and two
# head changes inside a block
HEADS = (0, 5, 30)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from prefix_shared_chunkwise_gb300 import build
    build.build()


def _samples(parent, seg_len, tw, rng):
    rows, ptr, leaves = expand_rows(parent, seg_len, tw["seg_offset"])
    n = len(leaves)
    depth = np.zeros(len(parent), np.int64)
    for i in range(len(parent)):
        depth[i] = 0 if parent[i] < 0 else depth[parent[i]] + 1
    seq_of_leaf = {chain[-1]: s for s, chain in enumerate(tw["seq_chain"])}
    rho = np.array([tw["seq_replay"][seq_of_leaf[int(lf)]] for lf in leaves])
    picks = {int(np.argmax(depth[leaves])), int(np.argmax(rho)), int(rng.integers(0, n))}
    return [(rows[ptr[i]:ptr[i + 1]], int(leaves[i]), seq_of_leaf[int(leaves[i])]) for i in sorted(picks)]


@pytest.mark.parametrize("name", ["wide256k_bf16", "deep128k_bf16", "fb64k_bf16", "fwd16k_bf16"])
def test_full_size_workload_sampled_trajectories(name):
    wl = WORKLOADS[name]
    H, D, B = wl.H, wl.dk, wl.chunk
    parent, seg_len = make_tree(name)
    tw = plan_twin.plan(parent, seg_len, B)
    pl = Plan(parent, seg_len, B).upload()
    assert pl.info["n_rounds"] == tw["n_rounds"]
    C = pl.info["C"]
    x = make_inputs(C, H, D, D, wl.dtype, seed=3, device="cuda")
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 1) // 2, dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((pl.info["n_seq"], H, D, D), device="cuda")
    o, states, fin, cs = kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], final_state=fin,
                                 chunk_states=cs)
    torch.cuda.synchronize()
    assert pl.device_error() == 0
    rng = np.random.Generator(np.random.PCG64(7))
    hs = [h for h in HEADS if h < H]
    for rows, leaf, seq in _samples(parent, seg_len, tw, rng):
        idx = torch.as_tensor(rows, device="cuda")
        sub = {k: v.index_select(0, idx)[:, hs].float().cpu().double().numpy() for k, v in x.items()}
        one = np.array([-1], np.int32)
        ref = oracle.kda_forest(one, np.array([len(rows)]), np.array([0]), sub["q"], sub["k"],
                                sub["v"], sub["g"], sub["beta"], chunk=B,
                                W=sub["W"] if wl.backward else None)
        got_o = o.index_select(0, idx)[:, hs].float().cpu().numpy()
        assert rel_l2(got_o, ref["o"]) <= TOL, (name, leaf, "o")
        got_f = fin[seq][hs].cpu().numpy()
        assert rel_l2(got_f, ref["final"][0]) <= TOL, (name, leaf, "final")
        if not wl.backward:
            continue
        dO = torch.zeros_like(x["W"])
        dO[idx] = x["W"][idx]
        gr = kda_bwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], dO, states=states,
                     chunk_states=cs)
        torch.cuda.synchronize()
        assert pl.device_error() == 0
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            got = gr[n].index_select(0, idx)[:, hs].float().cpu().numpy()
            assert rel_l2(got, ref[n]) <= TOL, (name, leaf, n, rel_l2(got, ref[n]))
            off = torch.ones(C, dtype=torch.bool, device="cuda")
            off[idx] = False
            assert float(gr[n][off].abs().max()) == 0.0, (name, leaf, n, "off-path gradient")


def _tree_properties(parent, seg_len, tw):
    """Per tree (by root segment): the rounds its sequences run in, how many side branches
    start by replay in their producer's round (delta = 0), how many boundary slots feed
    two or more consumers, and its expanded size S."""
    from prefix_shared_chunkwise_gb300.synth import tree_stats
    n = len(parent)
    root = np.zeros(n, np.int64)
    for i in range(n):
        root[i] = i if parent[i] < 0 else root[parent[i]]
    seq_tree = root[tw["seq_first_seg"]]
    ncons = np.diff(tw["state_cons_ptr"])
    slot_tree = seq_tree[tw["state_seq"]]
    out = []
    for r in np.unique(root):
        seqs = np.nonzero(seq_tree == r)[0]
        d0 = 0
        for s in seqs:
            f = tw["seq_first_seg"][s]
            if parent[f] >= 0 and tw["seq_round"][s] == tw["seq_round"][tw["seg_seq"][parent[f]]]:
                d0 += 1
        ids = np.nonzero(root == r)[0]
        remap = {int(v): j for j, v in enumerate(ids)}
        sub_parent = np.array([-1 if parent[v] < 0 else remap[int(parent[v])] for v in ids], np.int32)
        out.append(dict(ids=ids, sub_parent=sub_parent, rounds=len(np.unique(tw["seq_round"][seqs])),
                        d0=d0, multi=int((ncons[slot_tree == r] >= 2).sum()),
                        S=tree_stats(sub_parent, seg_len[ids])["S"]))
    return out


@pytest.mark.parametrize("name,need", [
    ("wide256k_bf16", dict(d0=1, multi=1, rounds=2)),     # 2-round forest: shared slots, delta = 0 starts
    ("deep128k_bf16", dict(d0=0, multi=0, rounds=6)),     # 7-round forest: handoffs nested 6 deep
])
def test_full_size_backward_whole_tree(name, need):
    """Backward at full size, in the bench's launch configuration, with the loss on every
    row of one whole tree: dO = W on the tree's rows, zero elsewhere.  Every handoff of the
    tree then carries gradient: consumers' initial-state gradients summed into shared slots,
    same-round (delta = 0) starts, replay rows of many branches folded into one ancestor
    row.  dq, dk, dv, dg, dbeta on all of the tree's rows are compared with the oracle run
    on that tree (relative L2 over the tree and over each segment), and every row outside
    the tree must get exactly zero gradient.  The tree is the smallest (in expanded
    tokens) that has the listed features."""
    wl = WORKLOADS[name]
    H, D, B = wl.H, wl.dk, wl.chunk
    parent, seg_len = make_tree(name)
    tw = plan_twin.plan(parent, seg_len, B)
    cands = [t for t in _tree_properties(parent, seg_len, tw)
             if t["d0"] >= need["d0"] and t["multi"] >= need["multi"] and t["rounds"] >= need["rounds"]]
    assert cands, name
    tree = min(cands, key=lambda t: t["S"])
    ids = tree["ids"]
    so = tw["seg_offset"]
    seg_rows = [np.arange(so[v], so[v] + seg_len[v]) for v in ids]
    rows = np.concatenate(seg_rows)
    sub_off = np.concatenate([[0], np.cumsum(seg_len[ids])[:-1]]).astype(np.int64)

    pl = Plan(parent, seg_len, B).upload()
    C = pl.info["C"]
    x = make_inputs(C, H, D, D, wl.dtype, seed=11, device="cuda")
    cs = torch.empty(pl.chunk_state_bytes(H, D, D, 1) // 2, dtype=torch.bfloat16, device="cuda")
    o, states, _, cs = kda_fwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], chunk_states=cs)
    idx = torch.as_tensor(rows, device="cuda")
    dO = torch.zeros_like(x["W"])
    dO[idx] = x["W"][idx]
    gr = kda_bwd(pl, x["q"], x["k"], x["v"], x["g"], x["beta"], dO, states=states, chunk_states=cs)
    torch.cuda.synchronize()
    assert pl.device_error() == 0

    hs = [0, H - 1]
    sub = {k: v.index_select(0, idx)[:, hs].float().cpu().double().numpy() for k, v in x.items()}
    ref = oracle.kda_forest(tree["sub_parent"], seg_len[ids], sub_off, sub["q"], sub["k"], sub["v"],
                            sub["g"], sub["beta"], chunk=B, W=sub["W"], n_threads=len(hs))
    off = torch.ones(C, dtype=torch.bool, device="cuda")
    off[idx] = False
    bounds = np.concatenate([[0], np.cumsum(seg_len[ids])])
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        got = gr[n].index_select(0, idx)[:, hs].float().cpu().numpy()
        assert rel_l2(got, ref[n]) <= TOL, (name, n, rel_l2(got, ref[n]))
        for j in range(len(ids)):
            a, b = bounds[j], bounds[j + 1]
            e = rel_l2(got[a:b], ref[n][a:b])
            assert e <= 2 * TOL, (name, n, "segment", int(ids[j]), e)
        assert float(gr[n][off].abs().max()) == 0.0, (name, n, "gradient outside the tree")
