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
HEADS = (0, 5)


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
