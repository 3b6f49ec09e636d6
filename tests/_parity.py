"""Helpers shared by the GPU parity tests: build a workload, run the library through
the C ABI, run the oracle on the same (cast) inputs, compare by relative L2."""
import numpy as np

import oracle
from oracle import plan_twin


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    return num / den if den > 0 else num


def leaf_order(parent):
    parent = np.asarray(parent)
    has_kid = np.zeros(len(parent), bool)
    has_kid[parent[parent >= 0]] = True
    return [i for i in range(len(parent)) if not has_kid[i]]


def oracle_run(parent, seg_len, B, inputs, *, backward, h0=None, d_final_seq=None, twin=None,
               scale=1.0):
    """Oracle over the whole forest.  `inputs` are torch CPU tensors (already cast);
    `d_final_seq` is [n_seq, H, dk, dv] in plan sequence order.  Returns dict with final
    states re-ordered to plan sequence order."""
    tw = twin if twin is not None else plan_twin.plan(parent, seg_len, B)
    f64 = lambda t: t.double().cpu().numpy()
    leaves = leaf_order(parent)
    seq_leaf = [chain[-1] for chain in tw["seq_chain"]]
    perm = [leaves.index(lf) for lf in seq_leaf]           # seq -> leaf position
    dF = None
    if d_final_seq is not None:
        dF = np.zeros_like(d_final_seq)
        dF[perm] = d_final_seq
    r = oracle.kda_forest(parent, seg_len, tw["seg_offset"], f64(inputs["q"]), f64(inputs["k"]),
                          f64(inputs["v"]), f64(inputs["g"]), f64(inputs["beta"]), chunk=B,
                          scale=scale, h0=h0, W=f64(inputs["W"]) if backward else None,
                          d_final=dF)
    r["final_seq"] = r["final"][perm]
    return r
