"""Pins of the fp64 recurrence oracle (oracle/kda_oracle.c): closed forms and special
cases of the gated delta rule, central finite differences for the backward pass,
the chunkwise form, and tree execution with bounded replay against trajectory-wise
execution."""
import numpy as np
import pytest

import oracle
from oracle import chunkwise, plan_twin


def _chain(n):
    return np.array([-1], np.int32), np.array([n], np.int64), np.array([0], np.int64)


def _rand(rng, C, H, dk, dv, decay=1.0):
    q = rng.standard_normal((C, H, dk)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((C, H, dk)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((C, H, dv))
    g = -decay * np.log1p(np.exp(rng.standard_normal((C, H, dk))))
    b = 1 / (1 + np.exp(-rng.standard_normal((C, H))))
    return q, k, v, g, b


def test_beta_zero_gives_zero():
    rng = np.random.default_rng(0)
    q, k, v, g, b = _rand(rng, 40, 2, 4, 3)
    p, l, off = _chain(40)
    r = oracle.kda_forest(p, l, off, q, k, v, g, 0 * b, chunk=8)
    assert np.all(r["o"] == 0) and np.all(r["final"] == 0)


def test_full_forgetting_gives_one_token_memory():
    # exp(g) = 0 erases the state: S_t = beta_t k_t v_t^T, o_t = beta_t (k_t.q_t) v_t
    rng = np.random.default_rng(1)
    q, k, v, g, b = _rand(rng, 30, 1, 5, 4)
    g[:] = -1e4
    p, l, off = _chain(30)
    r = oracle.kda_forest(p, l, off, q, k, v, g, b, chunk=8)
    want = (b * np.einsum("chd,chd->ch", k, q))[..., None] * v
    np.testing.assert_allclose(r["o"], want, rtol=0, atol=1e-14)


def test_delta_rule_writes_value_exactly():
    # beta = 1 and |k| = 1: S_t^T k_t = v_t; with q_t = k_t the output is v_t
    rng = np.random.default_rng(2)
    q, k, v, g, b = _rand(rng, 50, 2, 6, 5)
    p, l, off = _chain(50)
    r = oracle.kda_forest(p, l, off, k, k, v, g, np.ones_like(b), chunk=16)
    np.testing.assert_allclose(r["o"], v, rtol=0, atol=1e-12)


def test_orthonormal_keys_store_associations():
    # g = 0, beta = 1, distinct orthonormal keys: S_t = sum_s k_s v_s^T,
    # o_t = sum_{s<=t} (k_s . q_t) v_s
    rng = np.random.default_rng(3)
    d, n = 8, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm.T[:n][:, None, :]
    q = rng.standard_normal((n, 1, d))
    v = rng.standard_normal((n, 1, 3))
    p, l, off = _chain(n)
    r = oracle.kda_forest(p, l, off, q, k, v, np.zeros((n, 1, d)), np.ones((n, 1)), chunk=4)
    want = np.stack([sum((k[s, 0] @ q[t, 0]) * v[s, 0] for s in range(t + 1)) for t in range(n)])
    np.testing.assert_allclose(r["o"][:, 0], want, atol=1e-12)


def test_per_channel_decay_of_a_single_write():
    # only the first token writes: S_t = diag(exp(sum_{2..t} g)) beta_1 k_1 v_1^T
    rng = np.random.default_rng(4)
    q, k, v, g, b = _rand(rng, 12, 1, 4, 3)
    b[1:] = 0
    p, l, off = _chain(12)
    r = oracle.kda_forest(p, l, off, q, k, v, g, b, chunk=4)
    for t in range(12):
        dec = np.exp(g[1:t + 1, 0].sum(0))
        want = (q[t, 0] * dec * k[0, 0]).sum() * b[0, 0] * v[0, 0]
        np.testing.assert_allclose(r["o"][t, 0], want, atol=1e-14)


def test_scalar_state_closed_form():
    # dk = dv = 1: the state is a number, S_t = (1 - b k^2) e^g S_{t-1} + b k v
    rng = np.random.default_rng(5)
    n = 25
    q, k, v = rng.standard_normal((3, n, 1, 1))
    g = -np.abs(rng.standard_normal((n, 1, 1)))
    b = rng.random((n, 1))
    p, l, off = _chain(n)
    r = oracle.kda_forest(p, l, off, q, k, v, g, b, chunk=4)
    S, want = 0.0, []
    for t in range(n):
        kk, vv, bb = k[t, 0, 0], v[t, 0, 0], b[t, 0]
        S = (1 - bb * kk * kk) * np.exp(g[t, 0, 0]) * S + bb * kk * vv
        want.append(S * q[t, 0, 0])
    np.testing.assert_allclose(r["o"][:, 0, 0], want, atol=1e-13)


def _loss(r, W, dF):
    return float((r["o"] * W).sum() + (r["final"] * dF).sum())


@pytest.mark.parametrize("tree", ["chain", "fork"])
def test_backward_matches_central_differences(tree):
    rng = np.random.default_rng(6)
    if tree == "chain":
        parent, seg_len = np.array([-1], np.int32), np.array([11], np.int64)
    else:
        parent, seg_len = np.array([-1, 0, 0, 1, 1], np.int32), np.array([5, 3, 4, 2, 3], np.int64)
    pl = plan_twin.plan(parent, seg_len, 4)
    C, H, dk, dv = int(seg_len.sum()), 2, 3, 2
    q, k, v, g, b = _rand(rng, C, H, dk, dv, decay=0.3)
    n_roots = 1
    h0 = rng.standard_normal((n_roots, H, dk, dv))
    W = rng.standard_normal((C, H, dv))
    n_leaves = int(np.sum(np.bincount(parent[parent >= 0], minlength=len(parent)) == 0))
    dF = rng.standard_normal((n_leaves, H, dk, dv))
    args = dict(chunk=4, scale=0.7, h0=h0)
    base = oracle.kda_forest(parent, seg_len, pl["seg_offset"], q, k, v, g, b, W=W, d_final=dF, **args)
    grads = dict(q=base["dq"], k=base["dk"], v=base["dv"], g=base["dg"], beta=base["dbeta"], h0=base["dh0"])
    inputs = dict(q=q, k=k, v=v, g=g, beta=b, h0=h0)
    eps = 1e-6
    for name, x in inputs.items():
        flat = x.reshape(-1)
        for idx in rng.choice(flat.size, size=min(flat.size, 12), replace=False):
            old = flat[idx]
            flat[idx] = old + eps
            lp = _loss(oracle.kda_forest(parent, seg_len, pl["seg_offset"], inputs["q"], inputs["k"],
                                         inputs["v"], inputs["g"], inputs["beta"],
                                         chunk=4, scale=0.7, h0=inputs["h0"]), W, dF)
            flat[idx] = old - eps
            lm = _loss(oracle.kda_forest(parent, seg_len, pl["seg_offset"], inputs["q"], inputs["k"],
                                         inputs["v"], inputs["g"], inputs["beta"],
                                         chunk=4, scale=0.7, h0=inputs["h0"]), W, dF)
            flat[idx] = old
            fd = (lp - lm) / (2 * eps)
            an = grads[name].reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, an)


@pytest.mark.parametrize("B", [4, 16, 64])
def test_chunkwise_equals_recurrent(B):
    rng = np.random.default_rng(B)
    n = 3 * B + B // 2 + 1          # several chunks and a ragged tail
    q, k, v, g, b = _rand(rng, n, 1, 8, 6)
    S0 = rng.standard_normal((8, 6))
    p, l, off = _chain(n)
    r = oracle.kda_forest(p, l, off, q, k, v, g, b, chunk=B, h0=S0[None, None], scale=1.3)
    o, _, Sf = chunkwise.chunk_fwd_seq(q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], S0, B, scale=1.3)
    assert np.abs(o - r["o"][:, 0]).max() <= 1e-12 * max(1, np.abs(r["o"]).max())
    assert np.abs(Sf - r["final"][0, 0]).max() <= 1e-12 * max(1, np.abs(Sf).max())


@pytest.mark.parametrize("seed", range(6))
def test_tree_execution_with_replay_equals_trajectories(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(2, 14))
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    B = int(rng.choice([4, 8]))
    seg_len = rng.integers(1, 3 * B, size=n).astype(np.int64)
    pl = plan_twin.plan(parent, seg_len, B)
    q, k, v, g, b = _rand(rng, pl["C"], 2, 4, 3, decay=0.2)
    r = oracle.kda_forest(parent, seg_len, pl["seg_offset"], q, k, v, g, b, chunk=B)
    assert r["occ_diff"] == 0.0
    o, fin = chunkwise.tree_exec(pl, q, k, v, g, b, B)
    assert np.abs(o - r["o"]).max() < 1e-12
    leaves = [i for i in range(n) if not np.any(parent == i)]
    for s, chain in enumerate(pl["seq_chain"]):
        assert np.abs(fin[s] - r["final"][leaves.index(chain[-1])]).max() < 1e-12



@pytest.mark.parametrize("seed", range(6))
def test_nodewise_tree_execution_equals_trajectories(seed):
    """Node-wise plans (one sequence per segment, handoff at each segment's exact end,
    fresh chunk grid, no replay) compute the same outputs as the token recurrence; the
    end state of every internal sequence is the state at that segment's end, which the
    token recurrence gives at the first leaf below it (the path is shared)."""
    rng = np.random.default_rng(200 + seed)
    n = int(rng.integers(2, 14))
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    B = int(rng.choice([4, 8]))
    seg_len = rng.integers(1, 3 * B, size=n).astype(np.int64)
    pl = plan_twin.plan(parent, seg_len, B, nodewise=True)
    assert pl["n_seq"] == n and pl["R"] == 0
    depth = np.zeros(n, np.int64)
    for i in range(n):
        depth[i] = 0 if parent[i] < 0 else depth[parent[i]] + 1
    assert pl["n_rounds"] == depth.max() + 1
    q, k, v, g, b = _rand(rng, pl["C"], 2, 4, 3, decay=0.2)
    r = oracle.kda_forest(parent, seg_len, pl["seg_offset"], q, k, v, g, b, chunk=B)
    o, fin = chunkwise.tree_exec(pl, q, k, v, g, b, B)
    assert np.abs(o - r["o"]).max() < 1e-12
    leaves = [i for i in range(n) if not np.any(parent == i)]
    for s, chain in enumerate(pl["seq_chain"]):
        v_end = chain[-1]
        if v_end in leaves:
            assert np.abs(fin[s] - r["final"][leaves.index(v_end)]).max() < 1e-12
        else:
            # internal segment: run its path alone through the token recurrence
            path = []
            w = v_end
            while w >= 0:
                path.append(w)
                w = parent[w]
            rows = np.concatenate([np.arange(pl["seg_offset"][w], pl["seg_offset"][w] + seg_len[w])
                                   for w in reversed(path)])
            one = oracle.kda_forest(np.array([-1], np.int32), np.array([len(rows)]), np.array([0]),
                                    q[rows], k[rows], v[rows], g[rows], b[rows], chunk=B)
            assert np.abs(fin[s] - one["final"][0]).max() < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_noreplay_tree_execution_equals_trajectories(seed):
    """No-replay plans (side branches resume at the exact fork position from the
    producer's state there, no replay, own chunk grid) compute the same outputs and
    final states as the token recurrence; the handoff states are taken inside chunks."""
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(2, 14))
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    B = int(rng.choice([4, 8]))
    seg_len = rng.integers(1, 3 * B, size=n).astype(np.int64)
    pl = plan_twin.plan(parent, seg_len, B, noreplay=True)
    assert pl["R"] == 0
    q, k, v, g, b = _rand(rng, pl["C"], 2, 4, 3, decay=0.2)
    r = oracle.kda_forest(parent, seg_len, pl["seg_offset"], q, k, v, g, b, chunk=B)
    o, fin = chunkwise.tree_exec(pl, q, k, v, g, b, B)
    assert np.abs(o - r["o"]).max() < 1e-12
    leaves = [i for i in range(n) if not np.any(parent == i)]
    for s, chain in enumerate(pl["seq_chain"]):
        assert np.abs(fin[s] - r["final"][leaves.index(chain[-1])]).max() < 1e-12
