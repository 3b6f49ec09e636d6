"""Pins for the branch-attention oracle (oracle/attn.py): a plain chain equals torch's
scaled_dot_product_attention (causal), shared rows agree across trajectories, and a
hand case of the bottom-right alignment (a branch's first query sees the whole ancestor
prefix and itself, not its sibling)."""
import numpy as np
import pytest

from oracle import attn

torch = pytest.importorskip("torch")


def test_chain_equals_torch_sdpa():
    rng = np.random.default_rng(1)
    L, H, d = 37, 3, 16
    q, k, v = (rng.standard_normal((L, H, d)) for _ in range(3))
    r = attn.attn_forest(np.array([-1]), np.array([L]), np.array([0]), q, k, v, 0.25)
    t = lambda a: torch.as_tensor(a.transpose(1, 0, 2)[None])      # [1, H, L, d]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=0.25)
    np.testing.assert_allclose(r["o"], ref[0].numpy().transpose(1, 0, 2), atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_shared_rows_agree(seed):
    rng = np.random.default_rng(10 + seed)
    n = 9
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)])
    seg_len = rng.integers(1, 6, size=n)
    so = np.concatenate([[0], np.cumsum(seg_len)[:-1]])
    C = int(seg_len.sum())
    q, k, v = (rng.standard_normal((C, 2, 4)) for _ in range(3))
    r = attn.attn_forest(parent, seg_len, so, q, k, v, 0.5)
    assert r["occ_diff"] < 1e-12 and not np.isnan(r["o"]).any()


def test_branch_sees_ancestors_not_sibling():
    # root A (2 rows) -> B (1 row), C (1 row); rows: A0 A1 B0 C0
    parent = np.array([-1, 0, 0])
    seg_len = np.array([2, 1, 1])
    so = np.array([0, 2, 3])
    q = np.zeros((4, 1, 1))
    k = np.zeros((4, 1, 1))
    v = np.array([1.0, 2.0, 100.0, 5.0]).reshape(4, 1, 1)
    o = attn.attn_forest(parent, seg_len, so, q, k, v, 1.0)["o"][:, 0, 0]
    # zero scores: uniform over the visible rows
    assert o[3] == pytest.approx((1 + 2 + 5) / 3)      # C0 sees A0, A1, C0 -- not B0
    assert o[2] == pytest.approx((1 + 2 + 100) / 3)


def test_single_query_matches_forest():
    """attn_query over trajectory_prefix (used for sampled rows of large forests) gives
    the forest oracle's output for every row of a random forest, with the compact rows
    laid out in a shuffled segment order."""
    rng = np.random.default_rng(21)
    n = 10
    parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)])
    seg_len = rng.integers(1, 7, size=n)
    order = rng.permutation(n)
    so = np.zeros(n, np.int64)
    so[order] = np.concatenate([[0], np.cumsum(seg_len[order])[:-1]])
    C = int(seg_len.sum())
    q, k, v = (rng.standard_normal((C, 2, 5)) for _ in range(3))
    full = attn.attn_forest(parent, seg_len, so, q, k, v, 0.3)
    for r in range(C):
        view = attn.trajectory_prefix(parent, seg_len, so, r)
        assert view[-1] == r and len(np.unique(view)) == len(view)
        o, lse = attn.attn_query(q[r], k[view], v[view], 0.3)
        np.testing.assert_allclose(o, full["o"][r], atol=1e-12)
        np.testing.assert_allclose(lse, full["lse"][r], atol=1e-12)


def _expanded_autograd(parent, seg_len, so, q, k, v, do, scale):
    """Independent check: every trajectory through torch's causal scaled_dot_product_attention
    with autograd; each compact row's output gradient sits on one occurrence (the first
    trajectory, leaves by id), input gradients summed over occurrences."""
    from oracle.conv import _paths
    C = q.shape[0]
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    seen = np.zeros(C, bool)
    loss = 0
    for rows in _paths(parent, seg_len, so):
        idx = torch.as_tensor(rows)
        t = lambda a: a[idx].transpose(0, 1)[None]             # [1, H, L, d]
        o = torch.nn.functional.scaled_dot_product_attention(t(tq), t(tk), t(tv), is_causal=True,
                                                             scale=scale)[0].transpose(0, 1)
        w = torch.as_tensor(do[rows] * (~seen[rows])[:, None, None])
        seen[rows] = True
        loss = loss + (o * w).sum()
    loss.backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("seed", range(3))
def test_backward_equals_expanded_autograd(seed):
    rng = np.random.default_rng(30 + seed)
    n = 8
    parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, n)])
    seg_len = rng.integers(1, 6, size=n)
    so = np.concatenate([[0], np.cumsum(seg_len)[:-1]])
    C = int(seg_len.sum())
    q, k, v, do = (rng.standard_normal((C, 2, 4)) for _ in range(4))
    g = attn.attn_forest_bwd(parent, seg_len, so, q, k, v, do, 0.4)
    eq, ek, ev = _expanded_autograd(parent, seg_len, so, q, k, v, do, 0.4)
    np.testing.assert_allclose(g["dq"], eq, atol=1e-12)
    np.testing.assert_allclose(g["dk"], ek, atol=1e-12)
    np.testing.assert_allclose(g["dv"], ev, atol=1e-12)


def test_backward_finite_differences():
    rng = np.random.default_rng(40)
    parent = np.array([-1, 0, 0, 1])
    seg_len = np.array([3, 2, 2, 1])
    so = np.array([0, 3, 5, 7])
    C = 8
    q, k, v, do = (rng.standard_normal((C, 1, 3)) for _ in range(4))
    g = attn.attn_forest_bwd(parent, seg_len, so, q, k, v, do, 0.7)
    loss = lambda a, b, c: float((attn.attn_forest(parent, seg_len, so, a, b, c, 0.7)["o"] * do).sum())
    eps = 1e-6
    for name, arr in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a = [q.copy(), k.copy(), v.copy()]
            j = ("dq", "dk", "dv").index(name)
            a[j][i] += eps
            up = loss(*a)
            a[j][i] -= 2 * eps
            num[i] = (up - loss(*a)) / (2 * eps)
        np.testing.assert_allclose(g[name], num, rtol=1e-6, atol=1e-8)
