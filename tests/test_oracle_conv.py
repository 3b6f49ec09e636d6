"""Pins for the short-convolution oracle (oracle/conv.py) against things other than
itself: a library routine (np.convolve / np.correlate on a plain chain), finite
differences, and the tree property that a shared row has one value."""
import numpy as np
import pytest

from oracle import conv


def _tree(rng, n, max_len):
    parent = np.array([-1] + [int(rng.integers(0, i)) if rng.random() > 0.1 else -1 for i in range(1, n)],
                      np.int32)
    seg_len = rng.integers(1, max_len + 1, size=n).astype(np.int64)
    seg_offset = np.concatenate([[0], np.cumsum(seg_len)[:-1]])
    return parent, seg_len, seg_offset


@pytest.mark.parametrize("w", [1, 2, 4, 8])
def test_chain_equals_torch_style_causal_conv(w):
    """One segment: the causal depthwise conv with left zero padding, written with
    np.correlate on the padded signal (weight[w-1] on the current token)."""
    rng = np.random.default_rng(w)
    L, ch = 37, 5
    x = rng.standard_normal((L, ch))
    W = rng.standard_normal((ch, w))
    b = rng.standard_normal(ch)
    r = conv.conv_forest(np.array([-1]), np.array([L]), np.array([0]), x, W, b)
    for c in range(ch):
        padded = np.concatenate([np.zeros(w - 1), x[:, c]])
        ref = np.correlate(padded, W[c], mode="valid") + b[c]
        np.testing.assert_allclose(r["y"][:, c], ref, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
def test_tree_rows_shared_by_trajectories_agree(seed):
    rng = np.random.default_rng(10 + seed)
    parent, seg_len, so = _tree(rng, 12, 6)
    x = rng.standard_normal((int(seg_len.sum()), 3))
    W = rng.standard_normal((3, 4))
    r = conv.conv_forest(parent, seg_len, so, x, W, None, "silu")
    assert r["occ_diff"] == 0.0
    assert not np.isnan(r["y"]).any()


def test_window_reaches_into_ancestors_only():
    """A child's first token sees its parent's last tokens, never a sibling's rows that
    sit right before it in the compact layout."""
    parent = np.array([-1, 0, 0], np.int32)
    seg_len = np.array([3, 2, 2])
    so = np.array([0, 3, 5])
    x = np.zeros((7, 1))
    x[4, 0] = 1.0                   # last row of child 1, just before child 2's first row
    W = np.ones((1, 3))
    y = conv.conv_forest(parent, seg_len, so, x, W)["y"]
    assert y[5, 0] == 0.0 and y[6, 0] == 0.0       # child 2 ignores child 1
    assert y[4, 0] == 1.0                          # child 1 sees itself


def test_chain_backward_equals_correlation():
    """Plain chain, no activation: dx is the anti-causal correlation of dy with the
    weights, dW the lagged cross-correlation of x and dy, db the sum of dy."""
    rng = np.random.default_rng(3)
    L, ch, w = 29, 4, 4
    x = rng.standard_normal((L, ch))
    W = rng.standard_normal((ch, w))
    dy = rng.standard_normal((L, ch))
    g = conv.conv_forest_bwd(np.array([-1]), np.array([L]), np.array([0]), x, W, np.zeros(ch), "none", dy)
    for c in range(ch):
        # y[t] = sum_k W[k] x[t-(w-1)+k]  =>  dx[s] = sum_k W[k] dy[s+(w-1)-k]
        dyp = np.concatenate([dy[:, c], np.zeros(w - 1)])
        ref = np.convolve(dyp, W[c], mode="full")[w - 1:w - 1 + L]
        np.testing.assert_allclose(g["dx"][:, c], ref, atol=1e-12)
        for k in range(w):
            lag = w - 1 - k
            np.testing.assert_allclose(g["dweight"][c, k], np.dot(x[:L - lag, c], dy[lag:, c]), atol=1e-12)
    np.testing.assert_allclose(g["dbias"], dy.sum(0), atol=1e-12)


@pytest.mark.parametrize("act", ["none", "silu"])
def test_tree_backward_finite_differences(act):
    rng = np.random.default_rng(7)
    parent, seg_len, so = _tree(rng, 7, 4)
    C, ch, w = int(seg_len.sum()), 2, 3
    x = rng.standard_normal((C, ch))
    W = rng.standard_normal((ch, w))
    b = rng.standard_normal(ch)
    dy = rng.standard_normal((C, ch))
    g = conv.conv_forest_bwd(parent, seg_len, so, x, W, b, act, dy)

    def loss(x_, W_, b_):
        return float(np.sum(dy * conv.conv_forest(parent, seg_len, so, x_, W_, b_, act)["y"]))

    eps = 1e-6
    for arr, grad in ((x, g["dx"]), (W, g["dweight"]), (b, g["dbias"])):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a0 = arr[idx]
            arr[idx] = a0 + eps; lp = loss(x, W, b)
            arr[idx] = a0 - eps; lm = loss(x, W, b)
            arr[idx] = a0
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=1e-6, rtol=1e-6)
