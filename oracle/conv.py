"""Causal short convolution over the compact layout: fp64 oracle.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module; only
``tests/`` and ``bench.py``'s reference leg do.  It shares no code with the library.

What it restates (page "HARTS ... 精读", section 4.3, KDA paragraph; summary page,
section 4 "KDA execution"): the causal convolution that precedes KDA in the layer runs
once per compact token; its window over the previous w - 1 tokens takes them from the
token's real ancestors along its own trajectory (a temporary prefix of the parent's
activations), and never from the neighbouring rows of another packed sequence.

Readings taken where the pages are silent:
* depthwise (one filter per channel), width w, weight[c, w-1] on the current token and
  weight[c, w-1-j] on the token j positions earlier: pre[t] = bias +
  sum_j weight[:, w-1-j] * x[t-j], with zeros before the trajectory start;
* activation "none" or "silu" (y = pre * sigmoid(pre));
* the loss gradient dy is given per compact row (downstream layers already summed it over
  the trajectories that share the row), so the backward is the chain rule on the compact
  rows: a row feeds every row within w - 1 positions after it on every branch.
"""
from __future__ import annotations

import numpy as np


def _paths(parent, seg_len, seg_offset):
    """Compact rows of every root-to-leaf trajectory, leaves in increasing id."""
    parent = np.asarray(parent)
    n = len(parent)
    has_kid = np.zeros(n, bool)
    has_kid[parent[parent >= 0]] = True
    out = []
    for leaf in range(n):
        if has_kid[leaf]:
            continue
        chain = []
        v = leaf
        while v >= 0:
            chain.append(v)
            v = parent[v]
        rows = [np.arange(seg_offset[v], seg_offset[v] + seg_len[v]) for v in reversed(chain)]
        out.append(np.concatenate(rows))
    return out


def _act(pre, act):
    if act == "none":
        return pre, np.ones_like(pre)
    if act == "silu":
        s = 1.0 / (1.0 + np.exp(-pre))
        return pre * s, s * (1.0 + pre * (1.0 - s))
    raise ValueError(act)


def conv_forest(parent, seg_len, seg_offset, x, weight, bias=None, act="none"):
    """Forward.  x: [C, ch]; weight: [ch, w]; bias: [ch] or None.  Each trajectory is
    convolved on its own with np.convolve (per channel); a compact row shared by several
    trajectories must come out the same from each (its window looks back only).
    Returns dict(y, pre, occ_diff)."""
    x = np.asarray(x, np.float64)
    weight = np.asarray(weight, np.float64)
    C, ch = x.shape
    w = weight.shape[1]
    pre = np.full((C, ch), np.nan)
    occ_diff = 0.0
    for rows in _paths(parent, seg_len, seg_offset):
        X = x[rows]
        P = np.empty_like(X)
        for c in range(ch):
            # np.convolve(a, k)[t] = sum_j a[t-j] k[j]; k[j] = weight[c, w-1-j]
            P[:, c] = np.convolve(X[:, c], weight[c, ::-1])[:len(rows)]
        if bias is not None:
            P = P + np.asarray(bias, np.float64)[None, :]
        seen = ~np.isnan(pre[rows, 0])
        if seen.any():
            occ_diff = max(occ_diff, float(np.abs(pre[rows[seen]] - P[seen]).max()))
        pre[rows] = P
    y, _ = _act(pre, act)
    return dict(y=y, pre=pre, occ_diff=occ_diff)


def predecessors(parent, seg_len, seg_offset, w):
    """pred[r, j]: compact row of the token j positions before row r on its trajectory
    (j = 0 is r itself), -1 before the trajectory start."""
    C = int(np.sum(seg_len))
    pred = np.full((C, w), -1, np.int64)
    for rows in _paths(parent, seg_len, seg_offset):
        for t, r in enumerate(rows):
            for j in range(w):
                if t - j >= 0:
                    pred[r, j] = rows[t - j]
    return pred


def conv_forest_bwd(parent, seg_len, seg_offset, x, weight, bias, act, dy):
    """Backward of L = sum_r <dy[r], y[r]> over compact rows.  Returns dict(dx, dweight,
    dbias)."""
    x = np.asarray(x, np.float64)
    weight = np.asarray(weight, np.float64)
    dy = np.asarray(dy, np.float64)
    w = weight.shape[1]
    f = conv_forest(parent, seg_len, seg_offset, x, weight, bias, act)
    _, dact = _act(f["pre"], act)
    dpre = dy * dact
    pred = predecessors(parent, seg_len, seg_offset, w)
    dx = np.zeros_like(x)
    dW = np.zeros_like(weight)
    for r in range(x.shape[0]):
        for j in range(w):
            p = pred[r, j]
            if p >= 0:
                dx[p] += weight[:, w - 1 - j] * dpre[r]
                dW[:, w - 1 - j] += x[p] * dpre[r]
    return dict(dx=dx, dweight=dW, dbias=dpre.sum(axis=0), dpre=dpre)
